// pkd_decode_mma.cuh -- decode attention with Q.K^T and P.V on the tensor
// cores (sm_103a), for the group sizes where the fp32 FMA path runs out of
// issue slots before HBM runs out of bandwidth.
//
// The work split is the one of paged_decode_kernel: one CTA per (sequence b,
// kv head g, partition j); NW warps take the partition's 16-token sub-tiles
// in the stride-NW block order of Algorithm 1 of the review "Accelerating LLM
// Inference Throughput via Asynchronous KV Cache Prefetching" (section 3.4);
// each warp keeps its own online-softmax state, merged at the end.
//
// Staging.  Lane 0 of every warp streams its sub-tiles into a private ring of
// shared-memory slots with 3-D tensor copies (cp.async.bulk.tensor; the
// tensor map views a cache as [num_blocks][num_kv_heads * block_size][D]).
// A box is 16 rows x 64 halves (128 bytes) with the 128-byte swizzle, so the
// 16-byte chunk j of row r lands at chunk j ^ (r % 8): the eight rows an
// ldmatrix reads in one phase fall in eight different bank groups.  The ring
// is itself an asynchronous prefetch of the warp's next sub-tiles into SRAM;
// with prefetch_distance >= 1, whole tiles beyond it are also prefetched into
// L2 (cp.async.bulk.prefetch.L2), the pairing of SRAM staging with L2
// prefetch that the blog post "KV Cache Prefetching：三层预取如何隐藏 KV 访问延迟"
// suggests (section 2.3).  That extra prefetch measured slower on GB300, so
// it is off by default.
//
// Arithmetic per 16-token sub-tile, with mma.m16n8k16 (fp16 operands, fp32
// accumulators), c = lane % 4 and r = lane / 4:
//   S  = Q . K^T     M = the group's query heads (padded to 16 rows; rows 8..15
//                    are zero), N = 8 tokens (two n-tiles), K = 16 dims per
//                    step.  Q is held as A fragments for the whole CTA; K^T
//                    comes from ldmatrix (non-transposed) of the K rows.
//                    Lane (r, c) receives S[head r][tokens 2c, 2c+1, 8+2c, 9+2c].
//   softmax          fp32, log2 domain, lazy running max per head (the four
//                    lanes of a head agree through a 2-step butterfly).
//   O^T += V^T . P^T M = 16 dims per m-tile, N = 8 heads, K = 16 tokens.  V^T
//                    comes from ldmatrix.trans of the V rows; P^T's B fragment
//                    is exactly the lane's own four p values packed to fp16
//                    (tokens 2c, 2c+1 | 8+2c, 9+2c of head r), so no shuffle or
//                    shared-memory round trip sits between the two products.
// P is rounded to fp16 for the second product (relative error <= 2^-11 per
// weight); the normaliser sums the fp32 values.
//
// Multi-token queries (QC > 1): a CTA serves QC consecutive query tokens of
// its sequence, so the 16 rows of the tile are (query token r / G, head
// r % G).  Query jq sits at position L - q_len + jq and sees the tokens
// before and at its position (causal among the new tokens): row r masks
// tokens at or past min(partition end, L - q_len + jq + 1).  Rows 8..15 then
// hold real queries: every lane keeps softmax state for rows r and r + 8,
// and P.V runs one n-tile per 8 rows.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_fp16.h>
#include "pkd_decode.cuh"
#include "pkd_ptx.cuh"

namespace pkd {

// ---------------------------------------------------------------- primitives
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// d += A . B for one m16n8k16 tile; A rows 8..15 are zero (a1 = a3 = 0).
__device__ __forceinline__ void mma_16816_top(float (&d)[4], uint32_t a0, uint32_t a2, uint32_t b0,
                                              uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
}

// d += A . B for one full m16n8k16 tile.
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Four E4M3 bytes -> two fp16 pairs: bytes (0, 1) -> lo, bytes (2, 3) -> hi,
// the lower byte of each pair in the lower half (exact: every E4M3 value is
// an fp16 value).
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t x, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 l, h;\n\t"
      "mov.b32 {l, h}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, l;\n\t"
      "cvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(x));
}

// An ldmatrix.trans register of E4M3 data holds bytes (t0 d0, t0 d1, t1 d0,
// t1 d1) for tokens t0 < t1 and dims d0 < d1; regroup to (t0 d0, t1 d0,
// t0 d1, t1 d1) and convert: d0 -> (t0, t1) fp16 pair, d1 -> the same.
__device__ __forceinline__ void e4m3_tpair(uint32_t x, uint32_t& d0, uint32_t& d1) {
  uint32_t y;
  asm("prmt.b32 %0, %1, 0, 0x3120;" : "=r"(y) : "r"(x));
  e4m3x4_to_f16x2x2(y, d0, d1);
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// 3-D tiled tensor copy of the box at (x, y, z) into shared memory at `dst`,
// completing its bytes on `bar`; x (innermost, elements) is a multiple of 64.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* tmap, uint64_t* bar, int x,
                                            int y, int z, const L2Hints& h) {
  if (h.on) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar)),
        "l"(h.evict_first)
        : "memory");
  } else {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
  }
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// Query tokens per CTA of the multi-token kernel for group size G.
constexpr int mma_query_chunk(int G) { return 16 / G; }

// ---------------------------------------------------------------- layout
// QC: query tokens per CTA (1 = single-query decode); KVB: bytes per K/V
// element (2: fp16, 1: E4M3 with per-cache scales); CPS: resident CTAs per
// SM the build targets (0: the cache type's default).
template <int D, int BS, int G, int QC, int KVB = 2, int CPS = 0>
struct MmaTraits {
  static_assert(D == 64 || D == 128, "head_dim");
  static_assert(BS == 16 || BS == 32, "block_size");
  static_assert(G >= 1 && G <= 8, "group size");
  static constexpr int ROWS = G * QC;          // query rows of the 16-row tile in use
  static_assert(QC >= 1 && ROWS <= 16, "the CTA's queries fill one 16-row tile");
  static constexpr int NT = ROWS > 8 ? 2 : 1;  // 8-row halves in use (P.V n-tiles)
  static constexpr int NW = 4;
  static constexpr int THREADS = NW * 32;
  // Three CTAs per SM with 64 KiB rings: more warps to hide the latency of
  // the ldmatrix -> mma -> softmax chains.  Against two CTAs with 96 KiB
  // rings this measured 1.24-1.29x faster with E4M3 caches (half the bytes
  // per token, so twice the tokens per warp) and, with fp16, up to 1.02x on
  // single-query decode and 1.05-1.21x on multi-token queries.  Single-query
  // E4M3 grids of many waves go to four CTAs per SM (48 KiB rings, one QK
  // chain so the state fits in 128 registers): 2-9% faster there, but slower
  // where a few waves of long CTAs bound the grid.
  static constexpr int MIN_BLOCKS = CPS ? CPS : 3;
  static constexpr int RING_KIB = MIN_BLOCKS >= 4 ? 48 : (MIN_BLOCKS == 3 ? 64 : 96);
  static constexpr int QK_CHAINS = MIN_BLOCKS >= 4 ? 1 : 2;  // independent accumulator chains per QK n-tile
  static constexpr bool F8 = KVB == 1;
  static constexpr int KSTEPS = D / 16;       // QK k-steps and PV m-tiles
  // A box is 16 rows of BOX_ROWB bytes: 64 fp16 columns, or a whole E4M3 row
  static constexpr int BOX_X = F8 ? D : 64;               // elements per box row
  static constexpr int BOX_ROWB = BOX_X * KVB;            // 128, or 64 for E4M3 at D = 64
  static constexpr int SWZ_MASK = BOX_ROWB == 128 ? 7 : 3;  // 128- or 64-byte swizzle
  static constexpr int CHUNKS = BOX_ROWB / 16;            // 16-byte chunks per box row
  static constexpr int NBOX = D / BOX_X;                  // boxes per 16-row sub-tile
  static constexpr int BOX_BYTES = 16 * BOX_ROWB;         // one swizzled box
  static constexpr int SUB_BYTES = NBOX * BOX_BYTES;      // K (or V) of one sub-tile
  static constexpr int SLOT_BYTES = 2 * SUB_BYTES;        // K then V
  static constexpr int TILE_BYTES = BS * D * KVB;         // one (block, head) tile in HBM
  static constexpr int SW_RAW = (RING_KIB * 1024) / (NW * SLOT_BYTES);
  static constexpr int SW = SW_RAW > 8 ? 8 : (SW_RAW < 2 ? 2 : SW_RAW);
  static constexpr int RING_BYTES = NW * SW * SLOT_BYTES;
  // merge area: m, mt, l as [NW][16] each, then acc [NW][ROWS][D]
  static constexpr int MRG_ACC_OFF = 3 * NW * 16;  // floats (a multiple of 4)
  static constexpr int MERGE_BYTES = (MRG_ACC_OFF + NW * ROWS * D) * 4;
  static constexpr int MAIN_BYTES = RING_BYTES > MERGE_BYTES ? RING_BYTES : MERGE_BYTES;
  static constexpr int BAR_BYTES = NW * SW * 8;
  // the swizzle needs 1024-byte aligned boxes: the kernel aligns the base
  static constexpr int SMEM_BYTES = 1024 + MAIN_BYTES + BAR_BYTES;
  static_assert(BOX_BYTES % 1024 == 0 && SLOT_BYTES % 1024 == 0, "boxes must stay 1024-byte aligned");
  static_assert(!F8 || (D / 16) % 2 == 0, "E4M3 fragments come in pairs of 16-dim chunks");
  static_assert(MAIN_BYTES % 16 == 0, "barriers must stay 8-byte aligned");
};

// ---------------------------------------------------------------- kernel
template <int D, int BS, int G, int QC, int KVB = 2, int CPS = 0>
__global__ void __launch_bounds__(MmaTraits<D, BS, G, QC, KVB, CPS>::THREADS,
                                  MmaTraits<D, BS, G, QC, KVB, CPS>::MIN_BLOCKS)
    paged_decode_mma_kernel(const __grid_constant__ CUtensorMap tmap_k,
                            const __grid_constant__ CUtensorMap tmap_v, const DecodeParams P) {
  using T = MmaTraits<D, BS, G, QC, KVB, CPS>;
  constexpr bool F8 = T::F8;
  constexpr int NW = T::NW, SW = T::SW, KS = T::KSTEPS, NT = T::NT, ROWS = T::ROWS;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // 1024-byte aligned base for the swizzled boxes
  const uint32_t raw_u32 = smem_u32(smem_raw);
  unsigned char* smem = smem_raw + (((raw_u32 + 1023u) & ~1023u) - raw_u32);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + T::MAIN_BYTES);

  // work item: query chunk fastest, then partition j, then (b, g).  The
  // chunks of one (b, g, j) read the same K/V tiles; launched side by side,
  // all but the first find them in L2.
  const int np_grid = P.max_partitions;
  const int qc = blockIdx.x % P.q_chunks;
  const int rest = blockIdx.x / P.q_chunks;
  // a dependent grid (the split-K merge) may launch once every CTA of this
  // grid has started; it waits for this grid's completion itself
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  int j, b, g;
  if (P.piece_order) {
    // longest first: the grid walks pieces p (all kv heads of a piece side by
    // side); it is the programmatic dependent of the kernel writing the
    // order and waits for it here
    g = rest % P.num_kv_heads;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int piece = P.piece_order[rest / P.num_kv_heads];
    b = piece / np_grid;
    j = piece % np_grid;
  } else {
    j = rest % np_grid;
    const int bg = rest / np_grid;
    g = bg % P.num_kv_heads;
    b = bg / P.num_kv_heads;
  }
  const int L = row_clamped_len<BS>(P, b);
  const int QL = P.q_len;
  const int jq0 = qc * QC;               // first query token of this CTA
  const int nq = min(QC, QL - jq0);      // its query tokens (>= 1)
  const int PS = P.partition_size;
  const int np_b = min((L + PS - 1) / PS, np_grid);  // partitions inside the grid
  const bool final_out = (P.mode == 0) && np_b <= 1;
  const int h0 = g * G;
  const int Hq = P.num_q_heads;
  // output / partial row of tile row rr (< G * nq)
  auto out_row = [&](int rr) { return ((size_t)b * QL + jq0 + rr / G) * Hq + h0 + rr % G; };

  if (L <= 0) {
    if (final_out && j == 0) {
      for (int i = threadIdx.x; i < G * nq * D; i += blockDim.x)
        P.out[out_row(i / D) * D + i % D] = __float2half_rn(0.f);
    }
    return;
  }
  if (j >= np_b) return;

  const int t0 = j * PS;
  // the chunk's last query sees tokens < L - QL + jq0 + nq; nothing past that is read
  const int t1 = min(min(t0 + PS, L), L - QL + jq0 + nq);
  const int nblk = t1 > t0 ? (t1 - t0 + BS - 1) / BS : 0;
  const int32_t* bt = P.block_tables + (size_t)b * P.max_blocks_per_seq + t0 / BS;
  const size_t head_stride = (size_t)T::TILE_BYTES;  // bytes per (block, head) tile
  const size_t block_stride = (size_t)P.num_kv_heads * head_stride;
  const char* kbase = reinterpret_cast<const char*>(P.k_cache) + (size_t)g * head_stride;
  const char* vbase = reinterpret_cast<const char*>(P.v_cache) + (size_t)g * head_stride;
  const int pd = P.prefetch_distance;
  const L2Hints l2h = make_l2_hints(P.l2_hints != 0);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int r = lane / 4;  // tile row (of each 8-row half) in S, dim row of O^T
  const int c = lane % 4;

  // token limit of the lane's rows r + 8 * hf: tokens at or past it are masked
  int lim[NT];
#pragma unroll
  for (int hf = 0; hf < NT; ++hf) {
    const int rr = r + 8 * hf;
    lim[hf] = rr < G * nq ? min(t1, L - QL + jq0 + rr / G + 1) : t1;
  }
  const int lim_min = NT == 2 ? min(lim[0], lim[NT - 1]) : lim[0];

  // Q as A fragments: qa[k] = {row r, row r+8} x {k-slots 2c, 2c+1 | 8+2c, 9+2c}.
  // fp16 K: slot j of step k is dim 16k + j.  E4M3 K: a lane's 4 bytes of a
  // 16-dim chunk are dims 4c .. 4c+3, so slots (2c, 2c+1 | 8+2c, 9+2c) are
  // dims 16k + (4c, 4c+1 | 4c+2, 4c+3); Q follows the same map.
  constexpr int QHI = F8 ? 2 : 8, QMUL = F8 ? 4 : 2;
  uint32_t qa[KS][4];
#pragma unroll
  for (int hf = 0; hf < 2; ++hf) {
    const int rr = r + 8 * hf;
    const bool live = hf < NT && rr < G * nq;
    const __half* qr = P.q + (live ? out_row(rr) * D : 0);
#pragma unroll
    for (int k = 0; k < KS; ++k) {
      qa[k][hf] = live ? *reinterpret_cast<const uint32_t*>(qr + 16 * k + QMUL * c) : 0u;
      qa[k][2 + hf] = live ? *reinterpret_cast<const uint32_t*>(qr + 16 * k + QHI + QMUL * c) : 0u;
    }
  }
  // O^T m-tile k, n-tile hf: [dim 16k + r | 16k + 8 + r] x [row 8hf + 2c | 8hf + 2c + 1]
  float o[KS][NT][4];
#pragma unroll
  for (int k = 0; k < KS; ++k)
#pragma unroll
    for (int hf = 0; hf < NT; ++hf) o[k][hf][0] = o[k][hf][1] = o[k][hf][2] = o[k][hf][3] = 0.f;
  float m[NT], mt[NT], l[NT];  // per row r + 8hf: running shift, exact maximum, sum of p
#pragma unroll
  for (int hf = 0; hf < NT; ++hf) {
    m[hf] = -INFINITY;
    mt[hf] = -INFINITY;
    l[hf] = 0.f;
  }

  // ldmatrix row addresses: lane l addresses row (l & 7) + 8 * (l >> 4) of the
  // sub-tile, 16-byte chunk 2s + ((l >> 3) & 1) for step s; with the swizzle
  // the chunk offset of step s is ((2s & 7) ^ x) * 16, x = chunk bit ^ row % 8.
  uint32_t lm_off[4];
  if constexpr (!F8) {
    const int row = (lane & 7) + 8 * (lane >> 4);
    const int x = ((lane >> 3) & 1) ^ (row & 7);
#pragma unroll
    for (int i = 0; i < 4; ++i) lm_off[i] = row * 128 + (((2 * i) ^ x) << 4);
  } else {
    // E4M3: one ldmatrix.x4 covers chunks (2i, 2i+1) of 16 rows: lane l
    // addresses row (l & 7) + 8 * ((l >> 3) & 1), chunk 2i + (l >> 4)
    const int row = (lane & 7) + 8 * ((lane >> 3) & 1);
    const int swz = ((row * T::BOX_ROWB) >> 7) & T::SWZ_MASK;
#pragma unroll
    for (int i = 0; i < 4; ++i)
      lm_off[i] = row * T::BOX_ROWB + ((((2 * i + (lane >> 4)) & (T::CHUNKS - 1)) ^ swz) << 4);
  }

  uint64_t* full = bars + warp * SW;
  unsigned char* ring = smem + (size_t)warp * SW * T::SLOT_BYTES;
  if (threadIdx.x == 0) {
    prefetch_tensormap(&tmap_k);
    prefetch_tensormap(&tmap_v);
  }
  if (lane == 0) {
    for (int s = 0; s < SW; ++s) mbar_init(&full[s], 1);
    fence_mbarrier_init();
  }
  __syncwarp();

  SubCursor<BS, NW> ic, cc;
  ic.start(warp);
  cc.start(warp);
  auto block_id = [&](int k) { return k < nblk ? bt[k] : -1; };
  int ic_pb = block_id(ic.k);
  int pf_k = warp + NW * pd;
  int pf_pb = pd > 0 ? block_id(pf_k) : -1;
  uint32_t bad_slots = 0;
  auto issue_next = [&](int slot) {
    const bool bad = ic_pb < 0 || ic_pb >= P.num_blocks;
    bad_slots = bad ? (bad_slots | (1u << slot)) : (bad_slots & ~(1u << slot));
    if (lane == 0) {
      if (bad) {
        record_error(P.error_word, kErrBadBlock);
        mbar_arrive(&full[slot]);
      } else {
        const uint32_t dst = smem_u32(ring + (size_t)slot * T::SLOT_BYTES);
        const int y = g * BS + ic.rg * 16;
        mbar_arrive_expect_tx(&full[slot], T::SLOT_BYTES);
#pragma unroll
        for (int hb = 0; hb < T::NBOX; ++hb) {
          tma_load_3d(dst + hb * T::BOX_BYTES, &tmap_k, &full[slot], T::BOX_X * hb, y, ic_pb, l2h);
          tma_load_3d(dst + T::SUB_BYTES + hb * T::BOX_BYTES, &tmap_v, &full[slot], T::BOX_X * hb, y, ic_pb,
                      l2h);
        }
      }
    }
    if (ic.rg == 0 && pd > 0) {
      if (lane == 0 && pf_pb >= 0 && pf_pb < P.num_blocks) {
        prefetch_l2_bulk(kbase + (size_t)pf_pb * block_stride, T::TILE_BYTES, l2h);
        prefetch_l2_bulk(vbase + (size_t)pf_pb * block_stride, T::TILE_BYTES, l2h);
      }
      pf_k += NW;
      pf_pb = block_id(pf_k);
    }
    const int k_before = ic.k;
    ic.advance(t0, t1);
    if (ic.k != k_before) ic_pb = block_id(ic.k);
  };
  int issued = 0;  // sub-tiles issued into the ring so far
  for (int s = 0; s < SW && ic.live(nblk); ++s, ++issued) issue_next(s);

  for (int u = 0; cc.live(nblk); ++u) {
    const int slot = u % SW;
    const bool bad = (bad_slots >> slot) & 1u;
    if (!mbar_wait_bounded(&full[slot], (u / SW) & 1, P.timeout_ns)) {
      if (lane == 0) record_error(P.error_word, kErrTimeout);
      // let the copies still in flight land (each wait bounded again)
      for (int v = u + 1; v < issued; ++v) mbar_wait_bounded(&full[v % SW], (v / SW) & 1, P.timeout_ns);
      break;
    }
    if (!bad) {
      const int base = t0 + cc.k * BS + cc.rg * 16;  // token of the sub-tile's row 0
      const int valid = min(16, t1 - base);
      unsigned char* kslot = ring + (size_t)slot * T::SLOT_BYTES;
      const uint32_t ks = smem_u32(kslot);
      const uint32_t vs = ks + T::SUB_BYTES;
      if (valid < 16) {
        // rows past the CTA's tokens may hold anything (NaN included): zero the
        // V rows so that p = 0 times them stays 0; masked K rows get -inf below
        for (int i = lane; i < (16 - valid) * T::NBOX * T::CHUNKS; i += 32) {
          const int row = valid + i / (T::NBOX * T::CHUNKS);
          const int rest8 = i % (T::NBOX * T::CHUNKS);
          *reinterpret_cast<uint4*>(kslot + T::SUB_BYTES + (rest8 / T::CHUNKS) * T::BOX_BYTES +
                                    row * T::BOX_ROWB + (rest8 % T::CHUNKS) * 16) = make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();  // ordered before the next tensor copy into this slot
        __syncwarp();
      }
      // ---- S = Q K^T: two n-tiles (tokens 0..7, 8..15); the k-steps alternate
      // between QK_CHAINS accumulators so that dependent MMAs do not form one
      // long chain
      constexpr int QC_ = T::QK_CHAINS;
      float sa[QC_][4], sb[QC_][4];
#pragma unroll
      for (int ch = 0; ch < QC_; ++ch)
#pragma unroll
        for (int e = 0; e < 4; ++e) sa[ch][e] = sb[ch][e] = 0.f;
      auto qk = [&](int k, uint32_t b00, uint32_t b01, uint32_t b10, uint32_t b11) {
        if constexpr (NT == 1) {
          mma_16816_top(sa[k % QC_], qa[k][0], qa[k][2], b00, b01);
          mma_16816_top(sb[k % QC_], qa[k][0], qa[k][2], b10, b11);
        } else {
          mma_16816(sa[k % QC_], qa[k], b00, b01);
          mma_16816(sb[k % QC_], qa[k], b10, b11);
        }
      };
      if constexpr (!F8) {
#pragma unroll
        for (int k = 0; k < KS; ++k) {
          uint32_t kb[4];
          ldsm_x4(ks + (k / 4) * T::BOX_BYTES + lm_off[k % 4], kb);
          qk(k, kb[0], kb[1], kb[2], kb[3]);
        }
      } else {
        // kb: (tokens 0-7, chunk 2i), (8-15, 2i), (0-7, 2i+1), (8-15, 2i+1)
#pragma unroll
        for (int i = 0; i < KS / 2; ++i) {
          uint32_t kb[4];
          ldsm_x4(ks + lm_off[i], kb);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t b00, b01, b10, b11;
            e4m3x4_to_f16x2x2(kb[2 * h], b00, b01);
            e4m3x4_to_f16x2x2(kb[2 * h + 1], b10, b11);
            qk(2 * i + h, b00, b01, b10, b11);
          }
        }
      }
      float s0[4], s1[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        s0[e] = sa[0][e];
        s1[e] = sb[0][e];
#pragma unroll
        for (int ch = 1; ch < QC_; ++ch) {
          s0[e] += sa[ch][e];
          s1[e] += sb[ch][e];
        }
      }
      // ---- online softmax of rows r + 8hf over tokens 2c, 2c+1, 8+2c, 9+2c
      float sc[NT][4];
#pragma unroll
      for (int hf = 0; hf < NT; ++hf) {
        sc[hf][0] = s0[2 * hf] * P.scale_log2;
        sc[hf][1] = s0[2 * hf + 1] * P.scale_log2;
        sc[hf][2] = s1[2 * hf] * P.scale_log2;
        sc[hf][3] = s1[2 * hf + 1] * P.scale_log2;
      }
      if (base + 16 > lim_min) {
#pragma unroll
        for (int hf = 0; hf < NT; ++hf) {
          const int lt = lim[hf] - base;  // tokens of the sub-tile this row sees
          if (2 * c >= lt) sc[hf][0] = -INFINITY;
          if (2 * c + 1 >= lt) sc[hf][1] = -INFINITY;
          if (8 + 2 * c >= lt) sc[hf][2] = -INFINITY;
          if (9 + 2 * c >= lt) sc[hf][3] = -INFINITY;
        }
      }
      float lmax[NT];
      bool need = false;
#pragma unroll
      for (int hf = 0; hf < NT; ++hf) {
        lmax[hf] = fmaxf(fmaxf(sc[hf][0], sc[hf][1]), fmaxf(sc[hf][2], sc[hf][3]));
        mt[hf] = fmaxf(mt[hf], lmax[hf]);
        need |= lmax[hf] > m[hf] + kLazyTau;
      }
      if (__any_sync(0xffffffffu, need)) {
#pragma unroll
        for (int hf = 0; hf < NT; ++hf) {
          float mx = fmaxf(lmax[hf], __shfl_xor_sync(0xffffffffu, lmax[hf], 1));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
          const float mn = fmaxf(m[hf], mx);
          const float alpha = (mn == -INFINITY) ? 1.f : ex2_approx(m[hf] - mn);
          l[hf] *= alpha;
          m[hf] = mn;
          // O^T columns 8hf + 2c, 8hf + 2c + 1: their shifts live in lanes 8c, 8c + 4
          const float a_lo = __shfl_sync(0xffffffffu, alpha, 8 * c);
          const float a_hi = __shfl_sync(0xffffffffu, alpha, 8 * c + 4);
#pragma unroll
          for (int k = 0; k < KS; ++k) {
            o[k][hf][0] *= a_lo;
            o[k][hf][1] *= a_hi;
            o[k][hf][2] *= a_lo;
            o[k][hf][3] *= a_hi;
          }
        }
      }
      uint32_t pb[NT][2];
#pragma unroll
      for (int hf = 0; hf < NT; ++hf) {
        // a row that has seen no token yet keeps m = -inf: shift by 0 so that
        // its masked scores give p = 0 rather than NaN
        const float mu = m[hf] == -INFINITY ? 0.f : m[hf];
        const float p0 = ex2_approx(sc[hf][0] - mu), p1 = ex2_approx(sc[hf][1] - mu);
        const float p2 = ex2_approx(sc[hf][2] - mu), p3 = ex2_approx(sc[hf][3] - mu);
        l[hf] += (p0 + p1) + (p2 + p3);
        pb[hf][0] = pack_half2(p0, p1);  // P^T[tokens 2c, 2c+1][row 8hf + r]
        pb[hf][1] = pack_half2(p2, p3);  // P^T[tokens 8+2c, 9+2c][row 8hf + r]
      }
      // ---- O^T += V^T P^T, one m-tile of 16 dims per step
      if constexpr (!F8) {
#pragma unroll
        for (int k = 0; k < KS; ++k) {
          uint32_t va[4];
          ldsm_x4_trans(vs + (k / 4) * T::BOX_BYTES + lm_off[k % 4], va);
#pragma unroll
          for (int hf = 0; hf < NT; ++hf) mma_16816(o[k][hf], va, pb[hf][0], pb[hf][1]);
        }
      } else {
        // vt: (tokens 0-7, chunk 2i), (8-15, 2i), (0-7, 2i+1), (8-15, 2i+1), each
        // register (token pair) x (dim pair); m-tile rows r and r + 8 are dims
        // 2r and 2r + 1 of the chunk
#pragma unroll
        for (int i = 0; i < KS / 2; ++i) {
          uint32_t vt[4];
          ldsm_x4_trans(vs + lm_off[i], vt);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t va[4];
            e4m3_tpair(vt[2 * h], va[0], va[1]);
            e4m3_tpair(vt[2 * h + 1], va[2], va[3]);
#pragma unroll
            for (int hf = 0; hf < NT; ++hf) mma_16816(o[2 * i + h][hf], va, pb[hf][0], pb[hf][1]);
          }
        }
      }
    }
    __syncwarp();
    if (ic.live(nblk)) {
      if (lane == 0) fence_proxy_async_smem();  // our reads of the slot precede the next copy into it
      issue_next(slot);
      ++issued;
    }
    cc.advance(t0, t1);
  }

  // ------------------------------------------------------------------ merge
  __syncthreads();  // every warp is done with the ring that the merge area reuses
  float* mrg = reinterpret_cast<float*>(smem);
  float* mrg_m = mrg;                   // [NW][16] running shift
  float* mrg_mt = mrg + NW * 16;        // [NW][16] exact maximum
  float* mrg_l = mrg + 2 * NW * 16;     // [NW][16]
  float* mrg_acc = mrg + T::MRG_ACC_OFF;  // [NW][ROWS][D]
#pragma unroll
  for (int hf = 0; hf < NT; ++hf) {
    float lv = l[hf] + __shfl_xor_sync(0xffffffffu, l[hf], 1);
    lv += __shfl_xor_sync(0xffffffffu, lv, 2);
    float mx = fmaxf(mt[hf], __shfl_xor_sync(0xffffffffu, mt[hf], 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    if (c == 0) {
      mrg_m[warp * 16 + 8 * hf + r] = m[hf];
      mrg_mt[warp * 16 + 8 * hf + r] = mx;
      mrg_l[warp * 16 + 8 * hf + r] = lv;
    }
    float* acc = mrg_acc + warp * ROWS * D;
    const int ra = 8 * hf + 2 * c;
    // dims of m-tile rows r and r + 8: fp16 16k + r, 16k + 8 + r; E4M3 16k + 2r, 16k + 2r + 1
    const int d_lo = F8 ? 2 * r : r, d_hi = F8 ? 2 * r + 1 : 8 + r;
#pragma unroll
    for (int k = 0; k < KS; ++k) {
      if (ra < ROWS) {
        acc[ra * D + 16 * k + d_lo] = o[k][hf][0];
        acc[ra * D + 16 * k + d_hi] = o[k][hf][2];
      }
      if (ra + 1 < ROWS) {
        acc[(ra + 1) * D + 16 * k + d_lo] = o[k][hf][1];
        acc[(ra + 1) * D + 16 * k + d_hi] = o[k][hf][3];
      }
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < G * nq * D; i += blockDim.x) {
    const int rr = i / D, d = i % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, mrg_mt[w * 16 + rr]);  // the exact maximum
    float Z = 0.f, O = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float mw = mrg_m[w * 16 + rr];
      const float cw = (mw == -INFINITY) ? 0.f : ex2_approx(mw - M);
      Z = fmaf(cw, mrg_l[w * 16 + rr], Z);
      O = fmaf(cw, mrg_acc[(w * ROWS + rr) * D + d], O);
    }
    if constexpr (F8) O *= P.v_scale;  // V = code * v_scale
    const size_t row = out_row(rr);
    if (final_out) {
      P.out[row * D + d] = __float2half_rn(Z > 0.f ? O / Z : 0.f);  // Z = 0: the query saw no token
    } else {
      const size_t pidx = row * P.max_partitions + j;
      P.tmp_out[pidx * D + d] = O;
      if (d == 0) {
        P.max_logits[pidx] = M * 0.69314718055994530942f;  // log2 units -> natural; -inf if empty
        P.exp_sums[pidx] = Z;
      }
    }
  }
}

}  // namespace pkd
