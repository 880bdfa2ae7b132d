// pkd_decode.cuh -- paged single-query decode attention kernels (sm_103a).
//
// One CTA per (sequence b, kv head g, context partition j).  The CTA reads
// every K/V tile of its token range once and serves all G = Hq/Hkv query
// heads of the group from it.  NW compute warps take the partition's blocks
// in a stride-NW order (warp w: blocks w, w+NW, w+2NW, ...), the loop of
// Algorithm 1 in the review "Accelerating LLM Inference Throughput via
// Asynchronous KV Cache Prefetching" (section 3.4), each warp with its own
// online-softmax state; the warps are merged at the end.
//
// Per 16-row group of a block, with LPR = D/8 lanes per row (16 bytes = 8
// halves per lane) and RPW = 32/LPR rows per warp-wide access:
//   QK:  lane (row-half rh, slice ds) holds q[h][8*ds .. 8*ds+8) in fp32
//        registers for every head h; for each of its TPL = 16/RPW rows it
//        forms 8-element partial dot products for all G heads (packed fp32
//        FMAs over pairs of d), then a transpose-reduce over the LPR lanes
//        of a row leaves the full score of one row in lanes (2i, 2i+1).
//   softmax: fp32 online softmax in the log2 domain with a lazy running
//        max (rescale only when a score exceeds the max by more than TAU).
//   PV:  the same lane mapping reads V rows; p comes from a per-warp
//        shared-memory row [16][8] written by the lanes holding the scores.
//
// Data paths (template VARIANT):
//   NO_PREFETCH  each warp loads its current block with 16-byte global loads
//                straight into the registers the arithmetic uses (the paper's
//                baseline flow, section 3.2).
//   L2_PREFETCH  as NO_PREFETCH, and lane 0 of each warp issues
//                cp.async.bulk.prefetch.L2 for the K and V tiles of the block
//                the same warp will take `prefetch_distance` iterations later
//                (section 3.4 Algorithm 1 prefetches block_idx + w; section
//                4.1 applies the same to V blocks).
//   TMA_STAGED   a producer warp streams K and V tiles with 1-D bulk copies
//                (cp.async.bulk) into a ring of shared-memory slots completed
//                on mbarriers, and prefetches tiles beyond the ring to L2.
//                The blog post "KV Cache Prefetching：三层预取如何隐藏 KV
//                访问延迟", section 2.3, suggests this pairing of SRAM staging
//                with HBM->L2 prefetch.
#pragma once
#include <cstdint>
#include <cuda_fp16.h>
#include "pkd_ptx.cuh"

namespace pkd {

enum Variant : int { kNoPrefetch = 1, kL2Prefetch = 2, kTmaStaged = 3 };

constexpr float kLazyTau = 8.0f;  // log2-domain slack of the lazy running max
constexpr uint32_t kErrBadBlock = 1u;
constexpr uint32_t kErrTimeout = 2u;

struct DecodeParams {
  const __half* q;
  const __half* k_cache;
  const __half* v_cache;
  const int32_t* block_tables;
  const int32_t* context_lens;
  __half* out;          // final output; written for sequences with <= 1 partition (mode 0)
  float* tmp_out;       // [B][Hq][NP][D] partials (may be null when nothing splits)
  float* max_logits;    // [B][Hq][NP]
  float* exp_sums;      // [B][Hq][NP]
  int* error_word;      // nullable
  int num_seqs, num_q_heads, num_kv_heads, num_blocks, max_blocks_per_seq;
  int partition_size;   // tokens per partition (multiple of 32)
  int max_partitions;   // NP: grid stride and partial-array stride
  int mode;             // 0: final out when one partition, partials otherwise; 1: partials always
  int q_len;            // query tokens per sequence (1: single-query decode; > 1 tensor-core path only)
  int q_chunks;         // query chunks per (sequence, kv head) in the grid (1 when q_len == 1)
  float v_scale;        // E4M3 caches: V value = code * v_scale (the K scale is folded into scale_log2)
  float scale_log2;     // softmax scale * log2(e)
  int prefetch_distance;
  int l2_hints;         // 1: evict_first on consuming loads/copies, evict_last on prefetches
  unsigned long long timeout_ns;
  const int32_t* piece_order;  // nullable: grid piece p -> b * NP + j (longest first); tensor-core path only
  int parts_per_cta;           // tcgen05 path: consecutive partitions per CTA (0 or 1: one; needs no piece order)
  int tail_split;              // tcgen05 path with piece_order: pieces are b * 4 + a kPiece* code (a split tail)
};

// A grid walked longest first whose last round would be short splits its
// shortest sequences in two (the tcgen05 path; piece_order_kernel chooses
// them).  Piece codes, piece = b * 4 + code (-1: no piece):
constexpr int kPieceWhole = 0;       // the whole sequence, written to out
constexpr int kPieceFirstHalf = 1;   // tokens [0, tail_half_partition(L)), a partial
constexpr int kPieceSecondHalf = 2;  // the rest, a partial
// The partition of such a split sequence of L tokens: half of it, rounded up
// to whole 64-token tiles (so a sequence of at most 64 tokens stays whole).
__host__ __device__ __forceinline__ int tail_half_partition(int L) { return ((L + 1) / 2 + 63) / 64 * 64; }

template <int D, int BS, int G, int VARIANT>
struct DecodeTraits {
  static_assert(D == 64 || D == 128, "head_dim");
  static_assert(BS == 16 || BS == 32, "block_size");
  static_assert(G >= 1 && G <= 8, "group size");
  static constexpr int LPR = D / 8;         // lanes per row
  static constexpr int RPW = 32 / LPR;      // rows per warp-wide access
  static constexpr int TPL = 16 / RPW;      // rows per lane per 16-row group
  static constexpr int RG = BS / 16;        // 16-row groups per block
  static constexpr int TILE_ELEMS = BS * D; // one (block, head) tile
  static constexpr int TILE_BYTES = TILE_ELEMS * 2;
  static constexpr bool kTma = VARIANT == kTmaStaged;
  // CTAs of 4 warps.  Resident CTAs per SM: 2 (up to 255 registers a
  // thread, 2 warps per SM sub-partition), or 3 for the staged variant at
  // group sizes 2..5, whose state fits in 168 registers; more warps hide more
  // latency, and several CTAs let one CTA's start-up overlap another's tail.
  static constexpr int NW = 4;
  static constexpr int MIN_BLOCKS = (kTma && G >= 2 && G <= 5) ? 3 : 2;
  static constexpr int THREADS = NW * 32;
  // Staging unit of the staged variant: one 16-row group of K and of V
  // (each 16*D contiguous halves).  Every warp owns SW slots of its own:
  // about 96 KiB of slots per CTA at 2 CTAs per SM, 64 KiB at 3.
  static constexpr int SUB_ELEMS = 16 * D;
  static constexpr int SUB_BYTES = SUB_ELEMS * 2;
  static constexpr int SLOT_BYTES = 2 * SUB_BYTES;
  static constexpr int SW_RAW = ((MIN_BLOCKS == 3 ? 64 : 96) * 1024) / (NW * SLOT_BYTES);
  static constexpr int SW = kTma ? (SW_RAW > 8 ? 8 : (SW_RAW < 2 ? 2 : SW_RAW)) : 0;
  static constexpr int RING_BYTES = NW * SW * SLOT_BYTES;
  static constexpr int P_BYTES = NW * 16 * 8 * 8;           // per-warp p rows [16][8] as (p, p)
  // merge area: per warp the running shift m, the exact maximum mt and l
  // ([NW][G] each), then acc [NW][G][D] on a 16-byte boundary
  static constexpr int MRG_ACC_OFF = (3 * NW * G + 3) / 4 * 4;  // floats
  static constexpr int MERGE_BYTES = (MRG_ACC_OFF + NW * G * D) * 4;
  static constexpr int BAR_BYTES = NW * SW * 8;
  // layout: [ring / merge area][p rows][barriers]; the merge reuses the ring
  static constexpr int MAIN_BYTES = RING_BYTES > MERGE_BYTES ? RING_BYTES : MERGE_BYTES;
  static constexpr int SMEM_BYTES = MAIN_BYTES + P_BYTES + BAR_BYTES;
  // every shared-memory region is accessed with 16-byte (and 8-byte barrier) operations
  static_assert(MAIN_BYTES % 16 == 0 && P_BYTES % 16 == 0, "shared-memory regions must stay 16-byte aligned");
  static_assert(SLOT_BYTES % 16 == 0, "bulk-copy slots must be 16-byte aligned");
};

// ---------------------------------------------------------------------------
__device__ __forceinline__ void record_error(int* err, uint32_t bits) {
  if (err) atomicOr(reinterpret_cast<unsigned*>(err), bits);
}

// Sequence b's length as the decode kernels read it.  A length past the
// block-table row (max_blocks_per_seq * BS tokens) is cut to the row and
// reported as kErrBadBlock, so no table entry past the row is ever read.
template <int BS>
__device__ __forceinline__ int row_clamped_len(const DecodeParams& P, int b) {
  const int L = P.context_lens[b];
  const int row = P.max_blocks_per_seq * BS;
  if (L > row) {
    record_error(P.error_word, kErrBadBlock);
    return row;
  }
  return L;
}

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  // 16-byte global load; the KV stream is read once, so do not allocate in L1
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ uint4 ldg_stream(const void* p, const L2Hints& h) {
  if (!h.on) return ldg_stream(p);
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p), "l"(h.evict_first));
  return r;
}

__device__ __forceinline__ uint4 lds128(const void* p) {
  return *reinterpret_cast<const uint4*>(p);
}

// 2^x by the SFU approximation (ex2.approx, relative error about 2^-22;
// ex2(-inf) = +0); subnormal results flush to zero, which only drops weights
// below 2^-126 of the running maximum.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float2 h2f2(uint32_t u) {
  return __half22float2(*reinterpret_cast<const __half2*>(&u));
}

// ---------------------------------------------------------------------------
// Per-warp state and the per-16-row-group arithmetic.
template <int D, int BS, int G, int VARIANT>
struct WarpDecoder {
  using T = DecodeTraits<D, BS, G, VARIANT>;
  static constexpr int LPR = T::LPR, RPW = T::RPW, TPL = T::TPL;

  float2 q2[G][4];   // q[h][8*ds + 2c .. +2) for c < 4
  float2 acc[G][4];  // sum_t p_t v_t[8*ds + 2c .. +2) over this lane's rows
  float m[G];        // running shift (log2 domain), warp-uniform; lags the maximum by <= TAU
  float mt[G];       // exact maximum of the scores this lane has seen (log2 domain)
  float l[G];        // running sum of p over this lane's score slots
  int lane, rh, ds;
  int perm;          // this lane's row order: local row i is row i ^ perm of its half

  __device__ __forceinline__ void init(const __half* qrow0, int lane_) {
    lane = lane_;
    rh = lane / LPR;
    ds = lane % LPR;
    perm = (ds >> 1) & (TPL - 1);
#pragma unroll
    for (int h = 0; h < G; ++h) {
      uint4 u = *reinterpret_cast<const uint4*>(qrow0 + (size_t)h * D + ds * 8);
      q2[h][0] = h2f2(u.x);
      q2[h][1] = h2f2(u.y);
      q2[h][2] = h2f2(u.z);
      q2[h][3] = h2f2(u.w);
      m[h] = -INFINITY;
      mt[h] = -INFINITY;
      l[h] = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[h][c] = make_float2(0.f, 0.f);
    }
  }

  // Row (within a 16-row group) that this lane reads at local index i.
  __device__ __forceinline__ int k_row(int i) const { return RPW * (i ^ perm) + rh; }

  // Scores of one 16-row group.  krow(i) gives the 16 bytes of row k_row(i)
  // at slice ds.  Returns, in s2[h], the log2-domain score of row
  // my_score_row() (duplicated in lanes ds, ds^1).
  //
  // The transpose-reduce: at each level the partner lane (lane ^ mask) has
  // the opposite bit of `perm`, so its local index j + n/2 holds the same row
  // as our local index j; every lane keeps part[j] and sends part[j + n/2],
  // with no lane-dependent selects.
  template <typename KRow>
  __device__ __forceinline__ void scores(KRow krow, float scale_log2, float (&s2)[G]) {
    float part[TPL][G];
#pragma unroll
    for (int i = 0; i < TPL; ++i) {
      uint4 u = krow(i);
      float2 k0 = h2f2(u.x), k1 = h2f2(u.y), k2 = h2f2(u.z), k3 = h2f2(u.w);
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float2 a = fmul2(q2[h][0], k0);
        a = ffma2(q2[h][1], k1, a);
        a = ffma2(q2[h][2], k2, a);
        a = ffma2(q2[h][3], k3, a);
        part[i][h] = a.x + a.y;
      }
    }
    // transpose-reduce: halve the row set at lane masks LPR/2, LPR/4, ...
#pragma unroll
    for (int lvl = 0; (TPL >> lvl) > 1; ++lvl) {
      const int n = TPL >> lvl;
      const int mask = (LPR / 2) >> lvl;
#pragma unroll
      for (int j = 0; j < n / 2; ++j) {
#pragma unroll
        for (int h = 0; h < G; ++h)
          part[j][h] += __shfl_xor_sync(0xffffffffu, part[j + n / 2][h], mask);
      }
    }
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float v = part[0][h] + __shfl_xor_sync(0xffffffffu, part[0][h], 1);
      s2[h] = v * scale_log2;
    }
  }

  __device__ __forceinline__ int my_score_row() const { return RPW * perm + rh; }

  // Online-softmax update with scores s2 (masked rows already -inf); writes
  // p into prow as (p, p) pairs, [16 rows][8 heads][2], visible to the warp.
  __device__ __forceinline__ void softmax_update(float (&s2)[G], float* prow) {
    bool need = false;
#pragma unroll
    for (int h = 0; h < G; ++h) need |= s2[h] > m[h] + kLazyTau;
    if (__any_sync(0xffffffffu, need)) {
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float mx = s2[h];
#pragma unroll
        for (int msk = 2; msk < 32; msk <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, msk));
        const float mn = fmaxf(m[h], mx);
        const float alpha = (mn == -INFINITY) ? 1.f : ex2_approx(m[h] - mn);  // m = -inf -> 0
        l[h] *= alpha;
        const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[h][c] = fmul2(acc[h][c], a2);
        m[h] = mn;
      }
    }
    float p[8];
#pragma unroll
    for (int h = 0; h < 8; ++h) p[h] = 0.f;
#pragma unroll
    for (int h = 0; h < G; ++h) {
      p[h] = ex2_approx(s2[h] - m[h]);
      l[h] += p[h];
      mt[h] = fmaxf(mt[h], s2[h]);
    }
    if ((ds & 1) == 0) {
      float4* dst = reinterpret_cast<float4*>(prow + my_score_row() * 16);
#pragma unroll
      for (int h2 = 0; h2 < (G + 1) / 2; ++h2) dst[h2] = make_float4(p[2 * h2], p[2 * h2], p[2 * h2 + 1], p[2 * h2 + 1]);
    }
    __syncwarp();
  }

  // acc += p * V for the rows of one 16-row group; vrow(i) as krow.
  // Rows at or past `valid` (0..16) are skipped (their V may be garbage).
  template <typename VRow>
  __device__ __forceinline__ void accumulate(VRow vrow, const float* prow, int valid) {
    // rows are software-pipelined: row i+1's V and p loads are issued before
    // row i's FMAs, which hides the load latency
    constexpr int NH2 = (G + 1) / 2;
    auto load_row = [&](int i, uint4& v, float4 (&pp)[NH2]) {
      v = vrow(i);
      const int r = RPW * i + rh;
#pragma unroll
      for (int h2 = 0; h2 < NH2; ++h2) pp[h2] = *reinterpret_cast<const float4*>(prow + r * 16 + 4 * h2);
    };
    auto fma_row = [&](const uint4& v4, const float4 (&pp)[NH2]) {
      const float2 vv[4] = {h2f2(v4.x), h2f2(v4.y), h2f2(v4.z), h2f2(v4.w)};
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float2 pv = (h & 1) ? make_float2(pp[h / 2].z, pp[h / 2].w) : make_float2(pp[h / 2].x, pp[h / 2].y);
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[h][c] = ffma2(pv, vv[c], acc[h][c]);
      }
    };
    if (valid >= 16) {
      uint4 vc;
      float4 pc[NH2];
      load_row(0, vc, pc);
#pragma unroll
      for (int i = 0; i < TPL; ++i) {
        uint4 vn;
        float4 pn[NH2];
        if (i + 1 < TPL) load_row(i + 1, vn, pn);
        fma_row(vc, pc);
        if (i + 1 < TPL) {
          vc = vn;
#pragma unroll
          for (int h2 = 0; h2 < NH2; ++h2) pc[h2] = pn[h2];
        }
      }
    } else {
#pragma unroll
      for (int i = 0; i < TPL; ++i) {
        if (RPW * i + rh < valid) {
          uint4 vc;
          float4 pc[NH2];
          load_row(i, vc, pc);
          fma_row(vc, pc);
        }
      }
    }
    __syncwarp();
  }

  // Reduce this warp's state and store (m, l, acc) to the merge area.
  __device__ __forceinline__ void store_warp(float* mrg_m, float* mrg_mt, float* mrg_l, float* mrg_acc) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float lv = (ds & 1) ? 0.f : l[h];
      float mx = mt[h];
#pragma unroll
      for (int msk = 1; msk < 32; msk <<= 1) {
        lv += __shfl_xor_sync(0xffffffffu, lv, msk);
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, msk));
      }
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float2 a = acc[h][c];
#pragma unroll
        for (int msk = LPR; msk < 32; msk <<= 1) {
          a.x += __shfl_xor_sync(0xffffffffu, a.x, msk);
          a.y += __shfl_xor_sync(0xffffffffu, a.y, msk);
        }
        acc[h][c] = a;
      }
      if (lane == 0) {
        mrg_m[h] = m[h];
        mrg_mt[h] = mx;
        mrg_l[h] = lv;
      }
      if (rh == 0) {
        float4* dst = reinterpret_cast<float4*>(mrg_acc + h * D + ds * 8);
        dst[0] = make_float4(acc[h][0].x, acc[h][0].y, acc[h][1].x, acc[h][1].y);
        dst[1] = make_float4(acc[h][2].x, acc[h][2].y, acc[h][3].x, acc[h][3].y);
      }
    }
  }
};

// ---------------------------------------------------------------------------
// The block/row-group sequence one warp walks: blocks warp, warp+NW, ...
// and, inside each block, its 16-row groups that hold at least one token.
template <int BS, int NW>
struct SubCursor {
  int k, rg;
  __device__ __forceinline__ void start(int warp) { k = warp; rg = 0; }
  __device__ __forceinline__ bool live(int nblk) const { return k < nblk; }
  // tokens_left(k) = tokens of block k inside the partition
  __device__ __forceinline__ void advance(int t0, int t1) {
    ++rg;
    if (rg * 16 >= BS || t0 + k * BS + rg * 16 >= t1) {
      rg = 0;
      k += NW;
    }
  }
};

template <int D, int BS, int G, int VARIANT>
__global__ void __launch_bounds__(DecodeTraits<D, BS, G, VARIANT>::THREADS,
                                  DecodeTraits<D, BS, G, VARIANT>::MIN_BLOCKS)
    paged_decode_kernel(const DecodeParams P) {
  using T = DecodeTraits<D, BS, G, VARIANT>;
  constexpr int NW = T::NW, RPW = T::RPW, TPL = T::TPL;
  extern __shared__ __align__(128) unsigned char smem[];
  float* p_rows = reinterpret_cast<float*>(smem + T::MAIN_BYTES);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + T::MAIN_BYTES + T::P_BYTES);

  // work item: j fastest so a sequence's partitions run side by side
  const int np_grid = P.max_partitions;
  const int j = blockIdx.x % np_grid;
  const int bg = blockIdx.x / np_grid;
  const int g = bg % P.num_kv_heads;
  const int b = bg / P.num_kv_heads;
  // the split-K merge (a programmatic dependent) may launch once every CTA has started
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int L = row_clamped_len<BS>(P, b);
  const int PS = P.partition_size;
  // partitions of the sequence inside the grid (a length past max_context_len
  // is read up to the grid's last partition)
  const int np_b = min((L + PS - 1) / PS, np_grid);
  const bool final_out = (P.mode == 0) && np_b <= 1;
  const int h0 = g * G;

  if (L <= 0) {
    if (final_out && j == 0) {
      for (int i = threadIdx.x; i < G * D; i += blockDim.x)
        P.out[((size_t)b * P.num_q_heads + h0) * D + i] = __float2half_rn(0.f);
    }
    return;
  }
  if (j >= np_b) return;

  const int t0 = j * PS;
  const int t1 = min(t0 + PS, L);
  const int blk0 = t0 / BS;
  const int nblk = (t1 - t0 + BS - 1) / BS;
  const int32_t* bt = P.block_tables + (size_t)b * P.max_blocks_per_seq + blk0;
  const size_t head_stride = (size_t)T::TILE_ELEMS;  // elements per (block, head) tile
  const size_t block_stride = (size_t)P.num_kv_heads * head_stride;
  const __half* kbase = P.k_cache + (size_t)g * head_stride;
  const __half* vbase = P.v_cache + (size_t)g * head_stride;
  const int pd = P.prefetch_distance;
  const L2Hints l2h = make_l2_hints(P.l2_hints != 0);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  WarpDecoder<D, BS, G, VARIANT> wd;
  wd.init(P.q + ((size_t)b * P.num_q_heads + h0) * D, lane);
  float* prow = p_rows + warp * (16 * 16);
  const int col_off = wd.ds * 8;              // element offset of slice ds in a row
  const int row_off = wd.rh * D + col_off;    // ... and of (row rh, slice ds)

  if constexpr (T::kTma) {
    // -------------------------------------------------------- staged path
    uint64_t* full = bars + warp * T::SW;
    unsigned char* ring = smem + (size_t)warp * T::SW * T::SLOT_BYTES;
    if (lane == 0) {
      for (int s = 0; s < T::SW; ++s) mbar_init(&full[s], 1);
      fence_mbarrier_init();
    }
    __syncwarp();
    // Block ids are read one step ahead into registers (every lane holds the
    // same values), so no global load sits on the critical path of the
    // lane-0 branch that issues copies:
    //   ic_pb  the block of the next row group to copy (issue cursor ic)
    //   pf_pb  the block `pd` of this warp's iterations beyond it, for L2
    SubCursor<BS, NW> ic, cc;
    ic.start(warp);
    cc.start(warp);
    auto block_id = [&](int k) { return k < nblk ? bt[k] : -1; };
    int ic_pb = block_id(ic.k);
    int pf_k = warp + NW * pd;
    int pf_pb = pd > 0 ? block_id(pf_k) : -1;
    uint32_t bad_slots = 0;  // bit s: the row group in slot s has an invalid block id
    // issue the row group at ic into `slot`; then advance ic (all lanes)
    auto issue_next = [&](int slot) {
      const bool bad = ic_pb < 0 || ic_pb >= P.num_blocks;
      bad_slots = bad ? (bad_slots | (1u << slot)) : (bad_slots & ~(1u << slot));
      if (lane == 0) {
        if (bad) {
          record_error(P.error_word, kErrBadBlock);
          mbar_arrive(&full[slot]);
        } else {
          unsigned char* dst = ring + (size_t)slot * T::SLOT_BYTES;
          const size_t off = (size_t)ic_pb * block_stride + (size_t)ic.rg * T::SUB_ELEMS;
          mbar_arrive_expect_tx(&full[slot], 2 * T::SUB_BYTES);
          bulk_copy_g2s(dst, kbase + off, T::SUB_BYTES, &full[slot], l2h);
          bulk_copy_g2s(dst + T::SUB_BYTES, vbase + off, T::SUB_BYTES, &full[slot], l2h);
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
    for (int s = 0; s < T::SW && ic.live(nblk); ++s) issue_next(s);
    bool abort = false;
    for (int u = 0; cc.live(nblk) && !abort; ++u) {
      const int slot = u % T::SW;
      const bool bad = (bad_slots >> slot) & 1u;
      const bool ok = mbar_wait_bounded(&full[slot], (u / T::SW) & 1, P.timeout_ns);
      if (!ok) {
        if (lane == 0) record_error(P.error_word, kErrTimeout);
        abort = true;
        break;
      }
      if (!bad) {
        const int valid = min(16, t1 - (t0 + cc.k * BS + cc.rg * 16));
        const __half* kg = reinterpret_cast<const __half*>(ring + (size_t)slot * T::SLOT_BYTES) + col_off;
        const __half* vg = kg + T::SUB_ELEMS + wd.rh * D;
        float s2[G];
        wd.scores([&](int i) { return lds128(kg + wd.k_row(i) * D); }, P.scale_log2, s2);
        if (wd.my_score_row() >= valid) {
#pragma unroll
          for (int h = 0; h < G; ++h) s2[h] = -INFINITY;
        }
        wd.softmax_update(s2, prow);
        wd.accumulate([&](int i) { return lds128(vg + i * RPW * D); }, prow, valid);
      }
      __syncwarp();
      if (ic.live(nblk)) {
        if (lane == 0) fence_proxy_async_smem();  // our reads of the slot precede the next copy into it
        issue_next(slot);
      }
      cc.advance(t0, t1);
    }
  } else {
    // -------------------------------------------------- register-direct path
    // block ids one iteration ahead in registers: pb for this block, and pp
    // for the block `pd` iterations later that the L2 prefetch targets
    const bool use_pf = VARIANT == kL2Prefetch && pd > 0;
    int pb_next = (warp < nblk) ? bt[warp] : 0;
    int pp_next = (use_pf && warp + NW * pd < nblk) ? bt[warp + NW * pd] : -1;
    for (int k = warp; k < nblk; k += NW) {
      const int pb = pb_next;
      if (k + NW < nblk) pb_next = bt[k + NW];
      const int pp = pp_next;
      if (use_pf) pp_next = (k + NW * (pd + 1) < nblk) ? bt[k + NW * (pd + 1)] : -1;
      if (use_pf && lane == 0 && pp >= 0 && pp < P.num_blocks) {
        // Algorithm 1: prefetch the block this warp takes `pd` iterations later
        prefetch_l2_bulk(kbase + (size_t)pp * block_stride, T::TILE_BYTES, l2h);
        prefetch_l2_bulk(vbase + (size_t)pp * block_stride, T::TILE_BYTES, l2h);
      }
      if (pb < 0 || pb >= P.num_blocks) {
        if (lane == 0) record_error(P.error_word, kErrBadBlock);
        continue;
      }
      const int valid_blk = min(BS, t1 - (t0 + k * BS));
      const __half* kt = kbase + (size_t)pb * block_stride + col_off;
      const __half* vt = vbase + (size_t)pb * block_stride + row_off;
#pragma unroll
      for (int rg = 0; rg < T::RG; ++rg) {
        const int valid = valid_blk - rg * 16;
        if (valid <= 0) break;
        uint4 kr[TPL];
#pragma unroll
        for (int i = 0; i < TPL; ++i) kr[i] = ldg_stream(kt + (rg * 16 + wd.k_row(i)) * D, l2h);
        uint4 vr[TPL];
        constexpr bool early_v = G <= 4;
        if (early_v) {
#pragma unroll
          for (int i = 0; i < TPL; ++i) vr[i] = ldg_stream(vt + (rg * 16 + i * RPW) * D, l2h);
        }
        float s2[G];
        wd.scores([&](int i) { return kr[i]; }, P.scale_log2, s2);
        if (wd.my_score_row() >= valid) {
#pragma unroll
          for (int h = 0; h < G; ++h) s2[h] = -INFINITY;
        }
        wd.softmax_update(s2, prow);
        if (!early_v) {
#pragma unroll
          for (int i = 0; i < TPL; ++i) vr[i] = ldg_stream(vt + (rg * 16 + i * RPW) * D, l2h);
        }
        wd.accumulate([&](int i) { return vr[i]; }, prow, valid);
      }
    }
  }

  // ------------------------------------------------------------------ merge
  __syncthreads();  // every warp is done with the ring that the merge area reuses
  float* mrg = reinterpret_cast<float*>(smem);
  float* mrg_m = mrg;                 // [NW][G] running shift
  float* mrg_mt = mrg + NW * G;       // [NW][G] exact maximum
  float* mrg_l = mrg + 2 * NW * G;    // [NW][G]
  float* mrg_acc = mrg + T::MRG_ACC_OFF;  // [NW][G][D]
  wd.store_warp(mrg_m + warp * G, mrg_mt + warp * G, mrg_l + warp * G, mrg_acc + warp * G * D);
  __syncthreads();
  for (int i = threadIdx.x; i < G * D; i += blockDim.x) {
    const int h = i / D, d = i % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, mrg_mt[w * G + h]);  // the exact maximum
    float Z = 0.f, O = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float mw = mrg_m[w * G + h];
      const float c = (mw == -INFINITY) ? 0.f : ex2_approx(mw - M);
      Z = fmaf(c, mrg_l[w * G + h], Z);
      O = fmaf(c, mrg_acc[(w * G + h) * D + d], O);
    }
    const size_t row = (size_t)b * P.num_q_heads + h0 + h;
    if (final_out) {
      P.out[row * D + d] = __float2half_rn(O / Z);
    } else {
      const size_t pidx = row * P.max_partitions + j;
      P.tmp_out[pidx * D + d] = O;
      if (d == 0) {
        P.max_logits[pidx] = M * 0.69314718055994530942f;  // log2 units -> natural
        P.exp_sums[pidx] = Z;
      }
    }
  }
}

}  // namespace pkd
