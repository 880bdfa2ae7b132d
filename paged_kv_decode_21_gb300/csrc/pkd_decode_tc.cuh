// pkd_decode_tc.cuh -- decode attention with both products on the fifth-
// generation tensor cores (tcgen05), scores and output accumulator held in
// tensor memory.
//
// Work split: one CTA per (sequence b, kv head g, partition j, query chunk),
// the split-K decomposition of the partitioned decode in the review
// "Accelerating LLM Inference Throughput via Asynchronous KV Cache
// Prefetching" (section 3.4).  The CTA's tile rows are (query token r / G,
// head r % G) for up to kTcRows rows: every query head of the group and up to
// kTcRows / G query tokens share one pass over the partition's K and V, so a
// multi-token query (speculative verification) reads the cache once per
// chunk of kTcRows / G tokens rather than once per 16 / G.
//
// Roles (four warps):
//   warp 2, lane 0   producer: 3-D tensor copies of the partition's K and V
//                    into a ring of NS stages of TN tokens (the 128-byte
//                    swizzled layout the MMA descriptors read), one mbarrier
//                    per stage with the transaction count of its copies.
//   warp 3, lane 0   MMA issuer: S = Q K^T (M = 128 rows, N = TN tokens,
//                    K = 128 dims) into one of two S buffers in tensor memory,
//                    then, once the softmax has written P, O += P V
//                    (M = 128, N = 128 dims, K = TN tokens) into O in tensor
//                    memory; completion is committed to mbarriers.  S of the
//                    next tile is issued before waiting for P of this one, so
//                    the tensor cores overlap the softmax.
//   warps 0-1        softmax, one thread per tile row (tensor-memory lane):
//                    the row of S into registers, mask, online softmax in the
//                    log2 domain with a lazy running maximum (the output is
//                    rescaled in tensor memory only when the maximum grows by
//                    more than kLazyTau), P rounded to fp16 into shared memory
//                    (the MMA's A operand), and at the end O / l to the output
//                    or the unnormalised partial for the split-K merge.
// The MMAs run M = 128 with the rows past kTcRows reading whatever follows
// Q and P in shared memory: those accumulator rows are never read.
//
// The causal rule of multi-token queries is the one of the mma.sync path:
// query jq sits at position L - q_len + jq and sees the tokens before and at
// its position.  Tokens past the CTA's range (the last tile) or in a block
// with a bad id get p = 0, and their V rows are zeroed before P.V so that
// whatever the stage held cannot turn 0 * V into NaN.
//
// Every mbarrier wait is bounded (timeout_ns); a role that gives up records
// kErrTimeout and raises a flag the others poll, the producer waits for the
// copies in flight, the issuer for the MMAs in flight, and tensor memory is
// freed by the warp that allocated it after a final barrier.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_fp16.h>
#include "pkd_decode_mma.cuh"
#include "pkd_tc.cuh"

namespace pkd {

constexpr int kTcRows = 64;  // query rows per CTA (query tokens x group heads)

// Query tokens per CTA of the tcgen05 kernel for group size G.
constexpr int tc_query_chunk(int G) { return kTcRows / G; }

template <int BS>
struct TcTraits {
  static_assert(BS == 16 || BS == 32, "block_size");
  static constexpr int D = 128;
  static constexpr int ROWS = kTcRows;
  static constexpr int TN = 64;            // tokens per tile
  static constexpr int NBT = TN / BS;      // cache blocks per tile
  static constexpr int NS = 2;             // ring stages
  static constexpr int ROWB = 128;         // bytes per swizzled row: 64 fp16
  static constexpr int QH = ROWS * ROWB;   // one 64-dim half of Q
  static constexpr int PB = ROWS * ROWB;   // one P buffer (TN = 64 tokens per row)
  static constexpr int KVH = TN * ROWB;    // one 64-dim half of a K or V tile
  static constexpr int STAGE = 4 * KVH;    // K halves, then V halves
  static constexpr int Q_OFF = 0;
  static constexpr int P_OFF = Q_OFF + 2 * QH;
  static constexpr int RING_OFF = P_OFF + 2 * PB;
  static constexpr int MAIN = RING_OFF + NS * STAGE;
  static_assert(Q_OFF + QH + 128 * ROWB <= MAIN && P_OFF + PB + 128 * ROWB <= MAIN,
                "the M = 128 operand reads stay inside shared memory");
  static_assert(TN == 64, "a P row is one 128-byte swizzled row");
  static constexpr int NBAR = 2 * NS + 7;  // full, empty, sfull[2], pfull[2], pfree[2], drain
  static constexpr int TAIL = NBAR * 8 + 8 + NS * 4;
  static constexpr int SMEM_BYTES = 1024 + MAIN + ((TAIL + 15) / 16) * 16;
  static constexpr int THREADS = 128;
  static constexpr int MIN_BLOCKS = 2;
  static constexpr uint32_t TMEM_COLS = 256;  // O: columns 0-127; S buffer s: 128 + 64 s
  static constexpr uint32_t IDESC_S = tc_idesc_f16(128, TN, false);
  static constexpr uint32_t IDESC_O = tc_idesc_f16(128, D, true);
};

template <int BS>
__global__ void __launch_bounds__(TcTraits<BS>::THREADS, TcTraits<BS>::MIN_BLOCKS)
    paged_decode_tc_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                           const DecodeParams P) {
  using T = TcTraits<BS>;
  constexpr int NS = T::NS, TN = T::TN, D = T::D;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  unsigned char* smem = smem_raw + (((raw_u32 + 1023u) & ~1023u) - raw_u32);
  const uint32_t sbase = smem_u32(smem);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + T::MAIN);  // [NS] a tile's copies landed
  uint64_t* empty = full + NS;   // [NS] a tile's MMAs completed: its stage is free
  uint64_t* sfull = empty + NS;  // [2] S of a tile is in tensor memory
  uint64_t* pfull = sfull + 2;   // [2] P of a tile is in shared memory and its S was read
  uint64_t* pfree = pfull + 2;   // [2] P.V of a tile completed
  uint64_t* drain = pfree + 2;   // every MMA issued completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile uint32_t* stage_bad = reinterpret_cast<volatile uint32_t*>(tmem_slot + 2);  // [NS]

  // work item: query chunk fastest, then partition j, then (b, g)
  const int G = P.num_q_heads / P.num_kv_heads;
  const int np_grid = P.max_partitions;
  const int qc = blockIdx.x % P.q_chunks;
  const int rest = blockIdx.x / P.q_chunks;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  int j, b, g;
  if (P.piece_order) {
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
  const int jq0 = qc * (T::ROWS / G);         // first query token of this CTA
  const int nq = min(T::ROWS / G, QL - jq0);  // its query tokens (>= 1)
  const int rows = G * nq;                    // tile rows in use
  const int PS = P.partition_size;
  const int np_b = min((L + PS - 1) / PS, np_grid);
  const bool final_out = (P.mode == 0) && np_b <= 1;
  const int Hq = P.num_q_heads;
  auto out_row = [&](int rr) { return ((size_t)b * QL + jq0 + rr / G) * Hq + g * G + rr % G; };

  if (L <= 0) {
    if (final_out && j == 0) {
      for (int i = threadIdx.x; i < rows * D; i += blockDim.x)
        P.out[out_row(i / D) * D + i % D] = __float2half_rn(0.f);
    }
    return;
  }
  if (j >= np_b) return;

  const int t0 = j * PS;
  // the chunk's last query sees tokens < L - QL + jq0 + nq; nothing past that is read
  const int t1 = min(min(t0 + PS, L), L - QL + jq0 + nq);
  const int ntiles = t1 > t0 ? (t1 - t0 + TN - 1) / TN : 0;
  const int nblk = t1 > t0 ? (t1 - t0 + BS - 1) / BS : 0;
  const int32_t* bt = P.block_tables + (size_t)b * P.max_blocks_per_seq + t0 / BS;
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int nsw = rows > 32 ? 2 : 1;  // softmax warps

  if (threadIdx.x == 0) {
    prefetch_tensormap(&tmap_k);
    prefetch_tensormap(&tmap_v);
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sfull[s], 1);
      mbar_init(&pfull[s], 32 * nsw);
      mbar_init(&pfree[s], 1);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 3) {
    tmem_alloc(tmem_slot, T::TMEM_COLS);
    tmem_relinquish();
  }
  if (warp < 2) {
    // Q rows into the two 64-dim halves, 128-byte swizzled; unused rows zero
    const int rr = threadIdx.x;
    const __half* qr = rr < rows ? P.q + out_row(rr) * D : nullptr;
#pragma unroll
    for (int c = 0; c < D / 8; ++c) {
      const uint4 v = qr ? *reinterpret_cast<const uint4*>(qr + 8 * c) : make_uint4(0u, 0u, 0u, 0u);
      *reinterpret_cast<uint4*>(smem + T::Q_OFF + (c / 8) * T::QH + rr * T::ROWB + (((c % 8) ^ (rr % 8)) << 4)) = v;
    }
    fence_proxy_async_smem();  // visible to the tensor cores
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 2) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const L2Hints l2h = make_l2_hints(P.l2_hints != 0);
      int issued = 0;
      for (int i = 0; i < ntiles; ++i) {
        const int st = i % NS;
        if (*abort_flag) break;
        if (i >= NS && !mbar_wait_bounded(&empty[st], ((i / NS) - 1) & 1, P.timeout_ns)) {
          record_error(P.error_word, kErrTimeout);
          *abort_flag = 1;
          break;
        }
        int pbs[T::NBT];
        uint32_t bad = 0, bytes = 0;
#pragma unroll
        for (int kk = 0; kk < T::NBT; ++kk) {
          const int k = i * T::NBT + kk;
          int pb = k < nblk ? bt[k] : -1;
          if (k < nblk && (pb < 0 || pb >= P.num_blocks)) {
            bad |= 1u << kk;
            record_error(P.error_word, kErrBadBlock);
            pb = -1;
          }
          pbs[kk] = pb;
          if (pb >= 0) bytes += 4 * BS * T::ROWB;  // K and V, two 64-dim halves each
        }
        stage_bad[st] = bad;
        const uint32_t stg = sbase + T::RING_OFF + st * T::STAGE;
        mbar_arrive_expect_tx(&full[st], bytes);
#pragma unroll
        for (int kk = 0; kk < T::NBT; ++kk) {
          if (pbs[kk] < 0) continue;
#pragma unroll
          for (int rg = 0; rg < BS / 16; ++rg) {
            const int y = g * BS + 16 * rg;
            const uint32_t row = (kk * BS + 16 * rg) * T::ROWB;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              tma_load_3d(stg + h * T::KVH + row, &tmap_k, &full[st], 64 * h, y, pbs[kk], l2h);
              tma_load_3d(stg + (2 + h) * T::KVH + row, &tmap_v, &full[st], 64 * h, y, pbs[kk], l2h);
            }
          }
        }
        issued = i + 1;
      }
      if (*abort_flag)  // let the copies in flight land before the CTA exits
        for (int k = issued > NS ? issued - NS : 0; k < issued; ++k)
          mbar_wait_bounded(&full[k % NS], (k / NS) & 1, P.timeout_ns);
    }
  } else if (warp == 3) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t qs = sbase + T::Q_OFF;
      bool any = false;
      auto issue_qk = [&](int i) -> bool {
        const int st = i % NS;
        if (!mbar_wait_bounded(&full[st], (i / NS) & 1, P.timeout_ns)) return false;
        tc_fence_after();
        const uint32_t ks = sbase + T::RING_OFF + st * T::STAGE;
        const uint32_t d = tmem + 128 + 64 * (i & 1);
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k / 4) * T::KVH + (k % 4) * 32;  // 16 dims = 32 bytes of a row
          tc_mma_f16(d, sw128_desc(qs + (k / 4) * T::QH + (k % 4) * 32, 16, 1024), sw128_desc(ks + off, 16, 1024),
                     T::IDESC_S, k > 0 ? 1u : 0u);
        }
        tc_commit(&sfull[i & 1]);
        any = true;
        return true;
      };
      bool ok = ntiles == 0 || issue_qk(0);
      for (int i = 0; ok && i < ntiles; ++i) {
        if (*abort_flag) {
          ok = false;
          break;
        }
        if (i + 1 < ntiles && !(ok = issue_qk(i + 1))) break;
        if (!(ok = mbar_wait_bounded(&pfull[i & 1], (i / 2) & 1, P.timeout_ns))) break;
        tc_fence_after();
        const uint32_t vs = sbase + T::RING_OFF + (i % NS) * T::STAGE + 2 * T::KVH;
        const uint32_t ps = sbase + T::P_OFF + (i & 1) * T::PB;
#pragma unroll
        for (int k = 0; k < TN / 16; ++k)  // 16 tokens: 32 bytes of a P row, 16 rows of V
          tc_mma_f16(tmem, sw128_desc(ps + k * 32, 16, 1024), sw128_desc(vs + k * 16 * T::ROWB, T::KVH, 1024),
                     T::IDESC_O, (i > 0 || k > 0) ? 1u : 0u);
        tc_commit(&pfree[i & 1]);
        tc_commit(&empty[i % NS]);
      }
      if (!ok) {
        record_error(P.error_word, kErrTimeout);
        *abort_flag = 1;
      }
      if (any) {  // every MMA completes before tensor memory is freed
        tc_commit(drain);
        mbar_wait_bounded(drain, 0, P.timeout_ns);
      }
    }
  } else if (warp < nsw) {
    // ------------------------------------------------------------ softmax
    const int rr = threadIdx.x;  // tile row = tensor-memory lane
    const bool live = rr < rows;
    // tokens at or past lim are masked for this row
    const int lim = live ? min(t1, L - QL + jq0 + rr / G + 1) : t0;
    const uint32_t tl = tmem + ((uint32_t)(warp * 32) << 16);
    float m = -INFINITY, mt = -INFINITY, l = 0.f;  // running shift, exact maximum, sum of p
    bool ok = true;
    for (int i = 0; i < ntiles; ++i) {
      const int st = i % NS, sb = i & 1;
      ok = __all_sync(0xffffffffu, !*abort_flag && mbar_wait_bounded(&sfull[sb], (i / 2) & 1, P.timeout_ns));
      if (!ok) break;
      tc_fence_after();
      float s[2][32];
      tmem_ld32(tl + 128 + 64 * sb, s[0]);
      tmem_ld32(tl + 128 + 64 * sb + 32, s[1]);
      tmem_ld_wait();
      // S implies the tile's K landed; its V and bad-block mask come with the same phase
      ok = __all_sync(0xffffffffu, mbar_wait_bounded(&full[st], (i / NS) & 1, P.timeout_ns));
      if (!ok) break;
      const uint32_t bad = stage_bad[st];
      const int tb = t0 + i * TN;
      const int nv = lim - tb;             // columns this row sees
      const int valid = min(TN, t1 - tb);  // columns holding the CTA's tokens
      if (nv >= TN && bad == 0) {
#pragma unroll
        for (int e = 0; e < TN; ++e) s[e / 32][e % 32] *= P.scale_log2;
      } else {
#pragma unroll
        for (int e = 0; e < TN; ++e)
          s[e / 32][e % 32] =
              (e < nv && !((bad >> (e / BS)) & 1u)) ? s[e / 32][e % 32] * P.scale_log2 : -INFINITY;
      }
      float mx[8];
#pragma unroll
      for (int a = 0; a < 8; ++a) {
        const float* v = &s[a / 4][(a % 4) * 8];
        mx[a] = fmaxf(fmaxf(fmaxf(v[0], v[1]), fmaxf(v[2], v[3])), fmaxf(fmaxf(v[4], v[5]), fmaxf(v[6], v[7])));
      }
      const float tmax = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                               fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
      mt = fmaxf(mt, tmax);
      if (__any_sync(0xffffffffu, tmax > m + kLazyTau)) {
        const float mn = fmaxf(m, tmax);
        const float alpha = (mn == -INFINITY) ? 1.f : ex2_approx(m - mn);
        l *= alpha;
        m = mn;
        if (i > 0) {
          // O holds the earlier tiles once the last P.V completed: rescale it in place
          ok = __all_sync(0xffffffffu, mbar_wait_bounded(&pfree[(i - 1) & 1], ((i - 1) / 2) & 1, P.timeout_ns));
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            float o[32];
            tmem_ld32(tl + 32 * c, o);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] *= alpha;
            tmem_st32(tl + 32 * c, o);
          }
          tmem_st_wait();
        }
      }
      // a row that has seen no token yet keeps m = -inf: shift by 0 so that
      // its masked scores give p = 0 rather than NaN
      const float mu = m == -INFINITY ? 0.f : m;
      // this P buffer was last read by the P.V of tile i - 2
      if (i >= 2) {
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(&pfree[sb], ((i - 2) / 2) & 1, P.timeout_ns));
        if (!ok) break;
      }
      unsigned char* prow = smem + T::P_OFF + sb * T::PB + rr * T::ROWB;
      float rs = 0.f;
#pragma unroll
      for (int c = 0; c < TN / 8; ++c) {
        const float* v = &s[c / 4][(c % 4) * 8];
        float p[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) p[e] = ex2_approx(v[e] - mu);
        rs += ((p[0] + p[1]) + (p[2] + p[3])) + ((p[4] + p[5]) + (p[6] + p[7]));
        uint4 w;
        w.x = pack_half2(p[0], p[1]);
        w.y = pack_half2(p[2], p[3]);
        w.z = pack_half2(p[4], p[5]);
        w.w = pack_half2(p[6], p[7]);
        *reinterpret_cast<uint4*>(prow + ((c ^ (rr & 7)) << 4)) = w;
      }
      l += rs;
      if (valid < TN || bad) {
        // V rows that hold no token of the CTA, or a bad block's: p = 0 there,
        // and 0 * NaN would not be 0
        unsigned char* vt = smem + T::RING_OFF + st * T::STAGE + 2 * T::KVH;
        for (int x = threadIdx.x; x < 2 * TN * 8; x += 32 * nsw) {
          const int h = x / (TN * 8), r = (x / 8) % TN, c = x % 8;
          if (r >= valid || ((bad >> (r / BS)) & 1u))
            *reinterpret_cast<uint4*>(vt + h * T::KVH + r * T::ROWB + c * 16) = make_uint4(0u, 0u, 0u, 0u);
        }
      }
      fence_proxy_async_smem();  // P (and zeroed V rows) visible to the tensor cores
      tc_fence_before();         // our reads of S ordered before the arrive
      mbar_arrive(&pfull[sb]);
    }
    if (ok && ntiles > 0)
      ok = __all_sync(0xffffffffu,
                      mbar_wait_bounded(&pfree[(ntiles - 1) & 1], ((ntiles - 1) / 2) & 1, P.timeout_ns));
    if (!ok) {
      if (lane == 0) record_error(P.error_word, kErrTimeout);
      *abort_flag = 1;
    } else {
      tc_fence_after();
      const size_t orow = live ? out_row(rr) : 0;
      const size_t pidx = orow * P.max_partitions + j;
      const float inv = l > 0.f ? 1.f / l : 0.f;  // l = 0: the query saw no token
      // partials are relative to the exact maximum mt; O and l to the shift m
      const float f = m == -INFINITY ? 0.f : ex2_approx(m - mt);
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        float o[32];
        if (ntiles > 0) {
          tmem_ld32(tl + 32 * c, o);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = 0.f;
        }
        if (!live) continue;
        if (final_out) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 w;
            w.x = pack_half2(o[8 * q] * inv, o[8 * q + 1] * inv);
            w.y = pack_half2(o[8 * q + 2] * inv, o[8 * q + 3] * inv);
            w.z = pack_half2(o[8 * q + 4] * inv, o[8 * q + 5] * inv);
            w.w = pack_half2(o[8 * q + 6] * inv, o[8 * q + 7] * inv);
            *reinterpret_cast<uint4*>(P.out + orow * D + 32 * c + 8 * q) = w;
          }
        } else {
          float* dst = P.tmp_out + pidx * D + 32 * c;
#pragma unroll
          for (int q = 0; q < 8; ++q)
            *reinterpret_cast<float4*>(dst + 4 * q) =
                make_float4(o[4 * q] * f, o[4 * q + 1] * f, o[4 * q + 2] * f, o[4 * q + 3] * f);
        }
      }
      if (live && !final_out) {
        P.max_logits[pidx] = mt * 0.69314718055994530942f;  // log2 units -> natural; -inf if empty
        P.exp_sums[pidx] = l * f;
      }
    }
  }

  // tensor memory is freed once every warp is done with it
  tc_fence_before();
  __syncthreads();
  if (warp == 3) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, T::TMEM_COLS);
  }
}

}  // namespace pkd
