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
  float scale_log2;     // softmax scale * log2(e)
  int prefetch_distance;
  unsigned long long timeout_ns;
};

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
  // Two resident CTAs of 4 warps per SM (2 warps per SM sub-partition, so up
  // to 255 registers a thread); two CTAs let one CTA's start-up overlap the
  // other's tail.
  static constexpr int NW = 4;
  static constexpr int MIN_BLOCKS = 2;
  static constexpr int THREADS = NW * 32;
  // Staging unit of the staged variant: one 16-row group of K and of V
  // (each 16*D contiguous halves).  Every warp owns SW slots of its own,
  // about 96 KiB of slots per CTA.
  static constexpr int SUB_ELEMS = 16 * D;
  static constexpr int SUB_BYTES = SUB_ELEMS * 2;
  static constexpr int SLOT_BYTES = 2 * SUB_BYTES;
  static constexpr int SW_RAW = (96 * 1024) / (NW * SLOT_BYTES);
  static constexpr int SW = kTma ? (SW_RAW > 8 ? 8 : (SW_RAW < 2 ? 2 : SW_RAW)) : 0;
  static constexpr int RING_BYTES = NW * SW * SLOT_BYTES;
  static constexpr int P_BYTES = NW * 16 * 8 * 4;           // per-warp p rows [16][8]
  static constexpr int MERGE_BYTES = NW * G * (D + 2) * 4;  // per-warp m, l, acc
  static constexpr int BAR_BYTES = NW * SW * 8;
  // layout: [ring / merge area][p rows][barriers]; the merge reuses the ring
  static constexpr int MAIN_BYTES = RING_BYTES > MERGE_BYTES ? RING_BYTES : MERGE_BYTES;
  static constexpr int SMEM_BYTES = MAIN_BYTES + P_BYTES + BAR_BYTES;
};

// ---------------------------------------------------------------------------
__device__ __forceinline__ void record_error(int* err, uint32_t bits) {
  if (err) atomicOr(reinterpret_cast<unsigned*>(err), bits);
}

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  // 16-byte global load; the KV stream is read once, so do not allocate in L1
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ uint4 lds128(const void* p) {
  return *reinterpret_cast<const uint4*>(p);
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

  float2 q2[G][4];  // q[h][8*ds + 2c .. +2) for c < 4
  float acc[G][8];  // sum_t p_t v_t[8*ds + c] over this lane's rows
  float m[G];       // running max (log2 domain), warp-uniform
  float l[G];       // running sum of p over this lane's score slots
  int lane, rh, ds;

  __device__ __forceinline__ void init(const __half* qrow0, int lane_) {
    lane = lane_;
    rh = lane / LPR;
    ds = lane % LPR;
#pragma unroll
    for (int h = 0; h < G; ++h) {
      uint4 u = *reinterpret_cast<const uint4*>(qrow0 + (size_t)h * D + ds * 8);
      q2[h][0] = h2f2(u.x);
      q2[h][1] = h2f2(u.y);
      q2[h][2] = h2f2(u.z);
      q2[h][3] = h2f2(u.w);
      m[h] = -INFINITY;
      l[h] = 0.f;
#pragma unroll
      for (int c = 0; c < 8; ++c) acc[h][c] = 0.f;
    }
  }

  // Scores of one 16-row group.  krow(i) gives the 16 bytes of row
  // RPW*i + rh at slice ds.  Returns, in s2[h], the log2-domain score of row
  // RPW*((ds>>1)&(TPL-1)) + rh (duplicated in lanes ds, ds^1).
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
      const bool hi = (lane & mask) != 0;
#pragma unroll
      for (int j = 0; j < n / 2; ++j) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
          float send = hi ? part[j][h] : part[j + n / 2][h];
          float keep = hi ? part[j + n / 2][h] : part[j][h];
          part[j][h] = keep + __shfl_xor_sync(0xffffffffu, send, mask);
        }
      }
    }
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float v = part[0][h] + __shfl_xor_sync(0xffffffffu, part[0][h], 1);
      s2[h] = v * scale_log2;
    }
  }

  __device__ __forceinline__ int my_score_row() const { return RPW * ((ds >> 1) & (TPL - 1)) + rh; }

  // Online-softmax update with scores s2 (masked rows already -inf); writes
  // p into prow (16 x 8 floats) and leaves it visible to the warp.
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
        const float alpha = (mn == -INFINITY) ? 1.f : exp2f(m[h] - mn);  // m = -inf -> 0
        l[h] *= alpha;
#pragma unroll
        for (int c = 0; c < 8; ++c) acc[h][c] *= alpha;
        m[h] = mn;
      }
    }
    float p[8];
#pragma unroll
    for (int h = 0; h < 8; ++h) p[h] = 0.f;
#pragma unroll
    for (int h = 0; h < G; ++h) {
      p[h] = exp2f(s2[h] - m[h]);
      l[h] += p[h];
    }
    if ((ds & 1) == 0) {
      float4* dst = reinterpret_cast<float4*>(prow + my_score_row() * 8);
      dst[0] = make_float4(p[0], p[1], p[2], p[3]);
      dst[1] = make_float4(p[4], p[5], p[6], p[7]);
    }
    __syncwarp();
  }

  // acc += p * V for the rows of one 16-row group; vrow(i) as krow.
  // Rows at or past `valid` (0..16) are skipped (their V may be garbage).
  template <typename VRow>
  __device__ __forceinline__ void accumulate(VRow vrow, const float* prow, int valid) {
#pragma unroll
    for (int i = 0; i < TPL; ++i) {
      const int r = RPW * i + rh;
      if (valid >= 16 || r < valid) {
        uint4 u = vrow(i);
        float2 v0 = h2f2(u.x), v1 = h2f2(u.y), v2 = h2f2(u.z), v3 = h2f2(u.w);
        const float4 pa = *reinterpret_cast<const float4*>(prow + r * 8);
        const float4 pb = *reinterpret_cast<const float4*>(prow + r * 8 + 4);
        const float pv[8] = {pa.x, pa.y, pa.z, pa.w, pb.x, pb.y, pb.z, pb.w};
        const float vv[8] = {v0.x, v0.y, v1.x, v1.y, v2.x, v2.y, v3.x, v3.y};
#pragma unroll
        for (int h = 0; h < G; ++h) {
#pragma unroll
          for (int c = 0; c < 8; ++c) acc[h][c] = fmaf(pv[h], vv[c], acc[h][c]);
        }
      }
    }
    __syncwarp();
  }

  // Reduce this warp's state and store (m, l, acc) to the merge area.
  __device__ __forceinline__ void store_warp(float* mrg_m, float* mrg_l, float* mrg_acc) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float lv = (ds & 1) ? 0.f : l[h];
#pragma unroll
      for (int msk = 1; msk < 32; msk <<= 1) lv += __shfl_xor_sync(0xffffffffu, lv, msk);
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        float a = acc[h][c];
#pragma unroll
        for (int msk = LPR; msk < 32; msk <<= 1) a += __shfl_xor_sync(0xffffffffu, a, msk);
        acc[h][c] = a;
      }
      if (lane == 0) {
        mrg_m[h] = m[h];
        mrg_l[h] = lv;
      }
      if (rh == 0) {
        float4* dst = reinterpret_cast<float4*>(mrg_acc + h * D + ds * 8);
        dst[0] = make_float4(acc[h][0], acc[h][1], acc[h][2], acc[h][3]);
        dst[1] = make_float4(acc[h][4], acc[h][5], acc[h][6], acc[h][7]);
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
  const int L = P.context_lens[b];
  const int PS = P.partition_size;
  const int np_b = (L + PS - 1) / PS;
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

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  WarpDecoder<D, BS, G, VARIANT> wd;
  wd.init(P.q + ((size_t)b * P.num_q_heads + h0) * D, lane);
  float* prow = p_rows + warp * (16 * 8);
  const int row_off = wd.rh * D + wd.ds * 8;  // element offset of (row rh, slice ds)

  if constexpr (T::kTma) {
    // -------------------------------------------------------- staged path
    uint64_t* full = bars + warp * T::SW;
    unsigned char* ring = smem + (size_t)warp * T::SW * T::SLOT_BYTES;
    if (lane == 0) {
      for (int s = 0; s < T::SW; ++s) mbar_init(&full[s], 1);
      fence_mbarrier_init();
    }
    __syncwarp();
    // lane 0 issues the bulk copies of one row group into `slot`
    auto issue = [&](const SubCursor<BS, NW>& c, int slot) {
      const int pb = bt[c.k];
      if (pb < 0 || pb >= P.num_blocks) {
        record_error(P.error_word, kErrBadBlock);
        mbar_arrive(&full[slot]);
      } else {
        unsigned char* dst = ring + (size_t)slot * T::SLOT_BYTES;
        const size_t off = (size_t)pb * block_stride + (size_t)c.rg * T::SUB_ELEMS;
        mbar_arrive_expect_tx(&full[slot], 2 * T::SUB_BYTES);
        bulk_copy_g2s(dst, kbase + off, T::SUB_BYTES, &full[slot]);
        bulk_copy_g2s(dst + T::SUB_BYTES, vbase + off, T::SUB_BYTES, &full[slot]);
      }
      if (c.rg == 0 && pd > 0) {
        const int kp = c.k + NW * pd;
        if (kp < nblk) {
          const int pp = bt[kp];
          if (pp >= 0 && pp < P.num_blocks) {
            prefetch_l2_bulk(kbase + (size_t)pp * block_stride, T::TILE_BYTES);
            prefetch_l2_bulk(vbase + (size_t)pp * block_stride, T::TILE_BYTES);
          }
        }
      }
    };
    SubCursor<BS, NW> ic, cc;
    ic.start(warp);
    cc.start(warp);
    for (int s = 0; s < T::SW && ic.live(nblk); ++s) {
      if (lane == 0) issue(ic, s);
      ic.advance(t0, t1);  // every lane keeps the same cursor
    }
    bool abort = false;
    for (int u = 0; cc.live(nblk) && !abort; ++u) {
      const int slot = u % T::SW;
      const int pb = bt[cc.k];
      const bool bad = pb < 0 || pb >= P.num_blocks;
      const bool ok = mbar_wait_bounded(&full[slot], (u / T::SW) & 1, P.timeout_ns);
      if (!ok) {
        if (lane == 0) record_error(P.error_word, kErrTimeout);
        abort = true;
        break;
      }
      if (!bad) {
        const int valid = min(16, t1 - (t0 + cc.k * BS + cc.rg * 16));
        const __half* kg = reinterpret_cast<const __half*>(ring + (size_t)slot * T::SLOT_BYTES) + row_off;
        const __half* vg = kg + T::SUB_ELEMS;
        float s2[G];
        wd.scores([&](int i) { return lds128(kg + i * RPW * D); }, P.scale_log2, s2);
        if (wd.my_score_row() >= valid) {
#pragma unroll
          for (int h = 0; h < G; ++h) s2[h] = -INFINITY;
        }
        wd.softmax_update(s2, prow);
        wd.accumulate([&](int i) { return lds128(vg + i * RPW * D); }, prow, valid);
      }
      __syncwarp();
      if (ic.live(nblk)) {
        if (lane == 0) {
          fence_proxy_async_smem();  // our generic reads of the slot precede the next copy into it
          issue(ic, slot);
        }
        ic.advance(t0, t1);
      }
      cc.advance(t0, t1);
    }
  } else {
    // -------------------------------------------------- register-direct path
    int pb_next = (warp < nblk) ? bt[warp] : 0;
    for (int k = warp; k < nblk; k += NW) {
      const int pb = pb_next;
      if (k + NW < nblk) pb_next = bt[k + NW];
      if (pb < 0 || pb >= P.num_blocks) {
        if (lane == 0) record_error(P.error_word, kErrBadBlock);
        continue;
      }
      if (VARIANT == kL2Prefetch && lane == 0 && pd > 0) {
        // Algorithm 1: prefetch the block this warp takes `pd` iterations later
        const int kp = k + NW * pd;
        if (kp < nblk) {
          const int pp = bt[kp];
          if (pp >= 0 && pp < P.num_blocks) {
            prefetch_l2_bulk(kbase + (size_t)pp * block_stride, T::TILE_BYTES);
            prefetch_l2_bulk(vbase + (size_t)pp * block_stride, T::TILE_BYTES);
          }
        }
      }
      const int valid_blk = min(BS, t1 - (t0 + k * BS));
      const __half* kt = kbase + (size_t)pb * block_stride + row_off;
      const __half* vt = vbase + (size_t)pb * block_stride + row_off;
#pragma unroll
      for (int rg = 0; rg < T::RG; ++rg) {
        const int valid = valid_blk - rg * 16;
        if (valid <= 0) break;
        uint4 kr[TPL];
#pragma unroll
        for (int i = 0; i < TPL; ++i) kr[i] = ldg_stream(kt + (rg * 16 + i * RPW) * D);
        uint4 vr[TPL];
        constexpr bool early_v = G <= 4;
        if (early_v) {
#pragma unroll
          for (int i = 0; i < TPL; ++i) vr[i] = ldg_stream(vt + (rg * 16 + i * RPW) * D);
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
          for (int i = 0; i < TPL; ++i) vr[i] = ldg_stream(vt + (rg * 16 + i * RPW) * D);
        }
        wd.accumulate([&](int i) { return vr[i]; }, prow, valid);
      }
    }
  }

  // ------------------------------------------------------------------ merge
  __syncthreads();  // every warp is done with the ring that the merge area reuses
  float* mrg = reinterpret_cast<float*>(smem);
  float* mrg_m = mrg;                 // [NW][G]
  float* mrg_l = mrg + NW * G;        // [NW][G]
  float* mrg_acc = mrg + 2 * NW * G;  // [NW][G][D]
  wd.store_warp(mrg_m + warp * G, mrg_l + warp * G, mrg_acc + warp * G * D);
  __syncthreads();
  for (int i = threadIdx.x; i < G * D; i += blockDim.x) {
    const int h = i / D, d = i % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, mrg_m[w * G + h]);
    float Z = 0.f, O = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float mw = mrg_m[w * G + h];
      const float c = (mw == -INFINITY) ? 0.f : exp2f(mw - M);
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
