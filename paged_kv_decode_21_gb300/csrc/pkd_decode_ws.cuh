// pkd_decode_ws.cuh -- warp-specialised staged decode kernel for large GQA
// groups.
//
// With many query heads per kv head, one warp that holds Q (8 dims x G heads)
// and the output accumulators (8 dims x G heads) at once needs about 255
// registers, so only two warps fit per SM sub-partition and the kernel is
// latency-bound.  Here each of NS block streams of a CTA (blocks s, s+NS,
// s+2NS, ... -- the stride order of Algorithm 1 in the review "Accelerating
// LLM Inference Throughput via Asynchronous KV Cache Prefetching", section
// 3.4) is served by two warps:
//   QK warp  holds Q; waits for the K sub-tile of a slot, forms the scores
//            (packed FMAs + transpose-reduce), runs the online softmax, and
//            publishes p (as (p, p) pairs) and the rescale factors of that
//            16-row group in the slot's p buffer;
//   PV warp  holds the output accumulators; waits for the p buffer,
//            rescales if asked, accumulates p * V from the slot's V sub-tile,
//            then refills the slot with the bulk copy of a later row group
//            and issues the L2 prefetch of the tiles further ahead.
// Each role needs about half the registers, so 2 CTAs of 6 warps fit per SM
// (12 warps), with no K/V element converted twice.  All waits are bounded.
#pragma once
#include <cstdint>
#include <cuda_fp16.h>
#include "pkd_decode.cuh"

namespace pkd {

template <int D, int BS, int G>
struct WsTraits {
  static constexpr int LPR = D / 8, RPW = 32 / LPR, TPL = 16 / RPW;
  static constexpr int TILE_ELEMS = BS * D, TILE_BYTES = TILE_ELEMS * 2;
  static constexpr int NS = 3;                 // block streams per CTA
  static constexpr int THREADS = 2 * NS * 32;  // one QK and one PV warp per stream
  static constexpr int MIN_BLOCKS = 2;
  static constexpr int SUB_ELEMS = 16 * D, SUB_BYTES = SUB_ELEMS * 2, SLOT_BYTES = 2 * SUB_BYTES;
  static constexpr int SW = (D == 128) ? 4 : 8;  // slots per stream
  // p buffer of a slot: (p, p) pairs [16 rows][8 heads], alpha[8], flags[4]
  static constexpr int PB_P = 16 * 8 * 2, PB_ALPHA = 8, PB_FLAGS = 4;
  static constexpr int PBUF_FLOATS = PB_P + PB_ALPHA + PB_FLAGS;
  static constexpr int PBUF_BYTES = PBUF_FLOATS * 4;
  static constexpr int RING_BYTES = NS * SW * SLOT_BYTES;
  static constexpr int PB_BYTES = NS * SW * PBUF_BYTES;
  // merge area: running shift m, exact maximum mt and l ([NS][G] each), then
  // acc [NS][G][D] starting on a 16-byte boundary (written with 16-byte stores)
  static constexpr int MRG_ACC_OFF = (3 * NS * G + 3) / 4 * 4;  // floats
  static constexpr int MERGE_BYTES = (MRG_ACC_OFF + NS * G * D) * 4;
  static_assert((MRG_ACC_OFF * 4) % 16 == 0, "accumulator merge area must be 16-byte aligned");
  static_assert((PBUF_FLOATS * 4) % 16 == 0, "p buffers must be 16-byte aligned");
  static constexpr int BAR_BYTES = NS * SW * 2 * 8;
  static constexpr int MAIN_BYTES = RING_BYTES > MERGE_BYTES ? RING_BYTES : MERGE_BYTES;
  static constexpr int SMEM_BYTES = MAIN_BYTES + PB_BYTES + BAR_BYTES;
  static_assert(MAIN_BYTES % 16 == 0 && PB_BYTES % 16 == 0 && SLOT_BYTES % 16 == 0,
                "shared-memory regions must stay 16-byte aligned");
};

// flags[0] of a p buffer: 1 if the row group's block id was invalid (skip);
// flags[1]: 1 if alpha must be applied before accumulating.

template <int D, int BS, int G>
__global__ void __launch_bounds__(WsTraits<D, BS, G>::THREADS, WsTraits<D, BS, G>::MIN_BLOCKS)
    paged_decode_ws_kernel(const DecodeParams P) {
  using T = WsTraits<D, BS, G>;
  constexpr int NS = T::NS, RPW = T::RPW, TPL = T::TPL, LPR = T::LPR, SW = T::SW;
  extern __shared__ __align__(128) unsigned char smem[];
  float* pbufs = reinterpret_cast<float*>(smem + T::MAIN_BYTES);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + T::MAIN_BYTES + T::PB_BYTES);

  const int np_grid = P.max_partitions;
  const int j = blockIdx.x % np_grid;
  const int bg = blockIdx.x / np_grid;
  const int g = bg % P.num_kv_heads;
  const int b = bg / P.num_kv_heads;
  // the split-K merge (a programmatic dependent) may launch once every CTA has started
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int L = row_clamped_len<BS>(P, b);
  const int PS = P.partition_size;
  const int np_b = min((L + PS - 1) / PS, np_grid);  // partitions inside the grid
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
  const int nblk = (t1 - t0 + BS - 1) / BS;
  const int32_t* bt = P.block_tables + (size_t)b * P.max_blocks_per_seq + t0 / BS;
  const size_t head_stride = (size_t)T::TILE_ELEMS;
  const size_t block_stride = (size_t)P.num_kv_heads * head_stride;
  const __half* kbase = P.k_cache + (size_t)g * head_stride;
  const __half* vbase = P.v_cache + (size_t)g * head_stride;
  const int pd = P.prefetch_distance;
  const L2Hints l2h = make_l2_hints(P.l2_hints != 0);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const bool is_pv = warp >= NS;
  const int s = is_pv ? warp - NS : warp;  // stream
  const int rh = lane / LPR, ds = lane % LPR;

  uint64_t* full = bars + s * SW;              // K/V landed (complete_tx)
  uint64_t* pready = bars + NS * SW + s * SW;  // p buffer published by the QK warp
  unsigned char* ring = smem + (size_t)s * SW * T::SLOT_BYTES;
  float* pbuf0 = pbufs + (size_t)s * SW * T::PBUF_FLOATS;
  if (threadIdx.x == 0) {
    for (int i = 0; i < 2 * NS * SW; ++i) mbar_init(&bars[i], 1);
    fence_mbarrier_init();
  }
  __syncthreads();

  float mrg_m_val[G], mrg_mt_val[G];
  float* mrg = reinterpret_cast<float*>(smem);  // used after the final __syncthreads

  if (!is_pv) {
    // ---------------------------------------------------------------- QK warp
    const int perm = (ds >> 1) & (TPL - 1);
    float2 q2[G][4];
    float m[G], l[G], mt[G];  // running shift (lazy), sum, exact maximum
    {
      const __half* qrow0 = P.q + ((size_t)b * P.num_q_heads + h0) * D;
#pragma unroll
      for (int h = 0; h < G; ++h) {
        uint4 u = *reinterpret_cast<const uint4*>(qrow0 + (size_t)h * D + ds * 8);
        // fold softmax scale and log2(e) into q: scores come out in log2 units
        const float2 sc = make_float2(P.scale_log2, P.scale_log2);
        q2[h][0] = fmul2(h2f2(u.x), sc);
        q2[h][1] = fmul2(h2f2(u.y), sc);
        q2[h][2] = fmul2(h2f2(u.z), sc);
        q2[h][3] = fmul2(h2f2(u.w), sc);
        m[h] = -INFINITY;
        mt[h] = -INFINITY;
        l[h] = 0.f;
      }
    }
    SubCursor<BS, NS> cc;
    cc.start(s);
    bool abort = false;
    for (int u = 0; cc.live(nblk) && !abort; ++u) {
      const int slot = u % SW;
      const uint32_t par = (u / SW) & 1;
      float* pb = pbuf0 + slot * T::PBUF_FLOATS;
      if (!mbar_wait_bounded(&full[slot], par, P.timeout_ns)) {
        if (lane == 0) record_error(P.error_word, kErrTimeout);
        abort = true;
        break;
      }
      const bool bad = pb[T::PB_P + T::PB_ALPHA] != 0.f;
      bool need = false;
      if (!bad) {
        const int valid = min(16, t1 - (t0 + cc.k * BS + cc.rg * 16));
        const __half* kg = reinterpret_cast<const __half*>(ring + (size_t)slot * T::SLOT_BYTES) + ds * 8;
        float part[TPL][G];
#pragma unroll
        for (int i = 0; i < TPL; ++i) {
          const uint4 kv = lds128(kg + (RPW * (i ^ perm) + rh) * D);
          const float2 kk[4] = {h2f2(kv.x), h2f2(kv.y), h2f2(kv.z), h2f2(kv.w)};
          // d-pair outermost: the G chains issue back to back
          float2 a[G];
#pragma unroll
          for (int h = 0; h < G; ++h) a[h] = fmul2(q2[h][0], kk[0]);
#pragma unroll
          for (int c = 1; c < 4; ++c)
#pragma unroll
            for (int h = 0; h < G; ++h) a[h] = ffma2(q2[h][c], kk[c], a[h]);
#pragma unroll
          for (int h = 0; h < G; ++h) part[i][h] = a[h].x + a[h].y;
        }
#pragma unroll
        for (int lvl = 0; (TPL >> lvl) > 1; ++lvl) {
          const int n = TPL >> lvl;
          const int mask = (LPR / 2) >> lvl;
#pragma unroll
          for (int jj = 0; jj < n / 2; ++jj) {
#pragma unroll
            for (int h = 0; h < G; ++h) part[jj][h] += __shfl_xor_sync(0xffffffffu, part[jj + n / 2][h], mask);
          }
        }
        const int myrow = RPW * perm + rh;
        float s2[G];
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float v = part[0][h] + __shfl_xor_sync(0xffffffffu, part[0][h], 1);
          s2[h] = myrow < valid ? v : -INFINITY;
          need |= s2[h] > m[h] + kLazyTau;
        }
        need = __any_sync(0xffffffffu, need);
        if (need) {
#pragma unroll
          for (int h = 0; h < G; ++h) {
            float mx = s2[h];
#pragma unroll
            for (int msk = 2; msk < 32; msk <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, msk));
            const float mn = fmaxf(m[h], mx);
            const float alpha = (mn == -INFINITY) ? 1.f : ex2_approx(m[h] - mn);
            l[h] *= alpha;
            m[h] = mn;
            if (lane == 0) pb[T::PB_P + h] = alpha;
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
          float4* dst = reinterpret_cast<float4*>(pb + myrow * 16);
#pragma unroll
          for (int h2 = 0; h2 < (G + 1) / 2; ++h2)
            dst[h2] = make_float4(p[2 * h2], p[2 * h2], p[2 * h2 + 1], p[2 * h2 + 1]);
        }
      }
      if (lane == 0) pb[T::PB_P + T::PB_ALPHA + 1] = need ? 1.f : 0.f;
      __syncwarp();
      if (lane == 0) mbar_arrive(&pready[slot]);
      cc.advance(t0, t1);
    }
    // this stream's (m, l)
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float lv = (ds & 1) ? 0.f : l[h];
      float mx = mt[h];
#pragma unroll
      for (int msk = 1; msk < 32; msk <<= 1) {
        lv += __shfl_xor_sync(0xffffffffu, lv, msk);
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, msk));
      }
      l[h] = lv;
      mrg_m_val[h] = m[h];
      mrg_mt_val[h] = mx;
    }
    __syncthreads();  // (1) every warp is past the ring before the merge area is written
    if (lane == 0) {
#pragma unroll
      for (int h = 0; h < G; ++h) {
        mrg[s * G + h] = mrg_m_val[h];
        mrg[NS * G + s * G + h] = mrg_mt_val[h];
        mrg[2 * NS * G + s * G + h] = l[h];
      }
    }
  } else {
    // ---------------------------------------------------------------- PV warp
    float2 acc[G][4];
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[h][c] = make_float2(0.f, 0.f);
    SubCursor<BS, NS> ic, cc;
    ic.start(s);
    cc.start(s);
    auto block_id = [&](int k) { return k < nblk ? bt[k] : -1; };
    int ic_pb = block_id(ic.k);
    int pf_k = s + NS * pd;
    int pf_pb = pd > 0 ? block_id(pf_k) : -1;
    // lane 0 copies the row group at ic into `slot` (flags first, then the
    // copies); every lane advances ic
    auto issue_next = [&](int slot) {
      const bool badb = ic_pb < 0 || ic_pb >= P.num_blocks;
      if (lane == 0) {
        float* pb = pbuf0 + slot * T::PBUF_FLOATS;
        pb[T::PB_P + T::PB_ALPHA] = badb ? 1.f : 0.f;
        if (badb) {
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
        pf_k += NS;
        pf_pb = block_id(pf_k);
      }
      const int k_before = ic.k;
      ic.advance(t0, t1);
      if (ic.k != k_before) ic_pb = block_id(ic.k);
    };
    for (int i = 0; i < SW && ic.live(nblk); ++i) issue_next(i);
    bool abort = false;
    for (int u = 0; cc.live(nblk) && !abort; ++u) {
      const int slot = u % SW;
      const uint32_t par = (u / SW) & 1;
      const float* pb = pbuf0 + slot * T::PBUF_FLOATS;
      if (!mbar_wait_bounded(&pready[slot], par, P.timeout_ns) ||
          !mbar_wait_bounded(&full[slot], par, P.timeout_ns)) {
        if (lane == 0) record_error(P.error_word, kErrTimeout);
        abort = true;
        break;
      }
      const bool bad = pb[T::PB_P + T::PB_ALPHA] != 0.f;
      if (!bad) {
        if (pb[T::PB_P + T::PB_ALPHA + 1] != 0.f) {
#pragma unroll
          for (int h = 0; h < G; ++h) {
            const float a = pb[T::PB_P + h];
            const float2 a2 = make_float2(a, a);
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[h][c] = fmul2(acc[h][c], a2);
          }
        }
        const int valid = min(16, t1 - (t0 + cc.k * BS + cc.rg * 16));
        const __half* vg =
            reinterpret_cast<const __half*>(ring + (size_t)slot * T::SLOT_BYTES) + T::SUB_ELEMS + rh * D + ds * 8;
        // rows are software-pipelined: row i+1's V and p loads are issued
        // before row i's FMAs, which hides the shared-memory latency
        constexpr int NH2 = (G + 1) / 2;
        auto load_row = [&](int i, uint4& v, float4 (&pp)[NH2]) {
          v = lds128(vg + i * RPW * D);
          const int r = RPW * i + rh;
#pragma unroll
          for (int h2 = 0; h2 < NH2; ++h2) pp[h2] = *reinterpret_cast<const float4*>(pb + r * 16 + 4 * h2);
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
            const int r = RPW * i + rh;
            if (r < valid) {
              uint4 vc;
              float4 pc[NH2];
              load_row(i, vc, pc);
              fma_row(vc, pc);
            }
          }
        }
      }
      __syncwarp();
      if (ic.live(nblk)) {
        if (lane == 0) fence_proxy_async_smem();  // our reads of the slot precede the next copy into it
        issue_next(slot);
      }
      cc.advance(t0, t1);
    }
    // this stream's accumulators, reduced over the row halves
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
#pragma unroll
        for (int msk = LPR; msk < 32; msk <<= 1) {
          acc[h][c].x += __shfl_xor_sync(0xffffffffu, acc[h][c].x, msk);
          acc[h][c].y += __shfl_xor_sync(0xffffffffu, acc[h][c].y, msk);
        }
      }
    __syncthreads();  // (1)
    if (rh == 0) {
      float* mrg_acc = mrg + T::MRG_ACC_OFF;
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float4* dst = reinterpret_cast<float4*>(mrg_acc + (s * G + h) * D + ds * 8);
        dst[0] = make_float4(acc[h][0].x, acc[h][0].y, acc[h][1].x, acc[h][1].y);
        dst[1] = make_float4(acc[h][2].x, acc[h][2].y, acc[h][3].x, acc[h][3].y);
      }
    }
  }
  __syncthreads();
  // ------------------------------------------------------------------ merge
  const float* mrg_m = mrg;
  const float* mrg_mt = mrg + NS * G;
  const float* mrg_l = mrg + 2 * NS * G;
  const float* mrg_acc = mrg + T::MRG_ACC_OFF;
  for (int i = threadIdx.x; i < G * D; i += blockDim.x) {
    const int h = i / D, d = i % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NS; ++w) M = fmaxf(M, mrg_mt[w * G + h]);  // the exact maximum
    float Z = 0.f, O = 0.f;
#pragma unroll
    for (int w = 0; w < NS; ++w) {
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
        P.max_logits[pidx] = M * 0.69314718055994530942f;
        P.exp_sums[pidx] = Z;
      }
    }
  }
}

}  // namespace pkd
