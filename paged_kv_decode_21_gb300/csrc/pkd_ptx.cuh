// pkd_ptx.cuh -- inline-PTX device primitives for sm_103a.
//
// * cp.async.bulk.prefetch.L2: the asynchronous HBM->L2 prefetch that the
//   review "Accelerating LLM Inference Throughput via Asynchronous KV Cache
//   Prefetching" builds its method on (section 3.5, the PTX prefetch
//   interface; section 3.4, Algorithm 1).
// * cp.async.bulk.tensor (TMA) tiled loads into shared memory completed on an
//   mbarrier: the shared-memory staging the blog post "KV Cache Prefetching：
//   三层预取如何隐藏 KV 访问延迟" pairs with the L2 prefetch (section 2.3).
// * mbarrier waits are bounded: after the budget (nanoseconds of
//   %globaltimer) the wait returns false and the caller records an error.
// * fma.rn.f32x2: packed fp32 FMA (two lanes of fp32 per instruction).
#pragma once
#include <cstdint>
#include <cuda_fp16.h>

namespace pkd {

// ---------------------------------------------------------------- misc
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- packed fp32
// d = a * b + c, lane-wise on (x, y), round to nearest (fma.rn.f32x2).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
// d = a * b, lane-wise (mul.rn.f32x2).
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) { return __fmul2_rn(a, b); }

// ---------------------------------------------------------------- L2 prefetch
// Asynchronous bulk prefetch of [p, p + bytes) into L2; bytes multiple of 16,
// p 16-byte aligned.  Non-blocking, no completion mechanism.
__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbarrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.release.cta.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(smem_u32(bar)),
      "r"(bytes)
      : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Wait for phase `parity` of `bar` to complete, giving up after about
// `budget_ns` nanoseconds.  Returns true on completion, false on time-out.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint64_t budget_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 0;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 63u && globaltimer_ns() - t0 > budget_ns) return false;
  }
}

// ---------------------------------------------------------------- TMA
// 4-D tiled load of the box at coordinates (c0..c3) of `tmap` into shared
// memory at `dst`, completing `bytes` on `bar`.  c0 (innermost) must be a
// multiple of 16 bytes / element size.
__device__ __forceinline__ void tma_load_4d(void* dst, const void* tmap, uint64_t* bar, int c0, int c1,
                                            int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_u32(dst)),
      "l"(tmap), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar))
      : "memory");
}

// 1-D bulk copy of `bytes` (multiple of 16) from global `src` to shared
// `dst` (both 16-byte aligned), completing `bytes` of transaction count on
// `bar`.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// ---------------------------------------------------------------- L2 policies
// Optional L2 eviction priorities for the KV stream: tiles are read exactly
// once, so the consuming load/copy marks them evict_first, while a tile that
// was prefetched ahead of use is marked evict_last until it is consumed.
struct L2Hints {
  bool on;
  uint64_t evict_first;
  uint64_t evict_last;
};

__device__ __forceinline__ L2Hints make_l2_hints(bool on) {
  L2Hints h{on, 0, 0};
  if (on) {
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(h.evict_first));
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(h.evict_last));
  }
  return h;
}

__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t bytes, const L2Hints& h) {
  if (h.on) {
    asm volatile("cp.async.bulk.prefetch.L2.global.L2::cache_hint [%0], %1, %2;" ::"l"(p), "r"(bytes),
                 "l"(h.evict_last)
                 : "memory");
  } else {
    prefetch_l2_bulk(p, bytes);
  }
}

__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                              const L2Hints& h) {
  if (h.on) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
        "%4;" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(h.evict_first)
        : "memory");
  } else {
    bulk_copy_g2s(dst, src, bytes, bar);
  }
}

}  // namespace pkd
