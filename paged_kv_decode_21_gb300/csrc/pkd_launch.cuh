// pkd_launch.cuh -- host-side launch of one kernel instantiation.
#pragma once
#include <cuda_runtime.h>
#include "pkd_decode.cuh"
#include "pkd_decode_ws.cuh"

namespace pkd {

// The staged data path switches to the warp-specialised kernel from this
// group size on (QK and PV in separate warps; see pkd_decode_ws.cuh).
constexpr int kWsMinGroup = 6;

template <int D, int BS, int G, int VARIANT>
cudaError_t launch_decode_inst(const DecodeParams& p, long long grid, cudaStream_t stream) {
  if constexpr (VARIANT == kTmaStaged && G >= kWsMinGroup) {
    using T = WsTraits<D, BS, G>;
    auto* fn = paged_decode_ws_kernel<D, BS, G>;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, T::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    fn<<<(unsigned)grid, T::THREADS, T::SMEM_BYTES, stream>>>(p);
  } else {
    using T = DecodeTraits<D, BS, G, VARIANT>;
    auto* fn = paged_decode_kernel<D, BS, G, VARIANT>;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, T::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    fn<<<(unsigned)grid, T::THREADS, T::SMEM_BYTES, stream>>>(p);
  }
  return cudaGetLastError();
}

// Dispatch over the compiled (head_dim, block_size, group) set for one data path.
template <int VARIANT>
cudaError_t launch_decode_variant(int D, int BS, int G, const DecodeParams& p, long long grid,
                                  cudaStream_t stream) {
#define PKD_CASE_G(D_, BS_)                                                   \
  switch (G) {                                                                \
    case 1: return launch_decode_inst<D_, BS_, 1, VARIANT>(p, grid, stream); \
    case 2: return launch_decode_inst<D_, BS_, 2, VARIANT>(p, grid, stream); \
    case 3: return launch_decode_inst<D_, BS_, 3, VARIANT>(p, grid, stream); \
    case 4: return launch_decode_inst<D_, BS_, 4, VARIANT>(p, grid, stream); \
    case 5: return launch_decode_inst<D_, BS_, 5, VARIANT>(p, grid, stream); \
    case 6: return launch_decode_inst<D_, BS_, 6, VARIANT>(p, grid, stream); \
    case 7: return launch_decode_inst<D_, BS_, 7, VARIANT>(p, grid, stream); \
    case 8: return launch_decode_inst<D_, BS_, 8, VARIANT>(p, grid, stream); \
    default: return cudaErrorInvalidValue;                                    \
  }
  if (D == 128 && BS == 16) { PKD_CASE_G(128, 16) }
  if (D == 128 && BS == 32) { PKD_CASE_G(128, 32) }
  if (D == 64 && BS == 16) { PKD_CASE_G(64, 16) }
  if (D == 64 && BS == 32) { PKD_CASE_G(64, 32) }
#undef PKD_CASE_G
  return cudaErrorInvalidValue;
}

// Defined in the per-variant translation units.
cudaError_t launch_decode_no_prefetch(int D, int BS, int G, const DecodeParams& p, long long grid,
                                      cudaStream_t stream);
cudaError_t launch_decode_l2_prefetch(int D, int BS, int G, const DecodeParams& p, long long grid,
                                      cudaStream_t stream);
cudaError_t launch_decode_tma_staged(int D, int BS, int G, const DecodeParams& p, long long grid,
                                     cudaStream_t stream);
cudaError_t launch_decode_tma_mma(int D, int BS, int G, const DecodeParams& p, long long grid,
                                  cudaStream_t stream);
cudaError_t launch_decode_tma_mma_multi(int D, int BS, int G, const DecodeParams& p, long long grid,
                                        cudaStream_t stream);
cudaError_t launch_decode_tma_mma_fp8(int D, int BS, int G, const DecodeParams& p, long long grid,
                                      cudaStream_t stream);
// Single-query decode over E4M3 caches at four CTAs per SM, for grids of
// many waves (pkd_inst_tma_mma_fp8_w4.cu).
cudaError_t launch_decode_tma_mma_fp8_w4(int D, int BS, int G, const DecodeParams& p, long long grid,
                                         cudaStream_t stream);

}  // namespace pkd
