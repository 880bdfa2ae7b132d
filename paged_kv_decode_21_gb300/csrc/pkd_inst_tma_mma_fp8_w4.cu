// Instantiations of the tensor-core decode kernel for single-query decode
// over E4M3 caches at four resident CTAs per SM.
#include "pkd_launch.cuh"
#include "pkd_mma_launch.cuh"

namespace pkd {
cudaError_t launch_decode_tma_mma_fp8_w4(int D, int BS, int G, const DecodeParams& p, long long grid,
                                         cudaStream_t stream) {
  if (p.q_len != 1) return cudaErrorInvalidValue;
  return mma_host::launch_all<mma_host::SingleQuery, 1, 4>(D, BS, G, p, grid, stream);
}
}  // namespace pkd
