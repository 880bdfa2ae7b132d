// Instantiations of the tensor-core decode kernel for single-query decode.
#include "pkd_launch.cuh"
#include "pkd_mma_launch.cuh"

namespace pkd {
cudaError_t launch_decode_tma_mma(int D, int BS, int G, const DecodeParams& p, long long grid,
                                  cudaStream_t stream) {
  if (p.q_len != 1) return launch_decode_tma_mma_multi(D, BS, G, p, grid, stream);
  return mma_host::launch_all<mma_host::SingleQuery>(D, BS, G, p, grid, stream);
}
}  // namespace pkd
