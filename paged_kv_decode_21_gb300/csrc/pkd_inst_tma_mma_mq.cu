// Instantiations of the tensor-core decode kernel for multi-token queries
// (16 / G query tokens per CTA).
#include "pkd_launch.cuh"
#include "pkd_mma_launch.cuh"

namespace pkd {
cudaError_t launch_decode_tma_mma_multi(int D, int BS, int G, const DecodeParams& p, long long grid,
                                        cudaStream_t stream) {
  return mma_host::launch_all<mma_host::MultiQuery>(D, BS, G, p, grid, stream);
}
}  // namespace pkd
