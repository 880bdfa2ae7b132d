// Instantiations of the decode kernel, bulk-copy shared-memory ring plus L2 prefetch.
#include "pkd_launch.cuh"
namespace pkd {
cudaError_t launch_decode_tma_staged(int D, int BS, int G, const DecodeParams& p, long long grid,
                                     cudaStream_t stream) {
  return launch_decode_variant<kTmaStaged>(D, BS, G, p, grid, stream);
}
}  // namespace pkd
