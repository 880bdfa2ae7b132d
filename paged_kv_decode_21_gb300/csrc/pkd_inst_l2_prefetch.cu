// Instantiations of the decode kernel, 16-byte global loads plus L2 bulk prefetch.
#include "pkd_launch.cuh"
namespace pkd {
cudaError_t launch_decode_l2_prefetch(int D, int BS, int G, const DecodeParams& p, long long grid,
                                      cudaStream_t stream) {
  return launch_decode_variant<kL2Prefetch>(D, BS, G, p, grid, stream);
}
}  // namespace pkd
