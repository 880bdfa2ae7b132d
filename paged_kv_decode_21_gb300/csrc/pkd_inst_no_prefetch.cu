// Instantiations of the decode kernel, 16-byte global loads, no prefetch.
#include "pkd_launch.cuh"
namespace pkd {
cudaError_t launch_decode_no_prefetch(int D, int BS, int G, const DecodeParams& p, long long grid,
                                      cudaStream_t stream) {
  return launch_decode_variant<kNoPrefetch>(D, BS, G, p, grid, stream);
}
}  // namespace pkd
