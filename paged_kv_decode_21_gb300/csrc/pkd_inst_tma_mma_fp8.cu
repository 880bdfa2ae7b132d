// Instantiations of the tensor-core decode kernel over E4M3 caches (single
// query and multi-token queries).
#include "pkd_launch.cuh"
#include "pkd_mma_launch.cuh"

namespace pkd {
cudaError_t launch_decode_tma_mma_fp8(int D, int BS, int G, const DecodeParams& p, long long grid,
                                      cudaStream_t stream) {
  if (p.q_len == 1) return mma_host::launch_all<mma_host::SingleQuery, 1>(D, BS, G, p, grid, stream);
  return mma_host::launch_all<mma_host::MultiQuery, 1>(D, BS, G, p, grid, stream);
}
}  // namespace pkd
