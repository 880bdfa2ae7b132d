// Instantiations and launch of the tcgen05 decode kernel (pkd_decode_tc.cuh):
// fp16 caches at head_dim 64 or 128, E4M3 caches at head_dim 128, block sizes
// 16 and 32.
#include "pkd_decode_tc.cuh"
#include "pkd_mma_launch.cuh"
#include "pkd_tc_launch.h"

namespace pkd {
static_assert(kTcRows == kTcRowsPerCta, "rows per CTA of the kernel and of its host entry");

namespace {

template <int BS, int KVB, int HD>
cudaError_t launch_tc_bs(const CUtensorMap& mk, const CUtensorMap& mv, const DecodeParams& p, long long grid,
                         cudaStream_t stream) {
  using T = TcTraits<BS, KVB, HD>;
  // runs of partitions per CTA: head_dim 128 only (the plan asks for them there)
  auto* fn = (HD == 128 && p.parts_per_cta > 1) ? paged_decode_tc_kernel<BS, KVB, HD, HD == 128>
                                                 : paged_decode_tc_kernel<BS, KVB, HD, false>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, T::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(T::THREADS);
  cfg.dynamicSmemBytes = T::SMEM_BYTES;
  cfg.stream = stream;
  if (p.piece_order) {
    // a programmatic dependent of the order kernel (griddepcontrol.wait in the kernel)
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  e = cudaLaunchKernelEx(&cfg, fn, mk, mv, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_tcgen05(int D, int BS, const DecodeParams& p, long long grid, cudaStream_t stream,
                                  int kvb) {
  if ((D != 128 && !(D == 64 && kvb == 2)) || (BS != 16 && BS != 32) || (kvb != 1 && kvb != 2))
    return cudaErrorInvalidValue;
  CUtensorMap mk, mv;
  cudaError_t e = mma_host::make_maps(p, D, BS, kvb, &mk, &mv);
  if (e != cudaSuccess) return e;
  if (kvb == 1)
    return BS == 16 ? launch_tc_bs<16, 1, 128>(mk, mv, p, grid, stream) : launch_tc_bs<32, 1, 128>(mk, mv, p, grid, stream);
  if (D == 64)
    return BS == 16 ? launch_tc_bs<16, 2, 64>(mk, mv, p, grid, stream) : launch_tc_bs<32, 2, 64>(mk, mv, p, grid, stream);
  return BS == 16 ? launch_tc_bs<16, 2, 128>(mk, mv, p, grid, stream) : launch_tc_bs<32, 2, 128>(mk, mv, p, grid, stream);
}

}  // namespace pkd
