// Instantiations of the tensor-core decode kernel, and the tensor maps its
// 3-D tiled copies read the caches through.
#include <cuda.h>
#include <cuda_runtime.h>
#include "pkd_decode_mma.cuh"

namespace pkd {
namespace {

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                 CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                 CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled from the driver, looked up once through the runtime
// (no link-time dependency on libcuda).
EncodeTiled encode_fn() {
  static const EncodeTiled fn = []() -> EncodeTiled {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeTiled>(p);
  }();
  return fn;
}

// A cache [num_blocks][num_kv_heads][block_size][D] fp16 viewed as the 3-D
// tensor (D, num_kv_heads * block_size, num_blocks); boxes of 64 x 16 x 1
// with the 128-byte swizzle.
cudaError_t make_map(CUtensorMap* m, const void* base, int D, int rows_per_block, int num_blocks) {
  EncodeTiled enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)rows_per_block, (cuuint64_t)num_blocks};
  const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)D * 2 * rows_per_block};
  const cuuint32_t box[3] = {64, 16, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(base), dims, strides, box,
                         estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int D, int BS, int G>
cudaError_t launch_mma_inst(const CUtensorMap& mk, const CUtensorMap& mv, const DecodeParams& p,
                            long long grid, cudaStream_t stream) {
  using T = MmaTraits<D, BS, G>;
  auto* fn = paged_decode_mma_kernel<D, BS, G>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, T::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  fn<<<(unsigned)grid, T::THREADS, T::SMEM_BYTES, stream>>>(mk, mv, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_tma_mma(int D, int BS, int G, const DecodeParams& p, long long grid,
                                  cudaStream_t stream) {
  CUtensorMap mk, mv;
  cudaError_t e = make_map(&mk, p.k_cache, D, p.num_kv_heads * BS, p.num_blocks);
  if (e != cudaSuccess) return e;
  e = make_map(&mv, p.v_cache, D, p.num_kv_heads * BS, p.num_blocks);
  if (e != cudaSuccess) return e;
#define PKD_CASE_G(D_, BS_)                                                  \
  switch (G) {                                                               \
    case 1: return launch_mma_inst<D_, BS_, 1>(mk, mv, p, grid, stream);    \
    case 2: return launch_mma_inst<D_, BS_, 2>(mk, mv, p, grid, stream);    \
    case 3: return launch_mma_inst<D_, BS_, 3>(mk, mv, p, grid, stream);    \
    case 4: return launch_mma_inst<D_, BS_, 4>(mk, mv, p, grid, stream);    \
    case 5: return launch_mma_inst<D_, BS_, 5>(mk, mv, p, grid, stream);    \
    case 6: return launch_mma_inst<D_, BS_, 6>(mk, mv, p, grid, stream);    \
    case 7: return launch_mma_inst<D_, BS_, 7>(mk, mv, p, grid, stream);    \
    case 8: return launch_mma_inst<D_, BS_, 8>(mk, mv, p, grid, stream);    \
    default: return cudaErrorInvalidValue;                                   \
  }
  if (D == 128 && BS == 16) { PKD_CASE_G(128, 16) }
  if (D == 128 && BS == 32) { PKD_CASE_G(128, 32) }
  if (D == 64 && BS == 16) { PKD_CASE_G(64, 16) }
  if (D == 64 && BS == 32) { PKD_CASE_G(64, 32) }
#undef PKD_CASE_G
  return cudaErrorInvalidValue;
}

}  // namespace pkd
