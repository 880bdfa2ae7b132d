// pkd_mma_launch.cuh -- host side of the tensor-core decode kernel: the
// tensor maps its 3-D tiled copies read the caches through, and the launch of
// one instantiation.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include "pkd_decode_mma.cuh"

namespace pkd {
namespace mma_host {

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                 CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                 CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled from the driver, looked up once through the runtime
// (no link-time dependency on libcuda).
inline EncodeTiled encode_fn() {
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

// A cache [num_blocks][num_kv_heads][block_size][D] viewed as the 3-D tensor
// (D, num_kv_heads * block_size, num_blocks).  fp16: boxes of 64 x 16 x 1
// with the 128-byte swizzle; E4M3 bytes (kvb = 1): boxes of a whole row
// (D bytes) x 16 x 1, with the 128-byte swizzle at D = 128 and the 64-byte
// swizzle at D = 64.
inline cudaError_t make_map(CUtensorMap* m, const void* base, int D, int rows_per_block, int num_blocks,
                            int kvb) {
  EncodeTiled enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)rows_per_block, (cuuint64_t)num_blocks};
  const cuuint64_t strides[2] = {(cuuint64_t)D * kvb, (cuuint64_t)D * kvb * rows_per_block};
  const cuuint32_t box[3] = {kvb == 2 ? 64u : (cuuint32_t)D, 16, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapSwizzle swz =
      (kvb == 1 && D == 64) ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
  const CUresult r = enc(m, kvb == 2 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 3,
                         const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

inline cudaError_t make_maps(const DecodeParams& p, int D, int BS, int kvb, CUtensorMap* mk, CUtensorMap* mv) {
  cudaError_t e = make_map(mk, p.k_cache, D, p.num_kv_heads * BS, p.num_blocks, kvb);
  if (e != cudaSuccess) return e;
  return make_map(mv, p.v_cache, D, p.num_kv_heads * BS, p.num_blocks, kvb);
}

template <int D, int BS, int G, int QC, int KVB, int CPS>
cudaError_t launch_qc(const CUtensorMap& mk, const CUtensorMap& mv, const DecodeParams& p, long long grid,
                      cudaStream_t stream) {
  using T = MmaTraits<D, BS, G, QC, KVB, CPS>;
  auto* fn = paged_decode_mma_kernel<D, BS, G, QC, KVB, CPS>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, T::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  if (!p.piece_order) {
    fn<<<(unsigned)grid, T::THREADS, T::SMEM_BYTES, stream>>>(mk, mv, p);
    return cudaGetLastError();
  }
  // a programmatic dependent of the order kernel: the CTAs become resident
  // while it runs and wait for its order with griddepcontrol.wait
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(T::THREADS);
  cfg.dynamicSmemBytes = T::SMEM_BYTES;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, fn, mk, mv, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// Dispatch over the compiled (head_dim, block_size, group) set; QCOF maps a
// group size to the query tokens per CTA of the instantiation, CPS selects
// the resident CTAs per SM (0: the cache type's default).
template <template <int> class QCOF, int KVB = 2, int CPS = 0>
cudaError_t launch_all(int D, int BS, int G, const DecodeParams& p, long long grid, cudaStream_t stream) {
  CUtensorMap mk, mv;
  cudaError_t e = make_maps(p, D, BS, KVB, &mk, &mv);
  if (e != cudaSuccess) return e;
#define PKD_CASE_G(D_, BS_)                                                                  \
  switch (G) {                                                                               \
    case 1: return launch_qc<D_, BS_, 1, QCOF<1>::value, KVB, CPS>(mk, mv, p, grid, stream); \
    case 2: return launch_qc<D_, BS_, 2, QCOF<2>::value, KVB, CPS>(mk, mv, p, grid, stream); \
    case 3: return launch_qc<D_, BS_, 3, QCOF<3>::value, KVB, CPS>(mk, mv, p, grid, stream); \
    case 4: return launch_qc<D_, BS_, 4, QCOF<4>::value, KVB, CPS>(mk, mv, p, grid, stream); \
    case 5: return launch_qc<D_, BS_, 5, QCOF<5>::value, KVB, CPS>(mk, mv, p, grid, stream); \
    case 6: return launch_qc<D_, BS_, 6, QCOF<6>::value, KVB, CPS>(mk, mv, p, grid, stream); \
    case 7: return launch_qc<D_, BS_, 7, QCOF<7>::value, KVB, CPS>(mk, mv, p, grid, stream); \
    case 8: return launch_qc<D_, BS_, 8, QCOF<8>::value, KVB, CPS>(mk, mv, p, grid, stream); \
    default: return cudaErrorInvalidValue;                                                   \
  }
  if (D == 128 && BS == 16) { PKD_CASE_G(128, 16) }
  if (D == 128 && BS == 32) { PKD_CASE_G(128, 32) }
  if (D == 64 && BS == 16) { PKD_CASE_G(64, 16) }
  if (D == 64 && BS == 32) { PKD_CASE_G(64, 32) }
#undef PKD_CASE_G
  return cudaErrorInvalidValue;
}

template <int G> struct SingleQuery { static constexpr int value = 1; };
template <int G> struct MultiQuery { static constexpr int value = mma_query_chunk(G); };

}  // namespace mma_host
}  // namespace pkd
