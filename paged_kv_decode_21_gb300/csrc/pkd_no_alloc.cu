// pkd_no_alloc.cu -- split-K decode attention whose scratch lives in a
// fixed, library-owned device array, for callers that cannot allocate.
//
// Some callers cannot call cudaMalloc or hand the library a workspace: code
// that runs inside another framework's allocator and may not allocate behind
// its back, plugins and embedded runtimes that only receive input and output
// pointers, and processes that have reserved the whole device pool up front.
// This entry point gives them the split-K path anyway.  Its scratch (the
// per-partition partials) is the array below, which every GPU that loads
// this library holds until the process exits.  The caller still passes the
// inputs and the output.
#include <cstddef>
#include <cstdint>
#include <mutex>
#include <cuda_runtime.h>

#include "../../include/paged_decode.h"

namespace {

// The scratch itself.  In host code `g_pkd_static_scratch` only names a
// host-side stand-in for the symbol, never a device address: the device
// address comes from cudaGetSymbolAddress below, once per device.
static __device__ __align__(256) unsigned char g_pkd_static_scratch[PKD_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Device address of the scratch on the current device, looked up on the
// first call per device (with that device current).  nullptr on failure.
// The address is kept until the process exits: after a cudaDeviceReset the
// reloaded module's array may sit elsewhere, so the entry point is not for
// use across a reset (the header says so).
void* scratch_for_current_device(cudaError_t* err) {
  int dev = -1;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= kMaxDevices) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_pkd_static_scratch);
    if (*err != cudaSuccess || !p) return nullptr;
    g_scratch_ptr[dev] = p;
  }
  return g_scratch_ptr[dev];
}

}  // namespace

extern "C" pkd_status paged_decode_attention_static_scratch(
    const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
    const int32_t* context_lens, void* out, int num_seqs, int num_q_heads, int num_kv_heads,
    int head_dim, int block_size, int num_blocks, int max_blocks_per_seq, int max_context_len,
    float scale, int partition_size, int variant, int prefetch_distance, int* error_word,
    cudaStream_t stream) {
  if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
      max_context_len < 0)
    return PKD_ERR_SHAPE;
  if (num_seqs == 0) return PKD_OK;
  if (!out) return PKD_ERR_NULL;
  if (partition_size < 0 || (partition_size > 0 && (partition_size % 32 != 0 || partition_size % block_size != 0)))
    return PKD_ERR_SHAPE;
  int P = partition_size;
  if (P == 0) {
    P = paged_decode_auto_partition_size(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                                         max_context_len, variant);
    if (P == -2) return PKD_ERR_SHAPE;
    if (P <= 0) P = (int)round_up((size_t)(max_context_len > 0 ? max_context_len : 1), 32);
  }
  const int np = max_context_len > 0 ? (max_context_len + P - 1) / P : 1;
  // partials [B][Hq][NP][D] fp32, then max and sum [B][Hq][NP] fp32
  const size_t rows = (size_t)num_seqs * num_q_heads * np;
  const size_t o_bytes = round_up(rows * head_dim * sizeof(float), 256);
  const size_t m_bytes = round_up(rows * sizeof(float), 256);
  if (o_bytes + 2 * m_bytes > (size_t)PKD_STATIC_SCRATCH_BYTES) return PKD_ERR_WORKSPACE;

  cudaError_t err;
  unsigned char* base = static_cast<unsigned char*>(scratch_for_current_device(&err));
  if (!base) return PKD_ERR_CUDA;
  float* tmp_out = reinterpret_cast<float*>(base);
  float* max_logits = reinterpret_cast<float*>(base + o_bytes);
  float* exp_sums = reinterpret_cast<float*>(base + o_bytes + m_bytes);
  // Nothing in the scratch needs to start at zero: the first kernel writes
  // every partial that the merge then reads, within this call.
  pkd_status st = paged_decode_partitions(q, k_cache, v_cache, block_tables, context_lens, num_seqs,
                                          num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                                          max_blocks_per_seq, max_context_len, scale, P, variant,
                                          prefetch_distance, tmp_out, max_logits, exp_sums, np,
                                          error_word, stream);
  if (st != PKD_OK) return st;
  return paged_decode_reduce(tmp_out, max_logits, exp_sums, context_lens, out, num_seqs, num_q_heads,
                             head_dim, P, np, /*min_partitions_to_merge=*/0, stream);
}
