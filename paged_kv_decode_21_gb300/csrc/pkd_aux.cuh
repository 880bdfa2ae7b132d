// pkd_aux.cuh -- the split-K merge kernel, the paged KV append kernel and the
// block-table validator.
#pragma once
#include <cstdint>
#include <cuda_fp16.h>
#include "pkd_decode.cuh"

namespace pkd {

// ---------------------------------------------------------------------------
// Split-K merge: one warp per (b, h) row, four CTA rows; lane l owns dims
// [V l, V l + V), V = D / 32.  Lane l computes the weights of partitions
// j = l (mod 32), a shuffle hands each weight to the whole warp, and every
// lane keeps 16 partitions' vectors in flight (a row's reads are a chain of
// DRAM round trips otherwise).  Per dim the sum runs over j in order, as the
// definition reads.
constexpr int kReduceRowsPerCta = 4;
template <int D>
__global__ void __launch_bounds__(32 * kReduceRowsPerCta) paged_decode_reduce_kernel(
    const float* __restrict__ tmp_out, const float* __restrict__ max_logits,
    const float* __restrict__ exp_sums, const int32_t* __restrict__ context_lens, __half* out,
    int num_rows, int num_q_heads, int partition_size, int max_partitions, int min_partitions_to_merge,
    const int32_t* __restrict__ tail_order, const int32_t* __restrict__ tail_info) {
  static_assert(D == 64 || D == 128, "head_dim 64 or 128");
  constexpr int V = D / 32;
  constexpr int U = 16;  // partitions in flight per lane
  // launched as a programmatic dependent of the decode grid: wait until that
  // grid has completed and its partials are visible (a no-op otherwise)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = threadIdx.x & 31;
  int row = blockIdx.x * kReduceRowsPerCta + (threadIdx.x >> 5);  // b * Hq + h
  if (row >= num_rows) return;
  if (tail_order) {
    // a grid whose order split its tail (piece_order_kernel): rows of the
    // split sequences only, sequence t of them at order position
    // tail_info[0] + 2 t, its partitions tail_half_partition(L) long
    const int t = row / num_q_heads;
    if (t >= tail_info[1]) return;
    row = (tail_order[tail_info[0] + 2 * t] >> 2) * num_q_heads + row % num_q_heads;
  }
  const int b = row / num_q_heads;
  const int L = context_lens[b];
  const int PS = tail_order ? tail_half_partition(L) : partition_size;
  // partitions the first kernel wrote (none past its grid)
  const int np = min((L + PS - 1) / PS, max_partitions);
  // min_partitions_to_merge > 0: those sequences were written by the
  // partition kernel itself; 0 merges every sequence (empty ones get zeros)
  if (min_partitions_to_merge > 0 && np <= min_partitions_to_merge) return;
  __half* o_row = out + (size_t)row * D + V * lane;
  float acc[V];
#pragma unroll
  for (int v = 0; v < V; ++v) acc[v] = 0.f;
  float Z = 0.f;
  if (np > 0) {
    const float* ml = max_logits + (size_t)row * max_partitions;
    const float* es = exp_sums + (size_t)row * max_partitions;
    float M = -INFINITY;  // the maximum over partitions
    for (int j = lane; j < np; j += 32) M = fmaxf(M, ml[j]);
#pragma unroll
    for (int msk = 16; msk > 0; msk >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, msk));
    const float* to = tmp_out + (size_t)row * max_partitions * D + V * lane;
    for (int j0 = 0; j0 < np; j0 += 32) {
      float w = 0.f;  // the weight of partition j0 + lane
      if (j0 + lane < np) {
        const float m = ml[j0 + lane];
        w = m == -INFINITY ? 0.f : __expf(m - M);
        Z = fmaf(w, es[j0 + lane], Z);
      }
      const int nj = min(32, np - j0);
      int k = 0;
      for (; k + U <= nj; k += U) {
        float x[U][V];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const float* src = to + (size_t)(j0 + k + u) * D;
          if constexpr (V == 4) {
            const float4 t = *reinterpret_cast<const float4*>(src);
            x[u][0] = t.x; x[u][1] = t.y; x[u][2] = t.z; x[u][3] = t.w;
          } else {
            const float2 t = *reinterpret_cast<const float2*>(src);
            x[u][0] = t.x; x[u][1] = t.y;
          }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const float wu = __shfl_sync(0xffffffffu, w, k + u);
#pragma unroll
          for (int v = 0; v < V; ++v) acc[v] = fmaf(wu, x[u][v], acc[v]);
        }
      }
      for (; k < nj; ++k) {
        const float wu = __shfl_sync(0xffffffffu, w, k);
        const float* src = to + (size_t)(j0 + k) * D;
#pragma unroll
        for (int v = 0; v < V; ++v) acc[v] = fmaf(wu, src[v], acc[v]);
      }
    }
#pragma unroll
    for (int msk = 16; msk > 0; msk >>= 1) Z += __shfl_xor_sync(0xffffffffu, Z, msk);
  }
  const float invz = Z > 0.f ? 1.f / Z : 0.f;  // Z = 0: no token (empty sequence, or a query that saw none)
#pragma unroll
  for (int v = 0; v < V; v += 2)
    *reinterpret_cast<__half2*>(o_row + v) = __floats2half2_rn(acc[v] * invz, acc[v + 1] * invz);
}

// ---------------------------------------------------------------------------
// Paged KV append: the new token of sequence b sits at logical position
// L = context_lens[b], i.e. in physical block block_tables[b][L / BS], slot
// L % BS, for every kv head.  One thread moves one 16-byte chunk of the K
// row and the same chunk of the V row; a grid-stride loop covers
// num_seqs * Hkv * (D / 8) chunks.  Plain write-back stores: the rows are
// read by the decode step that follows, so they may as well stay in L2.
// Sequences without room in their table row, or whose entry is outside
// [0, num_blocks), are skipped and recorded as kErrBadBlock.
__global__ void __launch_bounds__(256) paged_kv_append_kernel(
    const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
    const int32_t* __restrict__ block_tables, const int32_t* __restrict__ context_lens,
    uint4* __restrict__ k_cache, uint4* __restrict__ v_cache, int num_seqs, int num_kv_heads,
    int chunks_per_row, int block_size, int num_blocks, int max_blocks_per_seq, int* error_word) {
  const long long total = (long long)num_seqs * num_kv_heads * chunks_per_row;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
    const long long row = i / chunks_per_row;  // b * Hkv + g
    const int c = (int)(i - row * chunks_per_row);
    const int b = (int)(row / num_kv_heads);
    const int g = (int)(row - (long long)b * num_kv_heads);
    // the new rows do not depend on the table walk: load them first so their
    // latency overlaps the dependent context-length -> block-id loads
    const uint4 kv = __ldg(k_new + i);
    const uint4 vv = __ldg(v_new + i);
    const int L = __ldg(context_lens + b);
    const int lb = L / block_size;
    if (L < 0 || lb >= max_blocks_per_seq) {
      if (g == 0 && c == 0) record_error(error_word, kErrBadBlock);
      continue;
    }
    const int p = __ldg(block_tables + (size_t)b * max_blocks_per_seq + lb);
    if (p < 0 || p >= num_blocks) {
      if (g == 0 && c == 0) record_error(error_word, kErrBadBlock);
      continue;
    }
    const size_t dst = (((size_t)p * num_kv_heads + g) * block_size + (L - lb * block_size)) *
                           (size_t)chunks_per_row + c;
    k_cache[dst] = kv;
    v_cache[dst] = vv;
  }
}

// ---------------------------------------------------------------------------
// Paged KV append into E4M3 caches: as paged_kv_append_kernel, with each
// element stored as e4m3(fp32(x) / scale) -- an IEEE fp32 division, then
// round-to-nearest-even onto the E4M3 grid saturating at +-448
// (cvt.rn.satfinite).  One thread writes 16 bytes (16 elements) of the K row
// and of the V row.
__device__ __forceinline__ uint32_t quant4_e4m3(const __half2 a, const __half2 b, float scale) {
  const float2 fa = __half22float2(a), fb = __half22float2(b);
  const float x0 = __fdiv_rn(fa.x, scale), x1 = __fdiv_rn(fa.y, scale);
  const float x2 = __fdiv_rn(fb.x, scale), x3 = __fdiv_rn(fb.y, scale);
  uint16_t lo, hi;
  // the second source lands in the low byte
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(x1), "f"(x0));
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(x3), "f"(x2));
  return (uint32_t)lo | ((uint32_t)hi << 16);
}

__device__ __forceinline__ uint4 quant16_e4m3(const uint4 a, const uint4 b, float scale) {
  auto h2 = [](uint32_t u) { return *reinterpret_cast<const __half2*>(&u); };
  return make_uint4(quant4_e4m3(h2(a.x), h2(a.y), scale), quant4_e4m3(h2(a.z), h2(a.w), scale),
                    quant4_e4m3(h2(b.x), h2(b.y), scale), quant4_e4m3(h2(b.z), h2(b.w), scale));
}

__global__ void __launch_bounds__(256) paged_kv_append_fp8_kernel(
    const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
    const int32_t* __restrict__ block_tables, const int32_t* __restrict__ context_lens,
    uint4* __restrict__ k_cache, uint4* __restrict__ v_cache, int num_seqs, int num_kv_heads,
    int chunks_per_row, int block_size, int num_blocks, int max_blocks_per_seq, float k_scale, float v_scale,
    int* error_word) {
  const long long total = (long long)num_seqs * num_kv_heads * chunks_per_row;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
    const long long row = i / chunks_per_row;  // b * Hkv + g
    const int c = (int)(i - row * chunks_per_row);
    const int b = (int)(row / num_kv_heads);
    const int g = (int)(row - (long long)b * num_kv_heads);
    // 16 fp16 inputs = two 16-byte loads, issued before the table walk
    const uint4 k0 = __ldg(k_new + 2 * i), k1 = __ldg(k_new + 2 * i + 1);
    const uint4 v0 = __ldg(v_new + 2 * i), v1 = __ldg(v_new + 2 * i + 1);
    const int L = __ldg(context_lens + b);
    const int lb = L / block_size;
    if (L < 0 || lb >= max_blocks_per_seq) {
      if (g == 0 && c == 0) record_error(error_word, kErrBadBlock);
      continue;
    }
    const int p = __ldg(block_tables + (size_t)b * max_blocks_per_seq + lb);
    if (p < 0 || p >= num_blocks) {
      if (g == 0 && c == 0) record_error(error_word, kErrBadBlock);
      continue;
    }
    const size_t dst = (((size_t)p * num_kv_heads + g) * block_size + (L - lb * block_size)) *
                           (size_t)chunks_per_row + c;
    k_cache[dst] = quant16_e4m3(k0, k1, k_scale);
    v_cache[dst] = quant16_e4m3(v0, v1, v_scale);
  }
}

// ---------------------------------------------------------------------------
// Gather of the used cache blocks from host memory: CTA (k, b) copies
// physical block block_tables[b][k] of K and of V (all kv heads: one
// contiguous run of chunks_per_block 16-byte chunks each) from the
// device-mapped host pools into the device pools, for k < ceil(L_b / BS).
// The host pools are read in place over the host link (16-byte loads), so
// only the blocks the tables reference cross it.  A block two sequences
// share is copied twice, with the same bytes.  Entries outside
// [0, num_blocks) are skipped and recorded as kErrBadBlock.
__global__ void __launch_bounds__(256) gather_used_blocks_kernel(
    const uint4* __restrict__ k_src, const uint4* __restrict__ v_src, uint4* __restrict__ k_dst,
    uint4* __restrict__ v_dst, const int32_t* __restrict__ block_tables,
    const int32_t* __restrict__ context_lens, int max_blocks_per_seq, int block_size, int num_blocks,
    long long chunks_per_block, int* error_word) {
  const int k = blockIdx.x, b = blockIdx.y;
  const int L = context_lens[b];
  if (L <= 0 || (long long)k * block_size >= L || k >= max_blocks_per_seq) return;
  const int p = block_tables[(size_t)b * max_blocks_per_seq + k];
  if (p < 0 || p >= num_blocks) {
    if (threadIdx.x == 0) record_error(error_word, kErrBadBlock);
    return;
  }
  const size_t base = (size_t)p * (size_t)chunks_per_block;
  for (long long i = threadIdx.x; i < chunks_per_block; i += blockDim.x) {
    const uint4 kv = k_src[base + i];
    const uint4 vv = v_src[base + i];
    k_dst[base + i] = kv;
    v_dst[base + i] = vv;
  }
}

// ---------------------------------------------------------------------------
// Longest-first order of the grid's pieces.  A piece is partition j of
// sequence b, (b, j) for j < NP; its tokens are min(PS, L_b - j PS), none
// past the context.  piece_order[p] = b * NP + j lists every piece once:
//   1. the full pieces (all but each sequence's last), by sequence and j;
//   2. each sequence's last piece, by decreasing tokens (ties by sequence);
//   3. the empty pieces (past a sequence's context), by sequence and j.
// A decode grid that walks p hands its longest work out first and ends on
// the shortest.  Unsplit (NP = 1) the pieces are the sequences, sorted by
// decreasing length.  Each CTA holds every sequence's piece count and last
// piece in shared memory and places the pieces of 128 sequences.  The decode
// grid reading the order is launched as its programmatic dependent.
//
// tail_seqs = K > 0 (unsplit grids, NP = 1): of the K shortest sequences
// with tokens (the grid's last round), those at least half as long as the
// batch's longest are split in two, each half its own piece, so that the
// round holds twice as many pieces of half the length (shorter ones already
// make a short round).  The split ones are the longest of the K, ranks
// [fs, fs + S) with fs = (sequences with tokens) - K.  The pieces are coded
// b * 4 + kPiece*: ranks below fs whole, then the two halves of each split
// sequence, then the other ranks whole, then the empty sequences, then -1 for
// the K - S slots left.  tail_info = {fs, S} tells the merge where the split
// sequences' first halves sit in the order.
constexpr int kOrderMaxSeqs = 4096;  // sequences held in shared memory (2 x 16 KiB)
__global__ void __launch_bounds__(128) piece_order_kernel(const int32_t* __restrict__ context_lens, int num_seqs,
                                                          int partition_size, int num_partitions,
                                                          int32_t* __restrict__ piece_order, int tail_seqs,
                                                          int32_t* __restrict__ tail_info) {
  __shared__ __align__(16) int32_t s_np[kOrderMaxSeqs];    // pieces with tokens
  __shared__ __align__(16) int32_t s_last[kOrderMaxSeqs];  // tokens of the last of them
  __shared__ int32_t s_lmax;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int PS = partition_size, NP = num_partitions;
  if (threadIdx.x == 0) s_lmax = 0;
  __syncthreads();
  // the sequences in quads (four per shared-memory read below); the padding
  // has no piece and so counts for nothing
  const int n4 = (num_seqs + 3) / 4;
  int lmax = 0;
  for (int i = threadIdx.x; i < 4 * n4; i += blockDim.x) {
    const int L = i < num_seqs ? max(context_lens[i], 0) : 0;
    const int n = min((L + PS - 1) / PS, NP);
    s_np[i] = n;
    s_last[i] = n > 0 ? L - (n - 1) * PS : 0;
    lmax = max(lmax, L);
  }
  if (tail_seqs > 0) atomicMax(&s_lmax, lmax);
  __syncthreads();
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= num_seqs) return;
  const int n_b = s_np[b], last_b = s_last[b];
  int full = 0, full_before = 0, lasts = 0, last_rank = 0, empty_before = 0;
  int half_long = 0;  // tail split: sequences with at least half the longest one's tokens
  const int lhalf = (s_lmax + 1) / 2;
  auto count = [&](int n, int li, int i) {
    const int f = n > 0 ? n - 1 : 0;
    const bool before = i < b;
    full += f;
    lasts += n > 0;
    half_long += n > 0 && li >= lhalf;
    full_before += before ? f : 0;
    empty_before += before ? NP - n : 0;
    last_rank += (n > 0) & ((li > last_b) | ((li == last_b) & before));
  };
#pragma unroll 4
  for (int q = 0; q < n4; ++q) {
    const int4 nn = reinterpret_cast<const int4*>(s_np)[q];
    const int4 ll = reinterpret_cast<const int4*>(s_last)[q];
    count(nn.x, ll.x, 4 * q);
    count(nn.y, ll.y, 4 * q + 1);
    count(nn.z, ll.z, 4 * q + 2);
    count(nn.w, ll.w, 4 * q + 3);
  }
  if (tail_seqs > 0) {  // NP = 1: full = 0, n_b is 0 or 1, last_rank the rank among sequences with tokens
    // (with NP = 1 the last piece's tokens are the sequence's, so the half-long
    // sequences are exactly ranks [0, half_long))
    const int fs = lasts - min(tail_seqs, lasts);
    const int S = max(0, min(half_long, lasts) - fs);
    if (n_b == 0)
      piece_order[lasts + S + empty_before] = b * 4 + kPieceWhole;
    else if (last_rank < fs)
      piece_order[last_rank] = b * 4 + kPieceWhole;
    else if (last_rank < fs + S) {
      const int at = fs + 2 * (last_rank - fs);
      piece_order[at] = b * 4 + kPieceFirstHalf;
      piece_order[at + 1] = b * 4 + kPieceSecondHalf;
    } else
      piece_order[last_rank + S] = b * 4 + kPieceWhole;
    if (b < tail_seqs - S) piece_order[num_seqs + S + b] = -1;
    if (b == 0) {
      tail_info[0] = fs;
      tail_info[1] = S;
    }
    return;
  }
  const int base = b * NP;
  for (int j = 0; j + 1 < n_b; ++j) piece_order[full_before + j] = base + j;
  if (n_b > 0) piece_order[full + last_rank] = base + n_b - 1;
  for (int j = n_b; j < NP; ++j) piece_order[full + lasts + empty_before + (j - n_b)] = base + j;
}

// ---------------------------------------------------------------------------
__global__ void validate_tables_kernel(const int32_t* block_tables, const int32_t* context_lens,
                                       int num_seqs, int max_blocks_per_seq, int block_size,
                                       int num_blocks, int* error_word) {
  const int b = blockIdx.x;
  if (b >= num_seqs) return;
  const int L = context_lens[b];
  if (L < 0 || L > max_blocks_per_seq * block_size) {
    if (threadIdx.x == 0) record_error(error_word, kErrBadBlock);
    return;
  }
  const int nb = (L + block_size - 1) / block_size;
  for (int i = threadIdx.x; i < nb; i += blockDim.x) {
    const int p = block_tables[(size_t)b * max_blocks_per_seq + i];
    if (p < 0 || p >= num_blocks) record_error(error_word, kErrBadBlock);
  }
}

// ---------------------------------------------------------------------------
// Self-test of the bounded waits: one CTA waits on a shared-memory barrier
// that no thread or copy will ever complete.  The wait gives up after
// budget_ns of %globaltimer, records kErrTimeout and the kernel returns.
__global__ void selftest_bounded_wait_kernel(int* error_word, unsigned long long budget_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbarrier_init();
  }
  __syncthreads();
  const bool ok = mbar_wait_bounded(&bar, 0, budget_ns);
  if (!ok && threadIdx.x == 0) record_error(error_word, kErrTimeout);
}

}  // namespace pkd
