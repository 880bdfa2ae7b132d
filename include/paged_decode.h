/*
 * paged_decode.h -- C ABI of libpaged_decode.so: single-query decode
 * attention over a paged fp16 KV cache, for NVIDIA GB300 (sm_103a).
 *
 * The operation (for every sequence b and query head h, kv head
 * g = h / (num_q_heads / num_kv_heads)):
 *
 *   p_t   = block_tables[b][t / block_size]            (physical block)
 *   s_t   = scale * dot(q[b][h][:], K[p_t][g][t % block_size][:])
 *   out[b][h][:] = sum_{t < L_b} softmax(s)_t * V[p_t][g][t % block_size][:]
 *
 * Sources: the paged cache and its logical->physical page table are
 * described in the CSDN answer "如何优化LLM推理引擎的内存访问延迟？"
 * (section 2, section 3); the per-head loop over a block table, with Q
 * resident, Q*K^T per K block and logits*V per V block, is section 3.2 and
 * Algorithm 1 (section 3.4) of the review "Accelerating LLM Inference
 * Throughput via Asynchronous KV Cache Prefetching"; its section 3.5 and
 * section 4.1 give the asynchronous L2 prefetch of upcoming K and V blocks
 * (cp.async.bulk.prefetch.L2) that the L2-prefetch variants issue.
 *
 * Layouts (all row-major, C order):
 *   q, out        fp16 [num_seqs][num_q_heads][head_dim]
 *   k_cache       fp16 [num_blocks][num_kv_heads][block_size][head_dim]
 *   v_cache       fp16 same layout as k_cache
 *   block_tables  int32 [num_seqs][max_blocks_per_seq]; entries at or past
 *                 ceil(context_lens[b] / block_size) are never read as
 *                 addresses (they may hold -1)
 *   context_lens  int32 [num_seqs], each in [0, max_context_len]
 * fp16 is IEEE binary16 passed as raw 16-bit words.  Every pointer named
 * "device" must be CUDA device memory (or managed memory) of the current
 * device.  K and V rows that are used must hold finite values.
 *
 * Ownership and threading: every buffer belongs to the caller.  The library
 * allocates no memory and may be called from several host threads at once.
 * The only state it keeps between calls is read-only: each device's SM
 * count, L2 size and memory bandwidth, queried on the first call that needs
 * them (the prefetch-distance model), and the device address of the
 * static-scratch array.  Work is enqueued on `stream` and the calls return
 * without waiting for it.
 *
 * Errors: arguments are checked on the host before any launch; a failed
 * check returns a status and launches nothing.  PKD_ERR_LAUNCH reports a
 * CUDA launch failure.  Device-side problems (a block-table entry outside
 * [0, num_blocks), or a bounded wait that ran out) are recorded in the
 * optional `error_word` (device int, nullable): the kernel ORs PKD_DEVERR_*
 * bits into it and skips the affected work; read it with
 * pkd_read_device_error().
 */
#ifndef PAGED_DECODE_H_
#define PAGED_DECODE_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PKD_OK = 0,
  PKD_ERR_NULL = 1,         /* a required pointer is NULL */
  PKD_ERR_SHAPE = 2,        /* a size is out of range or inconsistent */
  PKD_ERR_UNSUPPORTED = 3,  /* head_dim / block_size / group size not compiled */
  PKD_ERR_ALIGN = 4,        /* a pointer is not 16-byte aligned */
  PKD_ERR_WORKSPACE = 5,    /* workspace missing or smaller than required */
  PKD_ERR_LAUNCH = 6,       /* the CUDA launch failed */
  PKD_ERR_DEVICE = 7,       /* the device reported an error (error word set) */
  PKD_ERR_CUDA = 8          /* a CUDA runtime query failed */
} pkd_status;

/* Bits of the device error word. */
#define PKD_DEVERR_BAD_BLOCK 1u /* a used block-table entry was outside [0, num_blocks), or a
                                   context length ran past its block-table row (the kernels
                                   then read only the row's blocks; that sequence's output is
                                   undefined, and nothing outside the inputs is read) */
#define PKD_DEVERR_TIMEOUT 2u   /* a bounded wait on a shared-memory barrier ran out */
#define PKD_DEVERR_LAYOUT 4u    /* a CTA's dynamic shared memory did not start 1024-byte aligned
                                   (the tcgen05 kernel relies on it for its swizzled operands and
                                   then computes nothing for that CTA; not seen on sm_103a) */

/* How K/V tiles reach the arithmetic.  All variants give the same result. */
typedef enum {
  PKD_VARIANT_AUTO = 0,        /* chosen per launch, see paged_decode_auto_variant */
  PKD_VARIANT_NO_PREFETCH = 1, /* each warp loads its current blocks (16-byte loads) */
  PKD_VARIANT_L2_PREFETCH = 2, /* as 1, plus cp.async.bulk.prefetch.L2 of blocks ahead */
  PKD_VARIANT_TMA_STAGED = 3,  /* bulk copies into a shared-memory ring, plus L2 prefetch */
  PKD_VARIANT_TMA_MMA = 4,     /* 128-byte-swizzled tensor copies into a shared-memory ring (L2
                                  prefetch beyond it with prefetch_distance >= 1); Q.K^T and P.V
                                  on the tensor cores (mma, fp16 operands, fp32 accumulation; p
                                  rounded to fp16 for P.V) */
  PKD_VARIANT_TCGEN05 = 5      /* the same copies into K and V rings of 64-token tiles; Q.K^T
                                  and P.V as tcgen05 MMAs with S and O in tensor memory, one
                                  softmax thread per query row; up to 64 query rows (query
                                  tokens x group heads) share one read of the K/V tiles.
                                  fp16 caches at head_dim 64 or 128 by this variant; E4M3
                                  caches at head_dim 128 through paged_decode_attention_fp8
                                  (its automatic choice) or _fp8_ex (on request), the bytes
                                  widened to fp16 in shared memory; PKD_ERR_UNSUPPORTED
                                  otherwise */
} pkd_variant;

/*
 * Flag bits that may be ORed into a `variant` argument.
 *   PKD_FLAG_L2_EVICT_HINTS  give the KV stream L2 eviction priorities: the
 *       loads or bulk copies that consume a K/V tile mark it evict_first (it
 *       is never read again), and L2 prefetches of tiles ahead mark them
 *       evict_last until they are consumed.  This is the "adjust eviction
 *       priority" mitigation for prefetched blocks overflowing L2 in section
 *       4.2 of the review "Accelerating LLM Inference Throughput via
 *       Asynchronous KV Cache Prefetching".  Results are unchanged.
 */
#define PKD_FLAG_L2_EVICT_HINTS 0x100
/*
 *   PKD_FLAG_LONGEST_FIRST  hand the decode grid's work out longest first:
 *       a kernel of one CTA per 128 sequences orders the grid's pieces
 *       (partition j of sequence b) into the workspace: the full partitions,
 *       then each sequence's last partition by decreasing length, then the
 *       empty ones.  The tensor-core decode grid walks that order, so the
 *       last CTAs to start hold the shortest work and the tail of a ragged
 *       batch shortens.  Unsplit, this is the sequences by decreasing
 *       length.  Results are unchanged.  Tensor-core path only, batches of
 *       2..4096 sequences; elsewhere it is ignored.  The workspace grows by
 *       the order, one int32 per piece (paged_decode_workspace_size counts
 *       it, after the split partials); a workspace without that room runs
 *       the plain order.
 */
#define PKD_FLAG_LONGEST_FIRST 0x200

/*
 * paged_decode_attention -- the whole operation, one partition per
 * (sequence, kv head): out[b][h][:] as defined above.  No workspace.
 *
 *   q, k_cache, v_cache, block_tables, context_lens : device, layouts above
 *   out            device fp16 [num_seqs][num_q_heads][head_dim] (written)
 *   num_seqs       >= 0 (0: nothing is launched)
 *   num_q_heads    multiple of num_kv_heads; group = num_q_heads/num_kv_heads
 *                  in 1..8
 *   head_dim       64 or 128
 *   block_size     16 or 32
 *   num_blocks     physical blocks in k_cache / v_cache (> 0)
 *   max_blocks_per_seq  row length of block_tables (> 0)
 *   max_context_len     host upper bound of context_lens (sizes the grid)
 *   scale          softmax scale applied to q.k (e.g. 1/sqrt(head_dim))
 *   stream         CUDA stream (0 = legacy default stream)
 * Sequences with context length 0 get out = 0.
 */
pkd_status paged_decode_attention(const void* q, const void* k_cache, const void* v_cache,
                                  const int32_t* block_tables, const int32_t* context_lens, void* out,
                                  int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                  int block_size, int num_blocks, int max_blocks_per_seq,
                                  int max_context_len, float scale, cudaStream_t stream);

/*
 * paged_decode_attention_host -- the whole operation from host buffers: the
 * inputs are copied to the caller's device buffers, the automatic decode
 * (as paged_decode_attention_ex with PKD_VARIANT_AUTO and partition_size 0)
 * runs on them, and out is copied back; every step is asynchronous on
 * `stream`, and the host `out` holds the result once the stream has
 * reached this point.
 *
 *   q, k_cache, v_cache, block_tables, context_lens, out
 *                  host buffers, layouts as above; page-locked (cudaHostAlloc
 *                  or cudaHostRegister) for the copies to be asynchronous
 *   q_dev, k_cache_dev, v_cache_dev, block_tables_dev, context_lens_dev, out_dev
 *                  device buffers of the same sizes (owned by the caller)
 *   used_blocks_only  non-zero: K and V cross the host link only for the
 *                  blocks the tables reference (context_lens[b] tokens of
 *                  sequence b, read in place from the mapped host pools by
 *                  a gather kernel); blocks of k_cache_dev / v_cache_dev that
 *                  no sequence references keep their old contents.  When the
 *                  host pools are not mapped into the device's address space,
 *                  or with 0, each pool is copied whole.
 *   workspace, workspace_bytes, error_word: as for paged_decode_attention_ex
 *                  (paged_decode_workspace_size with partition_size 0 and
 *                  PKD_VARIANT_AUTO); error_word is device memory
 * Other arguments as for paged_decode_attention_ex.  Returns PKD_ERR_CUDA if
 * a copy cannot be enqueued.
 */
pkd_status paged_decode_attention_host(const void* q, const void* k_cache, const void* v_cache,
                                       const int32_t* block_tables, const int32_t* context_lens, void* out,
                                       void* q_dev, void* k_cache_dev, void* v_cache_dev,
                                       int32_t* block_tables_dev, int32_t* context_lens_dev, void* out_dev,
                                       int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                       int block_size, int num_blocks, int max_blocks_per_seq,
                                       int max_context_len, float scale, int used_blocks_only, void* workspace,
                                       size_t workspace_bytes, int* error_word, cudaStream_t stream);

/*
 * paged_decode_attention_ex -- as paged_decode_attention, with control over
 * the context split and the data path.
 *
 *   partition_size  tokens per context partition (split-K): 0 = choose
 *                   automatically from the shape and the GPU; -1 = never
 *                   split; otherwise a positive multiple of 32 (and of
 *                   block_size).  A sequence longer than one partition is
 *                   computed by one CTA per (sequence, kv head, partition)
 *                   and merged by the split-K reduce; shorter ones are
 *                   written directly.  On the tcgen05 path at head_dim 128,
 *                   partitions of up to 1024 tokens (multiples of 64) of a
 *                   grid walked in plain order are taken in runs: one CTA
 *                   streams up to 4096 tokens of consecutive partitions of
 *                   its (sequence, kv head) and writes each one's partial,
 *                   while the grid keeps four waves of CTAs; the result is
 *                   the same.  On the tcgen05 path an unsplit grid walked
 *                   longest first whose last round of resident CTAs would
 *                   be at most half full has that round's sequences, those
 *                   at least half as long as the batch's longest, split in
 *                   two halves merged like partitions (when the workspace
 *                   has room: the *_workspace_size functions count it for
 *                   partition_size 0).  The automatic choice splits only
 *                   grids of fewer than two waves of (sequence, kv head)
 *                   units (on the mma.sync path also contexts of 8192
 *                   tokens or more below six waves), into power-of-two
 *                   partitions: for units below one resident wave the
 *                   shortest one (from 128 tokens, 256 on the tcgen05
 *                   path) whose grid still fits that wave, else from 512
 *                   tokens up, sized for six waves.  It walks unsplit
 *                   grids of one to six waves longest first
 *                   (PKD_FLAG_LONGEST_FIRST) when the workspace has room
 *                   for the order.
 *   variant         pkd_variant, optionally ORed with PKD_FLAG_* bits
 *   prefetch_distance  how many of a warp's iterations ahead the L2 prefetch
 *                   runs: -1 = no L2 prefetch; 0 = the default of the L2
 *                   capacity model (paged_decode_prefetch_model: the
 *                   smallest distance whose bytes in flight cover the HBM
 *                   latency, 0 when the ring of copies alone covers it,
 *                   capped so the prefetched blocks stay within an eighth of
 *                   L2); >= 1 = that distance.  Ignored by
 *                   PKD_VARIANT_NO_PREFETCH and PKD_VARIANT_TCGEN05.
 *   workspace, workspace_bytes  device scratch of at least
 *                   paged_decode_workspace_size(...) bytes, 256-byte aligned
 *                   (may be NULL when no sequence is split; the automatic
 *                   order then falls back to the plain one)
 *   error_word      device int or NULL; see "Errors" above
 * Calls that share a workspace must not overlap on the GPU.
 */
pkd_status paged_decode_attention_ex(const void* q, const void* k_cache, const void* v_cache,
                                     const int32_t* block_tables, const int32_t* context_lens,
                                     void* out, int num_seqs, int num_q_heads, int num_kv_heads,
                                     int head_dim, int block_size, int num_blocks,
                                     int max_blocks_per_seq, int max_context_len, float scale,
                                     int partition_size, int variant, int prefetch_distance,
                                     void* workspace, size_t workspace_bytes, int* error_word,
                                     cudaStream_t stream);

/*
 * The partition size paged_decode_attention_ex uses when given 0 with this
 * `variant` (a positive multiple of 32, or -1 when it would not split), for
 * the current device.  Returns -2 on invalid sizes.
 */
int paged_decode_auto_partition_size(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                     int block_size, int max_context_len, int variant);

/*
 * Workspace bytes paged_decode_attention_ex needs for a split into
 * partitions of partition_size tokens (0 = automatic for `variant`, as
 * above): the fp32
 * partials [num_seqs][num_q_heads][NP][head_dim] and the per-partition
 * max and sum [num_seqs][num_q_heads][NP], NP = ceil(max_context_len /
 * partition_size), then, for partition_size 0 or PKD_FLAG_LONGEST_FIRST,
 * the longest-first order (num_seqs x NP int32, NP = 1 unsplit), each region
 * 256-byte aligned.
 * 0 when nothing splits and no order is kept.
 */
/*
 * paged_decode_auto_variant -- the variant value (data path ORed with
 * PKD_FLAG_* bits) that PKD_VARIANT_AUTO runs for this shape, on the current
 * device, given partition_size as passed to paged_decode_attention_ex (0 =
 * automatic, -1 = unsplit, or a partition).  It is TMA_MMA; with
 * partition_size 0 it carries PKD_FLAG_LONGEST_FIRST where the automatic
 * choice orders the batch.
 * Returns -2 on an invalid shape or partition size.
 */
int paged_decode_auto_variant(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                              int block_size, int max_context_len, int partition_size);

size_t paged_decode_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                   int block_size, int max_context_len, int partition_size,
                                   int variant);

/*
 * paged_decode_partitions -- the first split-K kernel alone: for every
 * (b, h) and partition j < ceil(L_b / partition_size), covering logical
 * tokens [j*P, min((j+1)*P, L_b)):
 *   max_logits[b][h][j] = max_t s_t
 *   exp_sums[b][h][j]   = sum_t exp(s_t - max_logits)
 *   tmp_out[b][h][j][:] = sum_t exp(s_t - max_logits) * v_t   (not normalised)
 * Entries of partitions past ceil(L_b / P) are not written.
 *   tmp_out     device fp32 [num_seqs][num_q_heads][max_num_partitions][head_dim]
 *   max_logits, exp_sums  device fp32 [num_seqs][num_q_heads][max_num_partitions]
 *   max_num_partitions >= ceil(max_context_len / partition_size)
 * partition_size is a positive multiple of 32 and of block_size.
 */
pkd_status paged_decode_partitions(const void* q, const void* k_cache, const void* v_cache,
                                   const int32_t* block_tables, const int32_t* context_lens,
                                   int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                   int block_size, int num_blocks, int max_blocks_per_seq,
                                   int max_context_len, float scale, int partition_size,
                                   int variant, int prefetch_distance, float* tmp_out,
                                   float* max_logits, float* exp_sums, int max_num_partitions,
                                   int* error_word, cudaStream_t stream);

/*
 * paged_decode_reduce -- the split-K merge (log-sum-exp identity):
 *   M = max_j max_logits[b][h][j],  w_j = exp(max_logits_j - M)
 *   out[b][h][:] = sum_j w_j * tmp_out[b][h][j][:] / sum_j w_j * exp_sums[b][h][j]
 * over j < ceil(L_b / partition_size).  Sequences with
 * ceil(L_b / partition_size) <= min_partitions_to_merge are left untouched
 * (pass 0 to merge every sequence; a sequence with L_b = 0 then gets 0).
 * Layouts as in paged_decode_partitions; out device fp16.
 */
pkd_status paged_decode_reduce(const float* tmp_out, const float* max_logits, const float* exp_sums,
                               const int32_t* context_lens, void* out, int num_seqs, int num_q_heads,
                               int head_dim, int partition_size, int max_num_partitions,
                               int min_partitions_to_merge, cudaStream_t stream);

/*
 * paged_decode_validate_tables -- debug check: ORs PKD_DEVERR_BAD_BLOCK into
 * *error_word (device int, required) if any entry
 * block_tables[b][i], i < ceil(context_lens[b] / block_size), lies outside
 * [0, num_blocks), or a context length is negative or longer than the row.
 */
pkd_status paged_decode_validate_tables(const int32_t* block_tables, const int32_t* context_lens,
                                        int num_seqs, int max_blocks_per_seq, int block_size,
                                        int num_blocks, int* error_word, cudaStream_t stream);

/*
 * paged_decode_attention_multi -- decode of q_len > 1 new tokens per
 * sequence at once (verifying q_len draft tokens of speculative decoding in
 * one pass; the review "Accelerating LLM Inference Throughput via
 * Asynchronous KV Cache Prefetching", section 7.4, names working together
 * with speculative decoding as a direction).  The q_len new tokens are the
 * last q_len positions of each sequence and are already in the cache
 * (paged_kv_append, or the caller's own write); query jq of sequence b sits
 * at position L_b - q_len + jq and attends to every token up to and including
 * its own position:
 *   out[b][jq][h][:] = sum_{t <= L_b - q_len + jq} softmax(s)_t * V[..t..]
 * A query that sees no token (L_b - q_len + jq < 0) gets out = 0.
 *
 *   q, out         device fp16 [num_seqs][q_len][num_q_heads][head_dim]
 *   q_len          >= 1 (1 gives single-query decode)
 *   other arguments as for paged_decode_attention_ex; context_lens[b] counts
 *   the new tokens.  Runs a tensor-core path (PKD_VARIANT_AUTO of
 *   paged_decode_attention_multi_ex): where the rows of a (sequence, kv
 *   head), q_len x G, fit one 16-row tile, PKD_VARIANT_TMA_MMA, whose CTAs
 *   serve 16 / G query tokens each; otherwise PKD_VARIANT_TCGEN05, whose CTAs
 *   serve 64 / G, so every K/V tile is read once per group of 64 / G query
 *   tokens.
 *   workspace      required when the context is split
 *                  (paged_decode_multi_workspace_size bytes, 256-byte aligned);
 *                  with partition_size 0 it also keeps the longest-first
 *                  order (NULL then runs the plain order)
 */
pkd_status paged_decode_attention_multi(const void* q, const void* k_cache, const void* v_cache,
                                        const int32_t* block_tables, const int32_t* context_lens,
                                        void* out, int num_seqs, int q_len, int num_q_heads,
                                        int num_kv_heads, int head_dim, int block_size, int num_blocks,
                                        int max_blocks_per_seq, int max_context_len, float scale,
                                        int partition_size, void* workspace, size_t workspace_bytes,
                                        int* error_word, cudaStream_t stream);

/*
 * paged_decode_attention_multi_ex -- paged_decode_attention_multi with the
 * data path chosen by the caller: variant PKD_VARIANT_AUTO (the choice
 * paged_decode_attention_multi makes), PKD_VARIANT_TMA_MMA or
 * PKD_VARIANT_TCGEN05, optionally ORed with PKD_FLAG_* bits
 * (PKD_ERR_UNSUPPORTED for the CUDA-core paths when q_len > 1).  Both
 * tensor-core paths give the same result up to fp32 rounding order.
 */
pkd_status paged_decode_attention_multi_ex(const void* q, const void* k_cache, const void* v_cache,
                                           const int32_t* block_tables, const int32_t* context_lens,
                                           void* out, int num_seqs, int q_len, int num_q_heads,
                                           int num_kv_heads, int head_dim, int block_size, int num_blocks,
                                           int max_blocks_per_seq, int max_context_len, float scale,
                                           int partition_size, int variant, void* workspace,
                                           size_t workspace_bytes, int* error_word, cudaStream_t stream);

/*
 * paged_decode_call_plan -- the launch plan of a decode call on the current
 * device: q_len query tokens per sequence, kv_fp8 1 for E4M3 caches, and the
 * partition_size and variant the call is given.  Writes *partition_out (the
 * partition, or -1 when unsplit), *longest_first (1 when the batch is walked
 * longest first, given a workspace of the size the *_workspace_size
 * functions return), *variant_out (the data path with the PKD_FLAG_* bits
 * that apply), *grid_out (decode CTAs; with the tcgen05 path's split of a
 * short last round, room for its extra halves) and *prefetch_distance_out
 * (the L2 prefetch distance the call runs with prefetch_distance 0; 0 =
 * none); any pointer may be NULL.
 * Returns the kernel launches (decode grid, split-K merge, order kernel; 0
 * for an empty batch), or -2 for a shape, partition or variant the call
 * would refuse.
 */
int paged_decode_call_plan(int num_seqs, int q_len, int num_q_heads, int num_kv_heads, int head_dim,
                           int block_size, int max_context_len, int kv_fp8, int partition_size, int variant,
                           int* partition_out, int* longest_first, int* variant_out, long long* grid_out,
                           int* prefetch_distance_out);

/*
 * pkd_l2_prefetch_model -- the rule that sizes the default L2 prefetch
 * distance, as plain host arithmetic (no GPU is needed).  Source: section
 * 4.2 of the review "Accelerating LLM Inference Throughput via Asynchronous
 * KV Cache Prefetching": a (block, head) tile is M_block = b * d_h * T_block
 * bytes, and the prefetched tiles of one iteration of every warp occupy
 * M_total = M_block * (N_thread / 32) * H * B of L2, which must fit in it.
 * For resident_ctas CTAs in flight on sm_count SMs, each with
 * streams_per_cta warps (block streams) that prefetch tiles_per_step tiles of
 * m_block bytes per unit of distance d:
 *   footprint(d) = resident_ctas * d * streams_per_cta * tiles_per_step * m_block
 *     (M_total, with H * B the CTAs in flight and d tiles per warp)
 *   inflight(d)  = resident_ctas / active_sms * (ahead_bytes_per_cta + footprint(d) / resident_ctas)
 *   need         = hbm_bytes_per_s / active_sms * latency_s   (Little's law)
 * with active_sms = min(sm_count, resident_ctas).  Returns the smallest d in
 * [0, max_distance] with inflight(d) >= need, then lowered until
 * footprint(d) <= l2_fraction * l2_bytes (0 when no d >= 1 fits), and writes
 * footprint(d), inflight(d) and need (bytes; pointers may be NULL).  Returns
 * -2 for a negative size or fraction, or sm_count, streams_per_cta, m_block or
 * tiles_per_step <= 0.
 */
int pkd_l2_prefetch_model(long long resident_ctas, int sm_count, int streams_per_cta, long long m_block,
                          int tiles_per_step, long long ahead_bytes_per_cta, long long l2_bytes,
                          double l2_fraction, double hbm_bytes_per_s, double latency_s, int max_distance,
                          long long* footprint_bytes, long long* inflight_bytes_per_sm,
                          long long* need_bytes_per_sm);

/*
 * paged_decode_prefetch_model -- the default L2 prefetch distance
 * (prefetch_distance 0) of a decode call, for a GPU described by sm_count,
 * l2_bytes and hbm_bytes_per_s (its nominal bandwidth) instead of the
 * current device: pkd_l2_prefetch_model over the call's resident CTAs, with
 * the data path's warps per CTA, two tiles (K and V) of block_size x
 * head_dim elements per unit of distance, the bytes its ring or loads keep
 * in flight, an eighth of L2 and a loaded HBM latency of 1.5 us, and no
 * more blocks ahead than a warp's share of the partition holds.  The call's
 * partition and data path are planned as by paged_decode_call_plan (the
 * automatic split on the current device, or the fallback SM count without
 * one).  Writes the model's footprint, in-flight and need bytes (pointers
 * may be NULL).  Returns the distance (0 for paths that never prefetch to
 * L2), or -2 for an invalid shape, variant or description.
 */
int paged_decode_prefetch_model(int num_seqs, int q_len, int num_q_heads, int num_kv_heads, int head_dim,
                                int block_size, int max_context_len, int kv_fp8, int partition_size, int variant,
                                int sm_count, long long l2_bytes, double hbm_bytes_per_s,
                                long long* footprint_bytes, long long* inflight_bytes_per_sm,
                                long long* need_bytes_per_sm);

/*
 * paged_decode_auto_plan -- what a call with partition_size 0 runs on the
 * current device: paged_decode_attention_ex with PKD_VARIANT_AUTO (q_len 1,
 * kv_fp8 0), paged_decode_attention_multi (q_len > 1) or
 * paged_decode_attention_fp8 (kv_fp8 1).  Writes *partition_size (the
 * partition, or -1 when unsplit) and *longest_first (1 when the batch is
 * walked longest first, given a workspace of the size the *_workspace_size
 * functions return); either pointer may be NULL.  Returns the kernel launches
 * the call makes (the decode grid, plus the split-K merge when split or when
 * the order splits a short last round on the tcgen05 path, plus the order
 * kernel; 0 for an empty batch), or -2 on an invalid shape.
 */
int paged_decode_auto_plan(int num_seqs, int q_len, int num_q_heads, int num_kv_heads, int head_dim,
                           int block_size, int max_context_len, int kv_fp8, int* partition_size,
                           int* longest_first);

/* Workspace bytes paged_decode_attention_multi, paged_decode_attention_multi_ex
   (every variant) and paged_decode_attention_fp8 need (0 = none). */
size_t paged_decode_multi_workspace_size(int num_seqs, int q_len, int num_q_heads, int num_kv_heads,
                                         int head_dim, int block_size, int max_context_len,
                                         int partition_size);

/*
 * paged_decode_attention_fp8 -- decode over FP8 (E4M3) KV caches: k_cache
 * and v_cache hold one byte per element, same [num_blocks][num_kv_heads]
 * [block_size][head_dim] layout, with value = e4m3(byte) * k_scale for K and
 * * v_scale for V (E4M3: 1 sign, 4 exponent bits with bias 7, 3 mantissa
 * bits, no infinities, largest magnitude 448).  Source: the CSDN answer
 * "如何优化LLM推理引擎的内存访问延迟？", section 4 (FP8 precision to shrink
 * the KV footprint); the byte format and the per-cache scale are this
 * library's reading.  Halves the K/V bytes a step reads.
 *
 *   q, out         fp16, [num_seqs][q_len][num_q_heads][head_dim] (q_len = 1:
 *                  single-query decode; q_len > 1: causal as in
 *                  paged_decode_attention_multi)
 *   k_cache, v_cache  device E4M3 bytes, 16-byte aligned
 *   k_scale, v_scale  finite, > 0
 *   other arguments as for paged_decode_attention_multi (workspace:
 *   paged_decode_multi_workspace_size bytes when the context is split).
 * The scores use the exact fp16 value of every code (all E4M3 values are
 * fp16 values); the K scale multiplies the softmax scale, and the V scale the
 * result.  Codes that are NaN (0x7f, 0xff) must not appear in used rows.
 * Data path, as for paged_decode_attention_multi: PKD_VARIANT_TMA_MMA where
 * the q_len x G rows of a (sequence, kv head) fit one 16-row tile or
 * head_dim is 64, else PKD_VARIANT_TCGEN05.
 */
pkd_status paged_decode_attention_fp8(const void* q, const void* k_cache, const void* v_cache,
                                      const int32_t* block_tables, const int32_t* context_lens, void* out,
                                      int num_seqs, int q_len, int num_q_heads, int num_kv_heads,
                                      int head_dim, int block_size, int num_blocks, int max_blocks_per_seq,
                                      int max_context_len, float scale, float k_scale, float v_scale,
                                      int partition_size, void* workspace, size_t workspace_bytes,
                                      int* error_word, cudaStream_t stream);

/*
 * paged_decode_attention_fp8_ex -- paged_decode_attention_fp8 with the data
 * path chosen by the caller: variant PKD_VARIANT_AUTO (the choice
 * paged_decode_attention_fp8 makes), PKD_VARIANT_TMA_MMA or
 * PKD_VARIANT_TCGEN05 (head_dim 128), optionally ORed with PKD_FLAG_* bits;
 * PKD_ERR_UNSUPPORTED for the CUDA-core paths.  Both tensor-core paths give
 * the same result up to fp32 rounding order.
 */
pkd_status paged_decode_attention_fp8_ex(const void* q, const void* k_cache, const void* v_cache,
                                         const int32_t* block_tables, const int32_t* context_lens, void* out,
                                         int num_seqs, int q_len, int num_q_heads, int num_kv_heads,
                                         int head_dim, int block_size, int num_blocks, int max_blocks_per_seq,
                                         int max_context_len, float scale, float k_scale, float v_scale,
                                         int partition_size, int variant, void* workspace, size_t workspace_bytes,
                                         int* error_word, cudaStream_t stream);

/*
 * paged_kv_append_fp8 -- paged_kv_append into E4M3 caches: every element x
 * of the new fp16 rows is stored as e4m3(fp32(x) / scale), the division in
 * IEEE fp32 and the conversion round-to-nearest-even, saturating at +-448
 * (k_scale for K, v_scale for V; finite, > 0).  head_dim a multiple of 16;
 * k_cache / v_cache are E4M3 bytes.  Arguments and errors otherwise as for
 * paged_kv_append.
 */
pkd_status paged_kv_append_fp8(const void* k_new, const void* v_new, const int32_t* block_tables,
                               const int32_t* context_lens, void* k_cache, void* v_cache, int num_seqs,
                               int num_kv_heads, int head_dim, int block_size, int num_blocks,
                               int max_blocks_per_seq, float k_scale, float v_scale, int* error_word,
                               cudaStream_t stream);

/*
 * paged_kv_append -- the cache write that precedes each decode step: stores
 * one new token's K and V rows per sequence into the paged cache, at the
 * sequence's next logical position.  With L = context_lens[b] (the length
 * BEFORE the append) and for every kv head g:
 *   p = block_tables[b][L / block_size]
 *   K[p][g][L % block_size][:] = k_new[b][g][:]
 *   V[p][g][L % block_size][:] = v_new[b][g][:]
 * Source: the CSDN answer "如何优化LLM推理引擎的内存访问延迟？", section 2:
 * each sequence's KV lives in the pages its page table lists, filled in
 * logical order.  The caller allocates block_tables[b][L / block_size]
 * beforehand when L is a multiple of block_size, and raises context_lens[b]
 * to L + 1 afterwards (the library does neither).
 *
 *   k_new, v_new   device fp16 [num_seqs][num_kv_heads][head_dim], 16-byte aligned
 *   block_tables, context_lens   device int32, layouts as for the decode calls
 *   k_cache, v_cache   device fp16 [num_blocks][num_kv_heads][block_size][head_dim],
 *                  16-byte aligned, written in place (only the target rows)
 *   head_dim       any positive multiple of 8; block_size any positive size
 *   error_word     device int, nullable: PKD_DEVERR_BAD_BLOCK is ORed in for a
 *                  sequence with L < 0, L / block_size >= max_blocks_per_seq,
 *                  or a table entry outside [0, num_blocks); such a sequence
 *                  is skipped (nothing is written for it).
 * Every other row of the caches is left untouched, bit for bit.  Two
 * sequences whose targets coincide (a shared block) race: the caller keeps
 * appended-to blocks private to one sequence.
 */
pkd_status paged_kv_append(const void* k_new, const void* v_new, const int32_t* block_tables,
                           const int32_t* context_lens, void* k_cache, void* v_cache, int num_seqs,
                           int num_kv_heads, int head_dim, int block_size, int num_blocks,
                           int max_blocks_per_seq, int* error_word, cudaStream_t stream);

/*
 * pkd_selftest_bounded_wait -- exercises the failure path of the library's
 * bounded waits without faulting or hanging the GPU: launches one CTA that
 * waits on a shared-memory barrier nothing will complete; after budget_ns
 * nanoseconds (1e3 .. 1e8) of the GPU's global timer the wait gives up, ORs
 * PKD_DEVERR_TIMEOUT into *error_word (device int, required) and the kernel
 * returns normally.  Every wait in the decode kernels behaves the same way
 * with a 100 ms budget.
 */
pkd_status pkd_selftest_bounded_wait(int* error_word, unsigned long long budget_ns, cudaStream_t stream);

/*
 * pkd_read_device_error -- synchronises `stream`, copies *error_word to
 * *host_bits, and returns PKD_OK when it is 0, PKD_ERR_DEVICE otherwise.
 * Clears the word when `clear` is non-zero.
 */
pkd_status pkd_read_device_error(int* error_word, unsigned* host_bits, int clear, cudaStream_t stream);

/*
 * paged_decode_attention_static_scratch -- the split-K path of
 * paged_decode_attention_ex for callers that cannot allocate device memory
 * (code running under another framework's allocator, plugins that only
 * receive input and output pointers, processes that reserved the whole pool
 * ahead of time).  The pages have no counterpart: this is a property of the
 * library interface, not of the method.
 *
 * The caller passes inputs and the output exactly as for
 * paged_decode_attention_ex (same meanings; partition_size 0 = automatic,
 * otherwise a positive multiple of 32 and of block_size).  The per-partition
 * partials live in a library-owned device array of PKD_STATIC_SCRATCH_BYTES
 * bytes that every GPU which loads the library holds until the process
 * exits; no memory is allocated and no allocating routine is called.
 *   - A shape whose partials need more than PKD_STATIC_SCRATCH_BYTES
 *     (B * Hq * NP * (head_dim + 2) * 4 bytes plus alignment) is rejected
 *     with PKD_ERR_WORKSPACE before anything is launched.
 *   - The first call on a device looks up the array's device address (with
 *     that device current); make that first call before any stream capture.
 *     The address is kept for the life of the process, so this entry must
 *     not be used on a device after cudaDeviceReset (or any other teardown
 *     of its primary context) in the same process: the kept address would
 *     no longer name the array.
 *   - Every call shares the one array, and each call leaves its partials in
 *     it; nothing in it needs to start at zero.  Calls that overlap on the
 *     GPU (other streams, other host threads) race on the array: serialise
 *     them.
 */
#define PKD_STATIC_SCRATCH_BYTES (64u << 20)
pkd_status paged_decode_attention_static_scratch(
    const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
    const int32_t* context_lens, void* out, int num_seqs, int num_q_heads, int num_kv_heads,
    int head_dim, int block_size, int num_blocks, int max_blocks_per_seq, int max_context_len,
    float scale, int partition_size, int variant, int prefetch_distance, int* error_word,
    cudaStream_t stream);

/* Static text for a status code. */
const char* pkd_status_string(int status);

/* Library version, major*10000 + minor*100 + patch. */
int pkd_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGED_DECODE_H_ */
