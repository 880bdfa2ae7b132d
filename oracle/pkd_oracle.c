/*
 * pkd_oracle.c -- CPU oracle for single-query decode attention over a paged
 * fp16 KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, plain fp64 statement of
 * what the CUDA library computes; only the tests, the package's smoke check
 * and the benchmark's CPU-baseline leg may load it.  It shares no code,
 * header, table or helper with the CUDA path.
 *
 * What it computes (the plain definition; prefetching changes timing only):
 *
 *   for sequence b, query head h, kv head g = h / (Hq / Hkv):
 *     for logical token t in [0, L_b):
 *        p   = block_tables[b][t / bs]          physical block (page)
 *        k_t = K[p][g][t % bs][:],  v_t = V[p][g][t % bs][:]
 *        s_t = scale * sum_d q[b][h][d] * k_t[d]
 *     w_t = exp(s_t - max_u s_u) / sum_u exp(s_u - max_u s_u)
 *     out[b][h][:] = sum_t w_t * v_t
 *
 * Multi-token queries (pkd_oracle_attention_multi): q and out are
 * [num_seqs][q_len][num_q_heads][head_dim]; the q_len new tokens are the
 * last q_len positions of each sequence (already in the cache), and query jq
 * attends to the tokens t < L_b - q_len + jq + 1, i.e. up to and including
 * its own position (causal among the new tokens).  A query with no visible
 * token gets out = 0.  Source: the review's section 7.4 names working
 * together with speculative decoding as a direction; verifying q_len draft
 * tokens in one pass is that case.  The causal rule is the plain reading.
 *
 * Sources:
 *  - Paged KV cache, logical page -> physical page table: CSDN answer
 *    "如何优化LLM推理引擎的内存访问延迟？", section 2 (paged cache and page
 *    table) and section 3 (PagedAttention: look up the page table, load the
 *    KV pages, blockwise attention).
 *  - The block loop over a block table bt[] for one head, Q resident, Q*K^T
 *    per K block, then logits*V per V block: review "Accelerating LLM
 *    Inference Throughput via Asynchronous KV Cache Prefetching", section 3.2
 *    (XFormers flow), section 3.4 (Algorithm 1, range [s, e) of block
 *    indices), section 4.1 (the same scheme for V blocks).
 *  - One (block, kv-head) tile is block_size x head_dim fp16 values: the
 *    M_block = b * d_h * T_block of the same review's section 4.2.
 *  - Scaled softmax, fp16 inputs and a split of the context into partitions
 *    with a merge step: the benchmark spec of this library; the pages print
 *    no softmax formula, so the textbook definition above is used.
 *
 * Readings where the pages are silent (each listed in the design notes):
 *  - GQA: query head h reads kv head h / (Hq/Hkv) (contiguous groups).
 *  - KV layout [num_blocks][num_kv_heads][block_size][head_dim], K and V
 *    separate arrays.  Q and out are [num_seqs][num_q_heads][head_dim].
 *  - context_len == 0 gives out = 0; a partition holding no token has
 *    m = -inf, l = 0, o = 0 and is skipped by the merge.
 *
 * Precision: inputs are IEEE binary16, decoded exactly to double; all
 * arithmetic is IEEE double in the order written above.
 *
 * Parity pins (tests, CPU only): numpy's float16 decoding of all 65536 bit
 * patterns; torch's scaled_dot_product_attention over contiguous K/V; block
 * permutation invariance; softmax weights summing to one; identical keys or
 * scale 0 giving the mean of V; context length 1 giving v_0; a one-token
 * spike per position; GQA equal to repeated-KV MHA; the log-sum-exp merge of
 * partitions equal to the unsplit result; partition sums at scale 0 equal to
 * the exact token counts; append-then-attend equal to SDPA over the grown
 * contiguous sequence; multi-token queries equal to SDPA with an explicit
 * causal mask, independent of tokens after each query's position, and equal
 * to single-query decode for the last query; and mutation tests that plant mistakes in this
 * file (compile-time PKD_ORACLE_MUTANT) and require some pin to fail.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifndef PKD_ORACLE_MUTANT
#define PKD_ORACLE_MUTANT 0
#endif

/* ---------------------------------------------------------------------- */
/* IEEE 754 binary16 -> double, from the format's definition:             */
/*   sign 1 bit, exponent 5 bits (bias 15), fraction 10 bits;             */
/*   e = 0: subnormal  (-1)^s * 2^-14 * (f / 1024)                        */
/*   e = 31: inf (f = 0) or NaN;  else (-1)^s * 2^(e-15) * (1 + f/1024)   */
/* ---------------------------------------------------------------------- */
double pkd_oracle_half_to_double(uint16_t bits)
{
    int sign = (bits >> 15) & 1;
    int e = (bits >> 10) & 0x1f;
    int f = bits & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -24);            /* 2^-14 * f / 2^10 */
    } else if (e == 31) {
        v = (f == 0) ? INFINITY : NAN;
    } else {
        v = ldexp(1024.0 + (double)f, e - 25); /* 2^(e-15) * (1024+f) / 2^10 */
    }
    return sign ? -v : v;
}

static double g_half_table[65536];
static pthread_once_t g_table_once = PTHREAD_ONCE_INIT;
static void build_half_table(void)
{
    for (uint32_t i = 0; i < 65536u; ++i) g_half_table[i] = pkd_oracle_half_to_double((uint16_t)i);
}
static inline double h2d(uint16_t b) { return g_half_table[b]; }

/* ---------------------------------------------------------------------- */
/* FP8 E4M3 (the OCP 8-bit float "E4M3", no infinities) -> double, from   */
/* the format's definition: sign 1 bit, exponent 4 bits (bias 7),         */
/* mantissa 3 bits;  e = 0: subnormal (-1)^s * 2^-6 * (m / 8);            */
/* e = 15 and m = 7: NaN;  else (-1)^s * 2^(e-7) * (1 + m/8).  Largest    */
/* finite magnitude 448.                                                   */
/* ---------------------------------------------------------------------- */
double pkd_oracle_e4m3_to_double(uint8_t bits)
{
    int sign = (bits >> 7) & 1;
    int e = (bits >> 3) & 0xf;
    int m = bits & 0x7;
    double v;
    if (e == 0) v = ldexp((double)m, -9);                 /* 2^-6 * m / 8 */
    else if (e == 15 && m == 7) v = NAN;
    else v = ldexp(8.0 + (double)m, e - 10);              /* 2^(e-7) * (8+m) / 8 */
    return sign ? -v : v;
}

static double g_e4m3_table[256];
static pthread_once_t g_e4m3_once = PTHREAD_ONCE_INIT;
static void build_e4m3_table(void)
{
    for (int i = 0; i < 256; ++i) g_e4m3_table[i] = pkd_oracle_e4m3_to_double((uint8_t)i);
}
static inline double e4m3d(uint8_t b) { return g_e4m3_table[b]; }

/*
 * float -> E4M3 by round-to-nearest-even onto the E4M3 grid, saturating to
 * the largest finite magnitude (448) instead of overflowing; NaN stays NaN
 * (0x7f).  Written from the grid: the representable magnitudes are
 * (8+m)/8 * 2^(e-7) for e = 1..15 (m = 0..6 at e = 15) and m/8 * 2^-6.
 */
uint8_t pkd_oracle_float_to_e4m3(float x)
{
    if (x != x) return 0x7f;
    uint8_t sign = (x < 0.0f || (x == 0.0f && 1.0f / x < 0.0f)) ? 0x80 : 0x00;
    double a = fabs((double)x);
    if (a >= 448.0) return sign | 0x7e;                   /* saturate */
    /* exponent of the binade holding a; below 2^-6 the spacing is 2^-9 */
    int e;
    double step;
    if (a < ldexp(1.0, -6)) {
        e = 0;
        step = ldexp(1.0, -9);
    } else {
        e = (int)floor(log2(a)) + 7;                      /* biased, 1..15 */
        if (ldexp(1.0, e - 7) > a) e -= 1;                /* guard log2 rounding */
        if (ldexp(1.0, e - 6) <= a) e += 1;
        step = ldexp(1.0, e - 10);                        /* 2^(e-7) / 8 */
    }
    double n = a / step;                                  /* exact: step is a power of two */
    double fl = floor(n);
    double r = n - fl;
    double k = fl;
    if (r > 0.5 || (r == 0.5 && fmod(fl, 2.0) != 0.0)) k = fl + 1.0;
    double v = k * step;                                  /* the rounded magnitude */
#if PKD_ORACLE_MUTANT == 11     /* planted mistake: truncation instead of rounding */
    v = fl * step;
#endif
    if (v >= 448.0) return sign | 0x7e;
    if (v == 0.0) return sign;
    /* re-encode v */
    if (v < ldexp(1.0, -6)) return sign | (uint8_t)(v / ldexp(1.0, -9));
    int ee = (int)floor(log2(v)) + 7;
    if (ldexp(1.0, ee - 7) > v) ee -= 1;
    if (ldexp(1.0, ee - 6) <= v) ee += 1;
    int mm = (int)(v / ldexp(1.0, ee - 10)) - 8;
    return sign | (uint8_t)((ee << 3) | mm);
}

/* Quantize n binary16 values: out[i] = e4m3(fp32(half(x[i])) / scale), the
 * division in IEEE fp32 (round to nearest) and the E4M3 rounding as above. */
void pkd_oracle_quantize_e4m3(const uint16_t *x, int n, float scale, uint8_t *out)
{
    pthread_once(&g_table_once, build_half_table);
    for (int i = 0; i < n; ++i) {
        float f = (float)h2d(x[i]);
        float qv = f / scale;
        out[i] = pkd_oracle_float_to_e4m3(qv);
    }
}

/* ---------------------------------------------------------------------- */
/* Problem description shared by the entry points below.                   */
/* ---------------------------------------------------------------------- */
typedef struct {
    const uint16_t *q;
    const void *k_cache, *v_cache;   /* binary16 words, or E4M3 bytes when kv_fp8 */
    const int32_t *block_tables, *context_lens;
    int num_seqs, num_q_heads, num_kv_heads, head_dim, block_size;
    int num_blocks, max_blocks_per_seq;
    double scale;
    int q_len;      /* query tokens per sequence (1: single-query decode) */
    int kv_fp8;     /* 1: caches hold E4M3 bytes; value = e4m3(byte) * k_scale (v_scale) */
    double k_scale, v_scale;
} problem_t;

/* Tokens that query jq of sequence b attends to: query jq sits at position
 * L_b - q_len + jq and sees every token up to and including itself (the
 * causal rule among the new tokens); with q_len = 1 this is L_b. */
static int visible(const problem_t *P, int b, int jq)
{
    int n = P->context_lens[b] - P->q_len + jq + 1;
#if PKD_ORACLE_MUTANT == 9      /* planted mistake: a query does not see its own token */
    if (P->q_len > 1) n -= 1;
#endif
    return n > 0 ? n : 0;
}

/* Address of the K (or V) row of logical token t of sequence b, kv head g.
 * Returns NULL when the block table entry is outside the pool. */
static const void *kv_row(const problem_t *P, const void *cache, int b, int g, int t)
{
    int logical_block = t / P->block_size;
    int slot = t % P->block_size;
#if PKD_ORACLE_MUTANT == 1      /* planted mistake: block and slot swapped */
    logical_block = t % P->block_size;
    slot = t / P->block_size;
    if (slot >= P->block_size) slot = P->block_size - 1;
    if (logical_block >= P->max_blocks_per_seq) logical_block = P->max_blocks_per_seq - 1;
#endif
    int p = P->block_tables[(size_t)b * P->max_blocks_per_seq + logical_block];
    if (p < 0 || p >= P->num_blocks) return NULL;
    size_t off = (((size_t)p * P->num_kv_heads + g) * P->block_size + slot) * P->head_dim;
    return (const char *)cache + off * (P->kv_fp8 ? 1 : 2);
}

static int kv_head_of(const problem_t *P, int h)
{
    int group = P->num_q_heads / P->num_kv_heads;
#if PKD_ORACLE_MUTANT == 2      /* planted mistake: interleaved instead of contiguous groups */
    return h % P->num_kv_heads;
#else
    return h / group;
#endif
}

/* Scores s_t for t in [t0, t1) of query jq, head h of sequence b.  Returns
 * -1 on a bad block id. */
static int scores(const problem_t *P, int b, int jq, int h, int t0, int t1, double *s)
{
    int g = kv_head_of(P, h);
    const uint16_t *qv = P->q + (((size_t)b * P->q_len + jq) * P->num_q_heads + h) * P->head_dim;
    for (int t = t0; t < t1; ++t) {
        const void *k = kv_row(P, P->k_cache, b, g, t);
        if (!k) return -1;
        double dot = 0.0;
        if (P->kv_fp8) {
            const uint8_t *k8 = (const uint8_t *)k;
            for (int d = 0; d < P->head_dim; ++d) dot += h2d(qv[d]) * (e4m3d(k8[d]) * P->k_scale);
        } else {
            const uint16_t *k16 = (const uint16_t *)k;
            for (int d = 0; d < P->head_dim; ++d) dot += h2d(qv[d]) * h2d(k16[d]);
        }
#if PKD_ORACLE_MUTANT == 3      /* planted mistake: scale dropped */
        s[t - t0] = dot;
#else
        s[t - t0] = P->scale * dot;
#endif
    }
    return 0;
}

/* Softmax weights of (b, jq, h) over its visible tokens into w.  -1 on bad ids. */
static int weights(const problem_t *P, int b, int jq, int h, double *w)
{
    int L = visible(P, b, jq);
#if PKD_ORACLE_MUTANT == 4      /* planted mistake: last token dropped */
    if (L > 0) L -= 1;
#endif
    if (L <= 0) return 0;
    if (scores(P, b, jq, h, 0, L, w)) return -1;
    double m = -INFINITY;
    for (int t = 0; t < L; ++t) if (w[t] > m) m = w[t];
    double z = 0.0;
    for (int t = 0; t < L; ++t) { w[t] = exp(w[t] - m); z += w[t]; }
#if PKD_ORACLE_MUTANT == 5      /* planted mistake: normalisation dropped */
    z = 1.0;
#endif
    for (int t = 0; t < L; ++t) w[t] /= z;
    return 0;
}

/* out[0..D) = sum_t w_t v_t for (b, jq, h).  w is scratch of L_b doubles. */
static int attend_row(const problem_t *P, int b, int jq, int h, double *w, double *out)
{
    int D = P->head_dim;
    int L = visible(P, b, jq);
#if PKD_ORACLE_MUTANT == 4
    if (L > 0) L -= 1;
#endif
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    if (L <= 0) return 0;
    if (weights(P, b, jq, h, w)) return -1;
    int g = kv_head_of(P, h);
    for (int t = 0; t < L; ++t) {
#if PKD_ORACLE_MUTANT == 6      /* planted mistake: values read from the K cache */
        const void *v = kv_row(P, P->k_cache, b, g, t);
#else
        const void *v = kv_row(P, P->v_cache, b, g, t);
#endif
        if (!v) return -1;
        if (P->kv_fp8) {
            const uint8_t *v8 = (const uint8_t *)v;
#if PKD_ORACLE_MUTANT == 10     /* planted mistake: the V scale is left out */
            for (int d = 0; d < D; ++d) out[d] += w[t] * e4m3d(v8[d]);
#else
            for (int d = 0; d < D; ++d) out[d] += w[t] * (e4m3d(v8[d]) * P->v_scale);
#endif
        } else {
            const uint16_t *v16 = (const uint16_t *)v;
            for (int d = 0; d < D; ++d) out[d] += w[t] * h2d(v16[d]);
        }
    }
    return 0;
}

/* ---------------------------------------------------------------------- */
/* Threaded driver over rows (b, h).                                       */
/* ---------------------------------------------------------------------- */
typedef struct {
    const problem_t *P;
    const int32_t *rows;   /* row ids (b*q_len + jq)*Hq + h, or NULL for all */
    int num_rows;
    double *out;           /* [num_rows][D] */
    int next;              /* work counter (guarded by mu) */
    int status;
    pthread_mutex_t mu;
} job_t;

static void *worker(void *arg)
{
    job_t *J = (job_t *)arg;
    const problem_t *P = J->P;
    int maxL = 0;
    for (int b = 0; b < P->num_seqs; ++b) if (P->context_lens[b] > maxL) maxL = P->context_lens[b];
    double *w = (double *)malloc(sizeof(double) * (size_t)(maxL > 0 ? maxL : 1));
    if (!w) { pthread_mutex_lock(&J->mu); J->status = -2; pthread_mutex_unlock(&J->mu); return NULL; }
    for (;;) {
        pthread_mutex_lock(&J->mu);
        int i = J->next++;
        pthread_mutex_unlock(&J->mu);
        if (i >= J->num_rows) break;
        int row = J->rows ? J->rows[i] : i;
        int h = row % P->num_q_heads;
        int bj = row / P->num_q_heads;
        int b = bj / P->q_len, jq = bj % P->q_len;
        if (attend_row(P, b, jq, h, w, J->out + (size_t)i * P->head_dim)) {
            pthread_mutex_lock(&J->mu); J->status = -1; pthread_mutex_unlock(&J->mu);
        }
    }
    free(w);
    return NULL;
}

static int check_problem(const problem_t *P)
{
    if (!P->q || !P->k_cache || !P->v_cache || !P->block_tables || !P->context_lens) return -3;
    if (P->num_seqs < 0 || P->num_q_heads <= 0 || P->num_kv_heads <= 0 || P->head_dim <= 0 ||
        P->block_size <= 0 || P->max_blocks_per_seq <= 0 || P->num_blocks <= 0) return -3;
    if (P->num_q_heads % P->num_kv_heads) return -3;
    if (P->q_len < 1) return -3;
    for (int b = 0; b < P->num_seqs; ++b) {
        int L = P->context_lens[b];
        if (L < 0 || L > P->max_blocks_per_seq * P->block_size) return -3;
    }
    return 0;
}

/*
 * Exact attention for the listed rows (row = b * num_q_heads + h), or for
 * every row when rows == NULL (then out is [num_seqs][num_q_heads][head_dim]).
 * Returns 0; -1 if a used block-table entry is outside [0, num_blocks);
 * -2 on allocation failure; -3 on a bad argument.
 */
static int attention_impl(problem_t P, const int32_t *rows, int num_rows, double *out, int num_threads);

int pkd_oracle_attention_multi(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                               const int32_t *block_tables, const int32_t *context_lens,
                               int num_seqs, int q_len, int num_q_heads, int num_kv_heads,
                               int head_dim, int block_size, int num_blocks, int max_blocks_per_seq,
                               double scale, const int32_t *rows, int num_rows, double *out,
                               int num_threads)
{
    problem_t P = {q, k_cache, v_cache, block_tables, context_lens, num_seqs, num_q_heads,
                   num_kv_heads, head_dim, block_size, num_blocks, max_blocks_per_seq, scale, q_len, 0, 1.0, 1.0};
    return attention_impl(P, rows, num_rows, out, num_threads);
}

/*
 * FP8 KV: the caches hold E4M3 bytes in the same [num_blocks][num_kv_heads]
 * [block_size][head_dim] layout; element value = e4m3(byte) * k_scale for K,
 * * v_scale for V (one scale per cache).  q, out and the rest as in
 * pkd_oracle_attention_multi.  Source: CSDN answer "如何优化LLM推理引擎的内存
 * 访问延迟？", section 4 (FP8 precision to shrink the KV footprint); the
 * format and the per-cache scale are this library's plainest reading.
 */
int pkd_oracle_attention_fp8(const uint16_t *q, const uint8_t *k_cache, const uint8_t *v_cache,
                             const int32_t *block_tables, const int32_t *context_lens,
                             int num_seqs, int q_len, int num_q_heads, int num_kv_heads,
                             int head_dim, int block_size, int num_blocks, int max_blocks_per_seq,
                             double scale, double k_scale, double v_scale, const int32_t *rows,
                             int num_rows, double *out, int num_threads)
{
    problem_t P = {q, k_cache, v_cache, block_tables, context_lens, num_seqs, num_q_heads,
                   num_kv_heads, head_dim, block_size, num_blocks, max_blocks_per_seq, scale, q_len, 1,
                   k_scale, v_scale};
    return attention_impl(P, rows, num_rows, out, num_threads);
}

static int attention_impl(problem_t P, const int32_t *rows, int num_rows, double *out, int num_threads)
{
    pthread_once(&g_table_once, build_half_table);
    pthread_once(&g_e4m3_once, build_e4m3_table);
    const int num_seqs = P.num_seqs, q_len = P.q_len, num_q_heads = P.num_q_heads;
    int rc = check_problem(&P);
    if (rc) return rc;
    job_t J;
    const int total = num_seqs * q_len * num_q_heads;
    J.P = &P; J.rows = rows; J.out = out; J.next = 0; J.status = 0;
    J.num_rows = rows ? num_rows : total;
    if (rows) {
        for (int i = 0; i < num_rows; ++i)
            if (rows[i] < 0 || rows[i] >= total) return -3;
    }
    pthread_mutex_init(&J.mu, NULL);
    if (num_threads < 1) num_threads = 1;
    if (num_threads > 1024) num_threads = 1024;
    pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)num_threads);
    if (!tid) { pthread_mutex_destroy(&J.mu); return -2; }
    int started = 0;
    for (int i = 0; i < num_threads; ++i) {
        if (pthread_create(&tid[i], NULL, worker, &J) == 0) ++started;
        else break;
    }
    if (started == 0) worker(&J);
    for (int i = 0; i < started; ++i) pthread_join(tid[i], NULL);
    free(tid);
    pthread_mutex_destroy(&J.mu);
    return J.status;
}

/* Single-query decode (q_len = 1): rows b * num_q_heads + h. */
int pkd_oracle_attention(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                         const int32_t *block_tables, const int32_t *context_lens,
                         int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                         int block_size, int num_blocks, int max_blocks_per_seq, double scale,
                         const int32_t *rows, int num_rows, double *out, int num_threads)
{
    return pkd_oracle_attention_multi(q, k_cache, v_cache, block_tables, context_lens, num_seqs, 1,
                                      num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                                      max_blocks_per_seq, scale, rows, num_rows, out, num_threads);
}

/* Softmax weights w[0..L_b) of one row (b, h).  Same return codes. */
int pkd_oracle_weights(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                       const int32_t *block_tables, const int32_t *context_lens,
                       int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                       int block_size, int num_blocks, int max_blocks_per_seq, double scale,
                       int b, int h, double *w)
{
    pthread_once(&g_table_once, build_half_table);
    problem_t P = {q, k_cache, v_cache, block_tables, context_lens, num_seqs, num_q_heads,
                   num_kv_heads, head_dim, block_size, num_blocks, max_blocks_per_seq, scale, 1, 0, 1.0, 1.0};
    int rc = check_problem(&P);
    if (rc) return rc;
    if (b < 0 || b >= num_seqs || h < 0 || h >= num_q_heads) return -3;
    return weights(&P, b, 0, h, w);
}

/*
 * Per-partition statistics for a split of each context into partitions of
 * partition_size tokens: partition j of sequence b covers logical tokens
 * [j*P, min((j+1)*P, L_b)).  For each (b, h, j):
 *   m = max_t s_t,  l = sum_t exp(s_t - m),  o[:] = sum_t exp(s_t - m) v_t
 * (o unnormalised).  Partitions with no token: m = -inf, l = 0, o = 0.
 * Layouts: m, l [num_seqs][num_q_heads][max_partitions];
 *          o    [num_seqs][num_q_heads][max_partitions][head_dim].
 */
int pkd_oracle_partitions(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                          const int32_t *block_tables, const int32_t *context_lens,
                          int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                          int block_size, int num_blocks, int max_blocks_per_seq, double scale,
                          int partition_size, int max_partitions,
                          double *m_out, double *l_out, double *o_out)
{
    pthread_once(&g_table_once, build_half_table);
    problem_t P = {q, k_cache, v_cache, block_tables, context_lens, num_seqs, num_q_heads,
                   num_kv_heads, head_dim, block_size, num_blocks, max_blocks_per_seq, scale, 1, 0, 1.0, 1.0};
    int rc = check_problem(&P);
    if (rc) return rc;
    if (partition_size <= 0 || max_partitions <= 0) return -3;
    int D = head_dim;
    double *s = (double *)malloc(sizeof(double) * (size_t)partition_size);
    if (!s) return -2;
    for (int b = 0; b < num_seqs; ++b) {
        int L = context_lens[b];
        if ((L + partition_size - 1) / partition_size > max_partitions) { free(s); return -3; }
        for (int h = 0; h < num_q_heads; ++h) {
            int g = kv_head_of(&P, h);
            for (int j = 0; j < max_partitions; ++j) {
                size_t idx = ((size_t)b * num_q_heads + h) * max_partitions + j;
                double *o = o_out + idx * D;
                for (int d = 0; d < D; ++d) o[d] = 0.0;
                int t0 = j * partition_size;
                int t1 = t0 + partition_size;
#if PKD_ORACLE_MUTANT == 7      /* planted mistake: partitions overlap by one token */
                t1 += 1;
#endif
                if (t1 > L) t1 = L;
                if (t0 >= t1) { m_out[idx] = -INFINITY; l_out[idx] = 0.0; continue; }
                if (scores(&P, b, 0, h, t0, t1, s)) { free(s); return -1; }
                double m = -INFINITY;
                for (int t = t0; t < t1; ++t) if (s[t - t0] > m) m = s[t - t0];
                double l = 0.0;
                for (int t = t0; t < t1; ++t) {
                    double e = exp(s[t - t0] - m);
                    l += e;
                    const uint16_t *v = (const uint16_t *)kv_row(&P, v_cache, b, g, t);
                    if (!v) { free(s); return -1; }
                    for (int d = 0; d < D; ++d) o[d] += e * h2d(v[d]);
                }
                m_out[idx] = m;
                l_out[idx] = l;
            }
        }
    }
    free(s);
    return 0;
}

/*
 * Merge of partition statistics (log-sum-exp identity):
 *   M = max_j m_j,  out = sum_j exp(m_j - M) o_j / sum_j exp(m_j - M) l_j,
 * over the partitions that hold a token (j < ceil(L_b / P)); out = 0 when
 * L_b = 0.  Layouts as in pkd_oracle_partitions; out [num_seqs][num_q_heads][D].
 */
int pkd_oracle_merge(const double *m_in, const double *l_in, const double *o_in,
                     const int32_t *context_lens, int num_seqs, int num_q_heads, int head_dim,
                     int partition_size, int max_partitions, double *out)
{
    if (!m_in || !l_in || !o_in || !context_lens || !out) return -3;
    if (partition_size <= 0 || max_partitions <= 0 || head_dim <= 0) return -3;
    int D = head_dim;
    for (int b = 0; b < num_seqs; ++b) {
        int L = context_lens[b];
        int np = (L + partition_size - 1) / partition_size;
        if (np > max_partitions) return -3;
        for (int h = 0; h < num_q_heads; ++h) {
            size_t base = ((size_t)b * num_q_heads + h) * max_partitions;
            double *y = out + ((size_t)b * num_q_heads + h) * D;
            for (int d = 0; d < D; ++d) y[d] = 0.0;
            if (np == 0) continue;
            double M = -INFINITY;
            for (int j = 0; j < np; ++j) if (m_in[base + j] > M) M = m_in[base + j];
            double z = 0.0;
            for (int j = 0; j < np; ++j) {
                double c = exp(m_in[base + j] - M);
                z += c * l_in[base + j];
                for (int d = 0; d < D; ++d) y[d] += c * o_in[(base + j) * D + d];
            }
            for (int d = 0; d < D; ++d) y[d] /= z;
        }
    }
    return 0;
}

/*
 * Append of one new token per sequence into the paged cache (the cache write
 * that precedes each decode step): with L = context_lens[b] (the length
 * before the append), for every kv head g
 *   p = block_tables[b][L / bs],  K[p][g][L % bs][:] = k_new[b][g][:],
 *                                 V[p][g][L % bs][:] = v_new[b][g][:].
 * Operates on the caller's arrays in place (raw binary16 words).  Returns 0;
 * -1 if a sequence has no room in its table row or its block id is outside
 * [0, num_blocks) (that sequence is skipped); -3 on a bad argument.
 * Source: CSDN answer "如何优化LLM推理引擎的内存访问延迟？", section 2 (each
 * sequence's KV lives in pages listed by its page table; new tokens go into
 * the sequence's pages in logical order).
 */
int pkd_oracle_append(const uint16_t *k_new, const uint16_t *v_new, const int32_t *block_tables,
                      const int32_t *context_lens, uint16_t *k_cache, uint16_t *v_cache, int num_seqs,
                      int num_kv_heads, int head_dim, int block_size, int num_blocks,
                      int max_blocks_per_seq)
{
    if (!k_new || !v_new || !block_tables || !context_lens || !k_cache || !v_cache) return -3;
    if (num_seqs < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks <= 0 ||
        max_blocks_per_seq <= 0)
        return -3;
    int status = 0;
    for (int b = 0; b < num_seqs; ++b) {
        int L = context_lens[b];
        int logical_block = L / block_size;
        int slot = L % block_size;
#if PKD_ORACLE_MUTANT == 8      /* planted mistake: writes the last existing slot instead of the next */
        if (L > 0) { logical_block = (L - 1) / block_size; slot = (L - 1) % block_size; }
#endif
        if (L < 0 || logical_block >= max_blocks_per_seq) { status = -1; continue; }
        int p = block_tables[(size_t)b * max_blocks_per_seq + logical_block];
        if (p < 0 || p >= num_blocks) { status = -1; continue; }
        for (int g = 0; g < num_kv_heads; ++g) {
            size_t dst = (((size_t)p * num_kv_heads + g) * block_size + slot) * head_dim;
            size_t src = ((size_t)b * num_kv_heads + g) * head_dim;
            for (int d = 0; d < head_dim; ++d) {
                k_cache[dst + d] = k_new[src + d];
                v_cache[dst + d] = v_new[src + d];
            }
        }
    }
    return status;
}

/* The cache write with FP8 caches: as pkd_oracle_append, each element of the
 * new rows stored as pkd_oracle_quantize_e4m3 gives it (k_scale for K,
 * v_scale for V).  Same return codes. */
int pkd_oracle_append_fp8(const uint16_t *k_new, const uint16_t *v_new, const int32_t *block_tables,
                          const int32_t *context_lens, uint8_t *k_cache, uint8_t *v_cache, int num_seqs,
                          int num_kv_heads, int head_dim, int block_size, int num_blocks,
                          int max_blocks_per_seq, float k_scale, float v_scale)
{
    if (!k_new || !v_new || !block_tables || !context_lens || !k_cache || !v_cache) return -3;
    if (num_seqs < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks <= 0 ||
        max_blocks_per_seq <= 0 || !(k_scale > 0.0f) || !(v_scale > 0.0f))
        return -3;
    int status = 0;
    for (int b = 0; b < num_seqs; ++b) {
        int L = context_lens[b];
        int logical_block = L / block_size;
        int slot = L % block_size;
        if (L < 0 || logical_block >= max_blocks_per_seq) { status = -1; continue; }
        int p = block_tables[(size_t)b * max_blocks_per_seq + logical_block];
        if (p < 0 || p >= num_blocks) { status = -1; continue; }
        for (int g = 0; g < num_kv_heads; ++g) {
            size_t dst = (((size_t)p * num_kv_heads + g) * block_size + slot) * head_dim;
            size_t src = ((size_t)b * num_kv_heads + g) * head_dim;
            pkd_oracle_quantize_e4m3(k_new + src, head_dim, k_scale, k_cache + dst);
            pkd_oracle_quantize_e4m3(v_new + src, head_dim, v_scale, v_cache + dst);
        }
    }
    return status;
}

/* Which planted mistake (0 = none) this build carries; for the mutation tests. */
int pkd_oracle_mutant(void) { return PKD_ORACLE_MUTANT; }
