/*
 * Float64 CPU oracle for generalized paged attention.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the checker, not the product: only the tests, the
 * smoke check and the benchmark's CPU-baseline leg load it.  It shares no code with the CUDA
 * library and is written to be read against the pages, not to be fast.
 *
 * What it computes (one output row = one (sequence i, new token j, query head h)):
 *
 *   Attention(Q,K,V) = softmax(Q K^T / sqrt(d_k)) V
 *     -- "SOSP 2023論文解説: PagedAttention", section "PagedAttentionアルゴリズム", first equation.
 *     The scale 1/sqrt(d_k) is passed in by the caller as `scale`.
 *
 *   Blockwise form: with N = ceil(n / B) logical blocks,
 *     A_j = exp(q K_j^T / sqrt(d_k)) / sum_{i=1..N} sum_{k=1..B} exp(q k_{i,k}^T / sqrt(d_k)),
 *     o   = sum_j A_j V_j
 *     -- same page and section, second equation.  The oracle walks the logical blocks in order,
 *     finds each one's physical block through the sequence's block table ("ブロックテーブルによる
 *     メモリ管理"), and reads the B keys inside it.
 *
 *   Generalization to several new tokens per sequence with a causal mask over cached-plus-new
 *   positions -- "Stateful Large Language Model Serving with Pensieve", section
 *   "汎化PagedAttentionカーネル".  Reading taken here: the sequence has c = ctx_len tokens cached
 *   before this step and q = q_len new tokens whose K/V already sit in the cache at positions
 *   c .. c+q-1; new token j sits at absolute position P = c + j and sees keys 0 .. P (itself
 *   included).
 *
 *   GQA -- "KVキャッシュ管理の教科書", 第19章: groups of query heads share one K/V head.  Reading
 *   taken here: contiguous groups, query head h uses K/V head h / (Hq / Hkv).
 *
 * The softmax is evaluated with the usual max subtraction (exp(s - max) / sum exp(s - max)),
 * which is the same function, in float64 with C's exp().
 *
 *   8-bit caches -- "KVキャッシュ管理の教科書" 第3章 (fewer bits per element as the third way to
 *   shrink the cache) and 第22章 (quantising KV before decoding).  Reading taken here: K and V
 *   hold FP8 E4M3 codes and one scale each; a cached element's value is code value x scale, and
 *   attention is the same function of those values.
 *
 *   float64 caches hold values that are not float32 numbers (the dequantised 2-bit pages of the
 *   Kitty row, "KVキャッシュ管理の教科書" 第22章); attention is again the same function.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_F32 = 0, ORACLE_BF16 = 1, ORACLE_F16 = 2, ORACLE_E4M3 = 3, ORACLE_F64 = 4 };

/* IEEE-754 binary16 -> double, from the format's definition (1 sign, 5 exponent, 10 fraction
 * bits, bias 15); every binary16 value is exactly representable in double. */
static double half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);                    /* subnormal: m * 2^(1-15-10) */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(m + 1024), e - 25);        /* (1 + m/1024) * 2^(e-15) */
    return sign ? -v : v;
}

/* bfloat16 is the top half of an IEEE binary32; widen and convert exactly. */
static double bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* FP8 E4M3 -> double, from the format's definition: 1 sign, 4 exponent bits (bias 7), 3 fraction
 * bits, subnormals at exponent 0, no infinities, S.1111.111 is NaN. */
static double e4m3_to_double(uint8_t c)
{
    int sign = (c >> 7) & 1;
    int e = (c >> 3) & 0xf;
    int m = c & 7;
    double v;
    if (e == 15 && m == 7)
        v = NAN;
    else if (e == 0)
        v = ldexp((double)m, -9);                     /* subnormal: m/8 * 2^(1-7) */
    else
        v = ldexp((double)(m + 8), e - 10);           /* (1 + m/8) * 2^(e-7) */
    return sign ? -v : v;
}

static double element(const void *base, int dtype, int64_t idx)
{
    switch (dtype) {
    case ORACLE_F32: return (double)((const float *)base)[idx];
    case ORACLE_BF16: return bf16_to_double(((const uint16_t *)base)[idx]);
    case ORACLE_E4M3: return e4m3_to_double(((const uint8_t *)base)[idx]);
    case ORACLE_F64: return ((const double *)base)[idx];
    default: return half_to_double(((const uint16_t *)base)[idx]);
    }
}

/*
 * Computes the requested output rows.
 *   q        [total_q, Hq, d]            (q_dtype)
 *   k_cache  physical block b, head kh, slot s, dim x at  b*block_stride + (kh*B + s)*d + x
 *            (kv_dtype; an element's value is multiplied by k_scale)
 *   v_cache  same layout (value multiplied by v_scale)
 *   rows     n_rows triples (seq, token j within the sequence's new tokens, query head), or NULL
 *            for every row in order (packed token t, head h)
 *   out      n_rows * d doubles
 * Returns 0, or -1 if a row index is out of range, -2 if a block-table entry that must be read
 * is outside [0, num_blocks).
 */
int oracle_paged_attention_kv(const void *q, const void *k_cache, const void *v_cache,
                              int q_dtype, int kv_dtype, double k_scale, double v_scale,
                              const int32_t *block_tables, const int32_t *ctx_lens,
                              const int32_t *q_lens, int32_t num_seqs, int32_t num_q_heads,
                              int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                              int64_t num_blocks, int32_t max_blocks_per_seq, int64_t block_stride,
                              double scale, const int64_t *rows, int64_t n_rows, double *out,
                              int num_threads)
{
    const int64_t d = head_dim, B = block_size;
    const int64_t group = num_q_heads / num_kv_heads;
    int64_t *cu = (int64_t *)malloc(sizeof(int64_t) * ((size_t)num_seqs + 1));
    if (!cu) return -3;
    cu[0] = 0;
    for (int32_t i = 0; i < num_seqs; ++i) cu[i + 1] = cu[i] + q_lens[i];
    const int64_t total_rows = rows ? n_rows : cu[num_seqs] * num_q_heads;
    int status = 0;

#ifdef _OPENMP
    if (num_threads > 0) omp_set_num_threads(num_threads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t r = 0; r < total_rows; ++r) {
        int64_t i, j, h;
        if (rows) {
            i = rows[3 * r]; j = rows[3 * r + 1]; h = rows[3 * r + 2];
        } else {
            int64_t t = r / num_q_heads;
            h = r % num_q_heads;
            i = 0;
            while (cu[i + 1] <= t) ++i;
            j = t - cu[i];
        }
        double *o = out + r * d;
        if (i < 0 || i >= num_seqs || j < 0 || j >= q_lens[i] || h < 0 || h >= num_q_heads) {
            for (int64_t x = 0; x < d; ++x) o[x] = NAN;
#ifdef _OPENMP
#pragma omp atomic write
#endif
            status = -1;
            continue;
        }
        const int64_t kh = h / group;                  /* GQA: contiguous groups */
        const int64_t P = (int64_t)ctx_lens[i] + j;    /* absolute position of this query */
        const int64_t n = P + 1;                       /* keys it sees: 0 .. P */
        const int64_t N = (n + B - 1) / B;             /* logical blocks touched */
        const int64_t qrow = (cu[i] + j) * num_q_heads + h;
        double *s = (double *)malloc(sizeof(double) * (size_t)n);
        if (!s) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            status = -3;
            continue;
        }

        /* scores, block by block through the block table */
        int bad = 0;
        for (int64_t jb = 0; jb < N && !bad; ++jb) {
            int64_t phys = block_tables[i * (int64_t)max_blocks_per_seq + jb];
            if (phys < 0 || phys >= num_blocks) { bad = 1; break; }
            for (int64_t k = 0; k < B; ++k) {
                int64_t p = jb * B + k;
                if (p >= n) break;                     /* causal: positions after P unseen */
                int64_t kbase = phys * block_stride + (kh * B + k) * d;
                double dot = 0.0;
                for (int64_t x = 0; x < d; ++x)
                    dot += element(q, q_dtype, qrow * d + x) *
                           (element(k_cache, kv_dtype, kbase + x) * k_scale);
                s[p] = scale * dot;
            }
        }
        if (bad) {
            for (int64_t x = 0; x < d; ++x) o[x] = NAN;
#ifdef _OPENMP
#pragma omp atomic write
#endif
            status = -2;
            free(s);
            continue;
        }
        /* softmax over the visible keys */
        double mx = -INFINITY;
        for (int64_t p = 0; p < n; ++p) if (s[p] > mx) mx = s[p];
        double denom = 0.0;
        for (int64_t p = 0; p < n; ++p) { s[p] = exp(s[p] - mx); denom += s[p]; }
        /* o = sum_p w_p V_p, walking the blocks again */
        for (int64_t x = 0; x < d; ++x) o[x] = 0.0;
        for (int64_t jb = 0; jb < N; ++jb) {
            int64_t phys = block_tables[i * (int64_t)max_blocks_per_seq + jb];
            for (int64_t k = 0; k < B; ++k) {
                int64_t p = jb * B + k;
                if (p >= n) break;
                int64_t vbase = phys * block_stride + (kh * B + k) * d;
                double w = s[p] / denom;
                for (int64_t x = 0; x < d; ++x)
                    o[x] += w * (element(v_cache, kv_dtype, vbase + x) * v_scale);
            }
        }
        free(s);
    }
    free(cu);
    return status;
}

/* The same with q and caches in one dtype and unit scales. */
int oracle_paged_attention(const void *q, const void *k_cache, const void *v_cache, int dtype,
                           const int32_t *block_tables, const int32_t *ctx_lens,
                           const int32_t *q_lens, int32_t num_seqs, int32_t num_q_heads,
                           int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                           int64_t num_blocks, int32_t max_blocks_per_seq, int64_t block_stride,
                           double scale, const int64_t *rows, int64_t n_rows, double *out,
                           int num_threads)
{
    return oracle_paged_attention_kv(q, k_cache, v_cache, dtype, dtype, 1.0, 1.0, block_tables,
                                     ctx_lens, q_lens, num_seqs, num_q_heads, num_kv_heads, head_dim,
                                     block_size, num_blocks, max_blocks_per_seq, block_stride, scale,
                                     rows, n_rows, out, num_threads);
}

/* Number of OpenMP threads the oracle would use (1 when built without OpenMP). */
int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
