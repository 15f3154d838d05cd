/*
 * gqa_oracle.c -- TEST INFRASTRUCTURE, not product code.
 *
 * A plain, slow, fp64 CPU restatement of grouped-query decode attention and
 * of its sparse, paged, FP8-KV, sigmoid-gated variant.  It exists only to
 * check the CUDA path: the test suite, the package smoke check and the
 * benchmark's CPU-baseline leg are the only callers.  It shares no code with
 * the CUDA library and includes none of its headers.
 *
 * Sources (web pages on grouped-query decode attention):
 *  - "When the K/V copy costs more than the attention" (kv-copies-gqa),
 *    section "What I was looking at": query head h reads KV head
 *    h // (H_q // H_kv) in place; section "Why it closed, and the tests that
 *    merged", head-map table: the two wrong maps (h // H_kv) % H_kv and
 *    h % H_kv that a test must tell apart from the right one.
 *  - "Sparse paged GQA decode attention with FP8 KV cache on SM89",
 *    sections "Workload" and "Implementations": page size 16, a page table
 *    per request, top-K selected tokens, FP8 E4M3FN K/V with per-tensor
 *    k_scale / v_scale (k_scale goes into the score, v_scale onto the
 *    output), scaled dot-product attention over the selected tokens, then a
 *    sigmoid gate on the output.
 *  - The same page-table addressing without a top-K list (every token of the
 *    request, up to its own sequence length) is the serving layout the
 *    kv-copies page's "Open questions" and the FP8 page's "Workload" point
 *    to; its masking follows the dense rule below, per request.
 *  - "Profiling down to the register, then an extension that broke my
 *    assumptions twice", paragraph "int8 KV-cache" and section "What's still
 *    open": an int8 KV cache dequantised tile by tile inside the attention
 *    kernel.  The format is not printed; the reading taken here is the
 *    symmetric per-tensor one (value = int8 code * scale).
 *  - The masking rule for S_q > 1 is not printed on the pages; the reading
 *    taken here is bottom-right alignment: query row i of S_q sees keys
 *    j <= S_kv - S_q + i.
 *
 * Everything is computed in double precision from the exact input values.
 * bf16 inputs arrive as their 16-bit patterns and are widened exactly; FP8
 * inputs arrive as their byte codes and are decoded from the format's
 * definition (OCP 8-bit floating point, E4M3FN: bias 7, no infinities, NaN
 * at S.1111.111).  The only parallelism is an OpenMP loop over independent
 * output rows; there is no blocking, fusion or reordering inside a row.
 *
 * Mutation self-check: building with -DORACLE_PLANT_BUG=n plants one known
 * mistake (see the PLANT() sites below); the test suite builds each variant
 * and asserts that at least one pin fails on it.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#ifndef ORACLE_PLANT_BUG
#define ORACLE_PLANT_BUG 0
#endif
#define PLANT(n) (ORACLE_PLANT_BUG == (n))

/* ------------------------------------------------------------------ */
/* number formats                                                       */
/* ------------------------------------------------------------------ */

/* bf16 is the upper half of an IEEE binary32; widening is exact. */
static double bf16_value(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* OCP E4M3FN: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits.
 * Exponent field 0 is subnormal (2^-6 * m/8); all-ones exponent with all-ones
 * mantissa is NaN; there is no infinity. */
double oracle_e4m3fn_value(uint8_t code)
{
    int sign = (code >> 7) & 1;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double mag;
    if (e == 0xF && m == 0x7)
        return NAN;
    int bias = PLANT(8) ? 8 : 7;
    if (e == 0)
        mag = ldexp((double)m / 8.0, 1 - bias);
    else
        mag = ldexp(1.0 + (double)m / 8.0, e - bias);
    return sign ? -mag : mag;
}

/* ------------------------------------------------------------------ */
/* head mapping                                                         */
/* ------------------------------------------------------------------ */

/* Query head h reads KV head h // (Hq / Hkv). */
int oracle_kv_head(int h, int Hq, int Hkv)
{
    if (PLANT(1))
        return (h / Hkv) % Hkv;
    if (PLANT(2))
        return h % Hkv;
    return h / (Hq / Hkv);
}

/* Last visible key of query row i (bottom-right aligned causal mask). */
static long last_visible_key(int i, int Sq, int Skv)
{
    if (PLANT(3))
        return (long)Skv - Sq + i - 1;
    if (PLANT(10))
        return (long)i;
    return (long)Skv - Sq + i;
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Sets the number of threads later calls use (timing only; results do not
 * depend on it: rows are independent and each is computed by one thread). */
void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* ------------------------------------------------------------------ */
/* dense grouped-query decode attention                                 */
/* ------------------------------------------------------------------ */

/*
 * q   : bf16 [B, Sq, Hq, D]       k, v : bf16 [B, Skv, Hkv, D]
 * rows: optional list of n_rows flattened row ids r = (b*Hq + h)*Sq + i;
 *       NULL means every row, in that order (n_rows ignored).
 * out : [n_rows, D] double        lse  : [n_rows] double (natural log)
 *
 * For each row: s_j = scale * q.k_j over visible keys j,
 *   LSE = m + ln sum_j exp(s_j - m)   (m = max_j s_j),
 *   O   = sum_j exp(s_j - LSE) v_j.
 */
void oracle_gqa_decode(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                       int B, int Sq, int Skv, int Hq, int Hkv, int D, double scale,
                       const int32_t *rows, int n_rows, double *out, double *lse)
{
    long total = rows ? n_rows : (long)B * Hq * Sq;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(Skv > 0 ? Skv : 1));
#pragma omp for schedule(dynamic, 1)
        for (long n = 0; n < total; ++n) {
            long r = rows ? rows[n] : n;
            int i = (int)(r % Sq);
            int h = (int)((r / Sq) % Hq);
            int b = (int)(r / ((long)Sq * Hq));
            int g = oracle_kv_head(h, Hq, Hkv);
            long last = last_visible_key(i, Sq, Skv);
            const uint16_t *qrow = q + (((size_t)b * Sq + i) * Hq + h) * D;
            double m = -INFINITY;
            for (long j = 0; j <= last && j < Skv; ++j) {
                const uint16_t *krow = k + (((size_t)b * Skv + j) * Hkv + g) * D;
                double dot = 0.0;
                for (int d = 0; d < D; ++d)
                    dot += bf16_value(qrow[d]) * bf16_value(krow[d]);
                s[j] = PLANT(5) ? dot : scale * dot;
                if (s[j] > m)
                    m = s[j];
            }
            double sum = 0.0;
            for (long j = 0; j <= last && j < Skv; ++j)
                sum += exp(s[j] - m);
            double L = PLANT(4) ? m : m + log(sum);
            double *o = out + (size_t)n * D;
            for (int d = 0; d < D; ++d)
                o[d] = 0.0;
            for (long j = 0; j <= last && j < Skv; ++j) {
                double w = exp(s[j] - L);
                const uint16_t *vrow = v + (((size_t)b * Skv + j) * Hkv + g) * D;
                for (int d = 0; d < D; ++d)
                    o[d] += w * bf16_value(vrow[d]);
            }
            if (lse)
                lse[n] = L;
        }
        free(s);
    }
}

/*
 * Dense decode with different head sizes for the scores and the values
 * ("When the K/V copy costs more than the attention", section "Limits, and
 * what I'd do next": the d192x128 flavour): q, k : bf16 [.., Dqk],
 * v : bf16 [B, Skv, Hkv, Dv], out : [n_rows, Dv].  Otherwise exactly
 * oracle_gqa_decode (same rows, mask, scale, LSE).
 */
void oracle_gqa_decode_dv(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                          int B, int Sq, int Skv, int Hq, int Hkv, int Dqk, int Dv, double scale,
                          const int32_t *rows, int n_rows, double *out, double *lse)
{
    long total = rows ? n_rows : (long)B * Hq * Sq;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(Skv > 0 ? Skv : 1));
#pragma omp for schedule(dynamic, 1)
        for (long n = 0; n < total; ++n) {
            long r = rows ? rows[n] : n;
            int i = (int)(r % Sq);
            int h = (int)((r / Sq) % Hq);
            int b = (int)(r / ((long)Sq * Hq));
            int g = oracle_kv_head(h, Hq, Hkv);
            long last = last_visible_key(i, Sq, Skv);
            const uint16_t *qrow = q + (((size_t)b * Sq + i) * Hq + h) * Dqk;
            int dot_len = PLANT(14) ? Dv : Dqk;
            double m = -INFINITY;
            for (long j = 0; j <= last && j < Skv; ++j) {
                const uint16_t *krow = k + (((size_t)b * Skv + j) * Hkv + g) * Dqk;
                double dot = 0.0;
                for (int d = 0; d < dot_len; ++d)
                    dot += bf16_value(qrow[d]) * bf16_value(krow[d]);
                s[j] = scale * dot;
                if (s[j] > m)
                    m = s[j];
            }
            double sum = 0.0;
            for (long j = 0; j <= last && j < Skv; ++j)
                sum += exp(s[j] - m);
            double L = m + log(sum);
            double *o = out + (size_t)n * Dv;
            for (int d = 0; d < Dv; ++d)
                o[d] = 0.0;
            for (long j = 0; j <= last && j < Skv; ++j) {
                double w = exp(s[j] - L);
                const uint16_t *vrow = v + (((size_t)b * Skv + j) * Hkv + g) * Dv;
                for (int d = 0; d < Dv; ++d)
                    o[d] += w * bf16_value(vrow[d]);
            }
            if (lse)
                lse[n] = L;
        }
        free(s);
    }
}

/* ------------------------------------------------------------------ */
/* sparse paged FP8 decode with sigmoid gate                            */
/* ------------------------------------------------------------------ */

/* Byte offset of (page p, slot r, KV head g, dim 0) in a pool laid out
 * [num_pages, page_size, Hkv, D]. */
static size_t pool_row(long p, long r, int g, int ps, int Hkv, int D)
{
    return (((size_t)p * ps + r) * Hkv + g) * D;
}

/* Logical token t of request b lives in page page_table[b][t / ps], slot
 * t % ps.  Returns the physical page, or -1 for a padding index (t < 0). */
static long token_page(const int32_t *page_table, int b, int ppr, long t, int ps, long *slot)
{
    if (t < 0)
        return -1;
    long lp = PLANT(6) ? t % ps : t / ps;
    *slot = PLANT(6) ? t / ps : t % ps;
    return page_table[(size_t)b * ppr + lp];
}

/*
 * Byte-exact gather of the selected rows: out[b, k, g, :] = pool row of token
 * topk[b][k] for KV head g.  Padding indices (negative) give zero bytes.
 * out : uint8 [B, topk, Hkv, D]
 */
void oracle_paged_gather(const uint8_t *pool, const int32_t *page_table, const int32_t *topk,
                         int B, int Hkv, int D, int ps, int ppr, int topk_n, uint8_t *out)
{
    for (int b = 0; b < B; ++b)
        for (int kk = 0; kk < topk_n; ++kk) {
            long t = topk[(size_t)b * topk_n + kk];
            long r = 0;
            long p = token_page(page_table, b, ppr, t, ps, &r);
            for (int g = 0; g < Hkv; ++g) {
                uint8_t *dst = out + (((size_t)b * topk_n + kk) * Hkv + g) * D;
                if (p < 0)
                    memset(dst, 0, (size_t)D);
                else
                    memcpy(dst, pool + pool_row(p, r, g, ps, Hkv, D), (size_t)D);
            }
        }
}

/*
 * q, gate : bf16 [B, Hq, D]
 * k_pool, v_pool : E4M3FN codes [num_pages, ps, Hkv, D]
 * page_table : int32 [B, ppr]      topk : int32 [B, topk_n]
 * rows : optional list of flattened (b*Hq + h) ids; NULL = all.
 * out  : [n_rows, D] gated output   lse : [n_rows] (ungated scores)
 * attn : optional [n_rows, D] ungated attention output.
 *
 * K^ = dec(k) * k_scale, V^ = dec(v) * v_scale, s_k = scale * q.K^_k,
 * O = softmax(s) V^, out = sigmoid(gate) * O with sigmoid(x) = 1/(1+e^-x).
 * A row whose indices are all padding has O = 0 and LSE = -inf.
 */
void oracle_gqa_decode_paged_fp8(const uint16_t *q, const uint16_t *gate,
                                 const uint8_t *k_pool, const uint8_t *v_pool,
                                 const int32_t *page_table, const int32_t *topk,
                                 double k_scale, double v_scale,
                                 int B, int Hq, int Hkv, int D, int ps, int ppr, int num_pages,
                                 int topk_n, double scale,
                                 const int32_t *rows, int n_rows,
                                 double *out, double *lse, double *attn)
{
    (void)num_pages;
    long total = rows ? n_rows : (long)B * Hq;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(topk_n > 0 ? topk_n : 1));
        long *row_at = (long *)malloc(sizeof(long) * (size_t)(topk_n > 0 ? topk_n : 1));
#pragma omp for schedule(dynamic, 1)
        for (long n = 0; n < total; ++n) {
            long r = rows ? rows[n] : n;
            int h = (int)(r % Hq);
            int b = (int)(r / Hq);
            int g = oracle_kv_head(h, Hq, Hkv);
            const uint16_t *qrow = q + ((size_t)b * Hq + h) * D;
            double m = -INFINITY;
            for (int kk = 0; kk < topk_n; ++kk) {
                long slot = 0;
                long p = token_page(page_table, b, ppr, topk[(size_t)b * topk_n + kk], ps, &slot);
                if (p < 0) {
                    row_at[kk] = -1;
                    continue;
                }
                row_at[kk] = (long)pool_row(p, slot, g, ps, Hkv, D);
                double dot = 0.0;
                for (int d = 0; d < D; ++d)
                    dot += bf16_value(qrow[d]) * (oracle_e4m3fn_value(k_pool[row_at[kk] + d]) * k_scale);
                s[kk] = scale * dot;
                if (s[kk] > m)
                    m = s[kk];
            }
            double sum = 0.0;
            for (int kk = 0; kk < topk_n; ++kk)
                if (row_at[kk] >= 0)
                    sum += exp(s[kk] - m);
            double L = (sum > 0.0) ? m + log(sum) : -INFINITY;
            double *o = out + (size_t)n * D;
            double *a = attn ? attn + (size_t)n * D : NULL;
            for (int d = 0; d < D; ++d) {
                double acc = 0.0;
                for (int kk = 0; kk < topk_n; ++kk) {
                    if (row_at[kk] < 0)
                        continue;
                    double vs = PLANT(9) ? 1.0 : v_scale;
                    acc += exp(s[kk] - L) * (oracle_e4m3fn_value(v_pool[row_at[kk] + d]) * vs);
                }
                double gx = bf16_value(gate[((size_t)b * Hq + h) * D + d]);
                double sig = PLANT(7) ? gx : 1.0 / (1.0 + exp(-gx));
                if (a)
                    a[d] = acc;
                o[d] = sig * acc;
            }
            if (lse)
                lse[n] = L;
        }
        free(row_at);
        free(s);
    }
}

/* ------------------------------------------------------------------ */
/* paged decode over whole requests (no top-K), bf16 or FP8 pools       */
/* ------------------------------------------------------------------ */

/* Value of element d of pool row `row` (offset of the row's first element):
 * kv_type 0 = a bf16 pattern, 1 = an E4M3FN code, 2 = a two's-complement
 * int8 code. */
static double pool_value(const void *pool, int kv_type, size_t row, int d)
{
    if (kv_type == 1)
        return oracle_e4m3fn_value(((const uint8_t *)pool)[row + d]);
    if (kv_type == 2) {
        int8_t c = ((const int8_t *)pool)[row + d];
        return PLANT(13) ? (double)(uint8_t)c : (double)c;
    }
    return bf16_value(((const uint16_t *)pool)[row + d]);
}

/*
 * q : bf16 [B, Sq, Hq, D]
 * k_pool, v_pool : [num_pages, ps, Hkv, D] of bf16 patterns (kv_type 0),
 *                  E4M3FN codes (kv_type 1) or int8 codes (kv_type 2)
 * page_table : int32 [B, ppr]      seq_lens : int32 [B], 0 <= seq_lens[b] <= ppr*ps
 * rows : optional list of flattened row ids r = (b*Hq + h)*Sq + i; NULL = all.
 * out : [n_rows, D] double        lse : [n_rows] double (natural log)
 *
 * Request b holds tokens t = 0 .. seq_lens[b]-1, token t at page
 * page_table[b][t / ps], slot t % ps.  Query row i of Sq sees tokens
 * t <= seq_lens[b] - Sq + i (bottom-right alignment, as in the dense case).
 * K^ = val(k) * k_scale, V^ = val(v) * v_scale (pass 1 for bf16 pools; an
 * int8 code c has the value c, the per-tensor scale gives the dequantised
 * value, the usual symmetric int8 cache format),
 * s_t = scale * q.K^_t, LSE = m + ln sum_t exp(s_t - m),
 * O = sum_t exp(s_t - LSE) V^_t.  A row that sees no token has O = 0 and
 * LSE = -inf.
 */
void oracle_gqa_decode_paged(const uint16_t *q, const void *k_pool, const void *v_pool, int kv_type,
                             double k_scale, double v_scale,
                             const int32_t *page_table, const int32_t *seq_lens,
                             int B, int Sq, int Hq, int Hkv, int D, int ps, int ppr,
                             double scale, const int32_t *rows, int n_rows,
                             double *out, double *lse)
{
    long cap = (long)ppr * ps;
    long total = rows ? n_rows : (long)B * Hq * Sq;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(cap > 0 ? cap : 1));
        size_t *row_at = (size_t *)malloc(sizeof(size_t) * (size_t)(cap > 0 ? cap : 1));
#pragma omp for schedule(dynamic, 1)
        for (long n = 0; n < total; ++n) {
            long r = rows ? rows[n] : n;
            int i = (int)(r % Sq);
            int h = (int)((r / Sq) % Hq);
            int b = (int)(r / ((long)Sq * Hq));
            int g = oracle_kv_head(h, Hq, Hkv);
            long len = PLANT(11) ? cap : (long)seq_lens[b];
            long last = last_visible_key(i, Sq, (int)len);
            double ks = PLANT(12) ? v_scale : k_scale;
            double vs = PLANT(12) ? k_scale : v_scale;
            const uint16_t *qrow = q + (((size_t)b * Sq + i) * Hq + h) * D;
            double m = -INFINITY;
            for (long t = 0; t <= last && t < len; ++t) {
                long slot = 0;
                long p = token_page(page_table, b, ppr, t, ps, &slot);
                row_at[t] = pool_row(p, slot, g, ps, Hkv, D);
                double dot = 0.0;
                for (int d = 0; d < D; ++d)
                    dot += bf16_value(qrow[d]) * (pool_value(k_pool, kv_type, row_at[t], d) * ks);
                s[t] = scale * dot;
                if (s[t] > m)
                    m = s[t];
            }
            double sum = 0.0;
            for (long t = 0; t <= last && t < len; ++t)
                sum += exp(s[t] - m);
            double L = (sum > 0.0) ? m + log(sum) : -INFINITY;
            double *o = out + (size_t)n * D;
            for (int d = 0; d < D; ++d)
                o[d] = 0.0;
            for (long t = 0; t <= last && t < len; ++t) {
                double w = exp(s[t] - L);
                for (int d = 0; d < D; ++d)
                    o[d] += w * (pool_value(v_pool, kv_type, row_at[t], d) * vs);
            }
            if (lse)
                lse[n] = L;
        }
        free(row_at);
        free(s);
    }
}
