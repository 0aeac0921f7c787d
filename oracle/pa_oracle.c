/*
 * Plain fp64 CPU oracle for paged decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference legs of bench.py may load this library.  It shares
 * no code, header, table or helper with the CUDA library in
 * paged_kv_cache_64_gb300/csrc, and neither includes the other.
 *
 * Everything here is the plain definition, written out with loops:
 *
 *   For sequence i with L_i cached tokens and query head h:
 *     kv      = h / G                      (G = num_q_heads / num_kv_heads)
 *     K_i[p]  = K_pool[T_i[p / B], kv, p mod B, :]      p = 0 .. L_i - 1
 *     s_p     = scale * sum_x q[i, h, x] * K_i[p, x]
 *     w_p     = exp(s_p - max_p s_p) / sum_p exp(s_p - max_p s_p)
 *     out[i, h, :] = sum_p w_p * V_i[p, :]
 *
 * Sources (page title, section):
 *  - "PagedAttention and Virtual Memory Management: Mathematical Foundations
 *    of Non-Contiguous KV-Cache Allocation ..." (llms.blog), section 3
 *    (logical block index j = floor(t/B), offset o = t mod B, block-table
 *    lookup) and section 4 (Vectorized Address Computation: pool pointer +
 *    T[floor(tau/B)] * block stride + (tau mod B) * token stride + h * head
 *    stride; the decode pass over pools shaped
 *    [num_blocks, num_kv_heads, block_size, head_dim]).
 *  - "Why AI servers waste memory, and how paging fixes it" (spicyshark.co),
 *    "Reading through the table": scores over the valid slots of each block,
 *    softmax, weighted sum of values; "the math is ordinary attention".
 *  - Split-KV: same page on llms.blog, section 4 "Parallel Partitioning
 *    Across GPU Warps", steps 2 and 3: each partition k yields (m_k, l_k,
 *    O_k); the combine is m = max_k m_k, l = sum_k l_k exp(m_k - m),
 *    O = sum_k (l_k exp(m_k - m) / l) O_k.
 *
 * Readings where the pages are silent (also listed in the design notes):
 *  - GQA head map: query head h reads KV head h / G (consecutive groups).
 *  - A sequence with L_i = 0 gives an all-zero output row.
 *  - Slots past L_i (in the last block or in unreferenced blocks) are never
 *    read, whatever they hold.
 *
 * Element types are raw 16-bit patterns (IEEE binary16 or bfloat16), widened
 * exactly to double from their bit definitions below.
 *
 * FP8 KV cache (a variant): "b = 1 for FP8" in the KV-size formula of the
 * llms.blog page above, section 1, is the pages' only word on it.  Readings:
 * the format is OCP 8-bit floating point E4M3 (1 sign, 4 exponent bits with
 * bias 7, 3 mantissa bits; subnormals; no infinities; S.1111.111 is NaN; the
 * largest finite value is 448), and each K or V pool has one scale: element
 * value = scale * code value.  Quantisation (the cache write) takes the
 * fp32 value x of a 16-bit input, the fp32 product y = x * fl32(1 / scale),
 * and rounds y to the nearest E4M3 value (ties to even), saturating at
 * +-448.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_F16 = 0, ORACLE_BF16 = 1, ORACLE_E4M3 = 2 };

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double f16_bits_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24); /* subnormal: f * 2^(1 - 15 - 10) */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(f + 1024), e - 25); /* (1 + f/2^10) * 2^(e - 15) */
    return sign ? -v : v;
}

/* bfloat16 is the upper half of an IEEE binary32. */
static double bf16_bits_to_double(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double widen(uint16_t x, int dtype) {
    return dtype == ORACLE_BF16 ? bf16_bits_to_double(x) : f16_bits_to_double(x);
}

/* OCP E4M3: exponent field E, mantissa M; E = 0 is subnormal, M * 2^-9;
 * otherwise (1 + M/8) * 2^(E - 7); E = 15, M = 7 is NaN. */
static double e4m3_bits_to_double(uint8_t c) {
    int sign = (c >> 7) & 1;
    int e = (c >> 3) & 15;
    int m = c & 7;
    double v;
    if (e == 15 && m == 7)
        v = NAN;
    else if (e == 0)
        v = ldexp((double)m, -9);
    else
        v = ldexp((double)(8 + m), e - 10);
    return sign ? -v : v;
}

/* Nearest E4M3 code of y (ties to even), saturating at +-448.  Within the
 * binade [2^E, 2^(E+1)) the spacing is 2^(E-3); below 2^-6 it is the
 * subnormal spacing 2^-9.  NaN gives the NaN code. */
static uint8_t e4m3_from_float(float y) {
    uint8_t sign = signbit(y) ? 0x80 : 0x00;
    if (isnan(y)) return (uint8_t)(sign | 0x7F);
    double a = fabs((double)y);
    if (a >= 448.0) return (uint8_t)(sign | 0x7E); /* 448 = 1.75 * 2^8 */
    if (a == 0.0) return sign;
    int ex;
    frexp(a, &ex);          /* a = f * 2^ex, f in [0.5, 1) */
    int E = ex - 1;         /* 2^E <= a < 2^(E+1) */
    if (E < -6) E = -6;     /* subnormal range shares the spacing of 2^-6 */
    double spacing = ldexp(1.0, E - 3);
    double v = rint(a / spacing) * spacing; /* default rounding: nearest, ties to even */
    if (v == 0.0) return sign;
    if (v < ldexp(1.0, -6)) return (uint8_t)(sign | (int)(v / ldexp(1.0, -9)));
    frexp(v, &ex);
    E = ex - 1;
    int m = (int)(v / ldexp(1.0, E) * 8.0) - 8;
    return (uint8_t)(sign | ((E + 7) << 3) | m);
}

void pa_oracle_e4m3_decode(double *dst, const uint8_t *src, int64_t n) {
    for (int64_t i = 0; i < n; ++i) dst[i] = e4m3_bits_to_double(src[i]);
}

void pa_oracle_e4m3_encode(uint8_t *dst, const float *src, int64_t n) {
    for (int64_t i = 0; i < n; ++i) dst[i] = e4m3_from_float(src[i]);
}

/* A K or V pool as the decode reads it: element i of `data` is a 16-bit
 * pattern (f16 / bf16) or an E4M3 code times `scale`. */
typedef struct {
    const void *data;
    int kind;
    double scale;
} pool_view;

static double pool_elem(const pool_view *pv, int64_t i) {
    if (pv->kind == ORACLE_E4M3) return pv->scale * e4m3_bits_to_double(((const uint8_t *)pv->data)[i]);
    return widen(((const uint16_t *)pv->data)[i], pv->kind);
}

int pa_oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void pa_oracle_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* Widen a whole array of 16-bit patterns (used by tests to read GPU outputs
 * and by the contiguous cross-check). */
void pa_oracle_widen(double *dst, const uint16_t *src, int64_t n, int dtype) {
    for (int64_t i = 0; i < n; ++i) dst[i] = widen(src[i], dtype);
}

/* Element index of token p of sequence i, KV head kv, in a pool laid out
 * [num_blocks][num_kv_heads][block_size][head_dim]:
 *   physical block = T_i[p / B], slot = p mod B. */
static int64_t token_row(const int32_t *table_i, int p, int kv, int num_kv_heads, int block_size,
                         int head_dim) {
    int64_t j = p / block_size; /* logical block index */
    int64_t o = p % block_size; /* offset inside the block */
    int64_t phys = table_i[j];  /* block-table lookup */
    return ((phys * num_kv_heads + kv) * block_size + o) * head_dim;
}

/* Scores s_p for positions [p0, p1) of (sequence i, query head h). */
static void scores(double *s, const uint16_t *q_ih, const pool_view *k_pool, const int32_t *table_i,
                   int p0, int p1, int kv, int num_kv_heads, int block_size, int head_dim,
                   double scale, int dtype) {
    for (int p = p0; p < p1; ++p) {
        int64_t k = token_row(table_i, p, kv, num_kv_heads, block_size, head_dim);
        double dot = 0.0;
        for (int x = 0; x < head_dim; ++x) dot += widen(q_ih[x], dtype) * pool_elem(k_pool, k + x);
        s[p - p0] = scale * dot;
    }
}

/* Softmax-weighted sum over positions [p0, p1):
 *   m = max s, l = sum exp(s - m), o = sum exp(s - m) v / l.  */
static void attend_range(double *o, double *m_out, double *l_out, const uint16_t *q_ih,
                         const pool_view *k_pool, const pool_view *v_pool, const int32_t *table_i,
                         int p0, int p1, int kv, int num_kv_heads, int block_size, int head_dim,
                         double scale, int dtype) {
    int n = p1 - p0;
    for (int x = 0; x < head_dim; ++x) o[x] = 0.0;
    if (n <= 0) {
        *m_out = -INFINITY;
        *l_out = 0.0;
        return;
    }
    double *s = (double *)malloc(sizeof(double) * (size_t)n);
    scores(s, q_ih, k_pool, table_i, p0, p1, kv, num_kv_heads, block_size, head_dim, scale, dtype);
    double m = -INFINITY;
    for (int t = 0; t < n; ++t)
        if (s[t] > m) m = s[t];
    double l = 0.0;
    for (int t = 0; t < n; ++t) l += exp(s[t] - m);
    for (int t = 0; t < n; ++t) {
        double w = exp(s[t] - m) / l;
        int64_t v = token_row(table_i, p0 + t, kv, num_kv_heads, block_size, head_dim);
        for (int x = 0; x < head_dim; ++x) o[x] += w * pool_elem(v_pool, v + x);
    }
    free(s);
    *m_out = m;
    *l_out = l;
}

static int check_dims(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int block_size) {
    if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0)
        return 1;
    if (num_q_heads % num_kv_heads) return 1;
    return 0;
}

/* Decode over pools given as views (16-bit or E4M3 elements). */
static int decode_views(double *out, const uint16_t *q, const pool_view *kp, const pool_view *vp,
                        int dtype, const int32_t *block_tables, int max_blocks_per_seq,
                        const int32_t *seq_lens, int num_seqs, int num_q_heads, int num_kv_heads,
                        int head_dim, int block_size, double scale, const int32_t *seq_subset,
                        int n_subset) {
    if (check_dims(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size)) return 1;
    int G = num_q_heads / num_kv_heads;
    int n_rows = seq_subset ? n_subset : num_seqs;
    int64_t n_work = (int64_t)n_rows * num_q_heads;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t w = 0; w < n_work; ++w) {
        int i = seq_subset ? seq_subset[w / num_q_heads] : (int)(w / num_q_heads);
        int h = (int)(w % num_q_heads);
        int kv = h / G;
        const int32_t *table_i = block_tables + (int64_t)i * max_blocks_per_seq;
        const uint16_t *q_ih = q + ((int64_t)i * num_q_heads + h) * head_dim;
        double *o = out + ((int64_t)i * num_q_heads + h) * head_dim;
        double m, l;
        attend_range(o, &m, &l, q_ih, kp, vp, table_i, 0, seq_lens[i], kv, num_kv_heads,
                     block_size, head_dim, scale, dtype);
    }
    return 0;
}

/* out[num_seqs][num_q_heads][head_dim] (double).  If seq_subset is not NULL,
 * only those sequences' rows are computed (the rest are left untouched). */
int pa_oracle_decode(double *out, const uint16_t *q, const uint16_t *k_pool, const uint16_t *v_pool,
                     int dtype, const int32_t *block_tables, int max_blocks_per_seq,
                     const int32_t *seq_lens, int num_seqs, int num_q_heads, int num_kv_heads,
                     int head_dim, int block_size, double scale, const int32_t *seq_subset,
                     int n_subset) {
    pool_view kp = {k_pool, dtype, 1.0}, vp = {v_pool, dtype, 1.0};
    return decode_views(out, q, &kp, &vp, dtype, block_tables, max_blocks_per_seq, seq_lens,
                        num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, scale,
                        seq_subset, n_subset);
}

/* The same over E4M3 pools: K element = k_scale * code value, V element =
 * v_scale * code value; q (and the output) of 16-bit type q_dtype. */
int pa_oracle_decode_fp8(double *out, const uint16_t *q, const uint8_t *k_pool,
                         const uint8_t *v_pool, int q_dtype, double k_scale, double v_scale,
                         const int32_t *block_tables, int max_blocks_per_seq,
                         const int32_t *seq_lens, int num_seqs, int num_q_heads,
                         int num_kv_heads, int head_dim, int block_size, double scale,
                         const int32_t *seq_subset, int n_subset) {
    pool_view kp = {k_pool, ORACLE_E4M3, k_scale}, vp = {v_pool, ORACLE_E4M3, v_scale};
    return decode_views(out, q, &kp, &vp, q_dtype, block_tables, max_blocks_per_seq, seq_lens,
                        num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, scale,
                        seq_subset, n_subset);
}

/* Split-KV step 2: partition k of sequence i covers positions
 * [k*P, min((k+1)*P, L_i)).  For each (i, h, k):
 *   m[i][h][k] = max s,  l[i][h][k] = sum exp(s - m),  o[i][h][k][:] = normalised
 *   partial output.  Partitions past the end get m = -inf, l = 0, o = 0. */
int pa_oracle_partitions(double *m_out, double *l_out, double *o_out, const uint16_t *q,
                         const uint16_t *k_pool, const uint16_t *v_pool, int dtype,
                         const int32_t *block_tables, int max_blocks_per_seq,
                         const int32_t *seq_lens, int num_seqs, int num_q_heads, int num_kv_heads,
                         int head_dim, int block_size, double scale, int partition_tokens,
                         int max_partitions) {
    if (check_dims(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size)) return 1;
    if (partition_tokens <= 0 || max_partitions <= 0) return 1;
    pool_view kp = {k_pool, dtype, 1.0}, vp = {v_pool, dtype, 1.0};
    int G = num_q_heads / num_kv_heads;
    int64_t n_work = (int64_t)num_seqs * num_q_heads * max_partitions;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t w = 0; w < n_work; ++w) {
        int k = (int)(w % max_partitions);
        int h = (int)((w / max_partitions) % num_q_heads);
        int i = (int)(w / ((int64_t)max_partitions * num_q_heads));
        int L = seq_lens[i];
        int p0 = k * partition_tokens;
        int p1 = p0 + partition_tokens < L ? p0 + partition_tokens : L;
        const int32_t *table_i = block_tables + (int64_t)i * max_blocks_per_seq;
        const uint16_t *q_ih = q + ((int64_t)i * num_q_heads + h) * head_dim;
        attend_range(o_out + w * head_dim, &m_out[w], &l_out[w], q_ih, &kp, &vp, table_i, p0,
                     p1, h / G, num_kv_heads, block_size, head_dim, scale, dtype);
    }
    return 0;
}

/* Split-KV step 3 (the cross-partition combine), for every row r of
 * num_rows rows with max_partitions partials each:
 *   m = max_k m_k ;  l = sum_k l_k exp(m_k - m) ;
 *   out = sum_k (l_k exp(m_k - m) / l) O_k .
 * Partials with m_k = -inf (empty partitions) contribute nothing; a row with
 * no non-empty partial gives zeros. */
void pa_oracle_reduce(double *out, const double *m, const double *l, const double *o,
                      int64_t num_rows, int max_partitions, int head_dim) {
    for (int64_t r = 0; r < num_rows; ++r) {
        const double *mr = m + r * max_partitions;
        const double *lr = l + r * max_partitions;
        double *dst = out + r * head_dim;
        double mg = -INFINITY;
        for (int k = 0; k < max_partitions; ++k)
            if (mr[k] > mg) mg = mr[k];
        for (int x = 0; x < head_dim; ++x) dst[x] = 0.0;
        if (mg == -INFINITY) continue;
        double lg = 0.0;
        for (int k = 0; k < max_partitions; ++k)
            if (mr[k] != -INFINITY) lg += lr[k] * exp(mr[k] - mg);
        for (int k = 0; k < max_partitions; ++k) {
            if (mr[k] == -INFINITY) continue;
            double wk = lr[k] * exp(mr[k] - mg) / lg;
            const double *ok = o + (r * max_partitions + k) * head_dim;
            for (int x = 0; x < head_dim; ++x) dst[x] += wk * ok[x];
        }
    }
}
