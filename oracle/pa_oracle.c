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
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_F16 = 0, ORACLE_BF16 = 1 };

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

/* Address of token p of sequence i, KV head kv, in a pool laid out
 * [num_blocks][num_kv_heads][block_size][head_dim]:
 *   physical block = T_i[p / B], slot = p mod B. */
static const uint16_t *token_row(const uint16_t *pool, const int32_t *table_i, int p, int kv,
                                 int num_kv_heads, int block_size, int head_dim) {
    int64_t j = p / block_size; /* logical block index */
    int64_t o = p % block_size; /* offset inside the block */
    int64_t phys = table_i[j];  /* block-table lookup */
    return pool + ((phys * num_kv_heads + kv) * block_size + o) * head_dim;
}

/* Scores s_p for positions [p0, p1) of (sequence i, query head h). */
static void scores(double *s, const uint16_t *q_ih, const uint16_t *k_pool, const int32_t *table_i,
                   int p0, int p1, int kv, int num_kv_heads, int block_size, int head_dim,
                   double scale, int dtype) {
    for (int p = p0; p < p1; ++p) {
        const uint16_t *k = token_row(k_pool, table_i, p, kv, num_kv_heads, block_size, head_dim);
        double dot = 0.0;
        for (int x = 0; x < head_dim; ++x) dot += widen(q_ih[x], dtype) * widen(k[x], dtype);
        s[p - p0] = scale * dot;
    }
}

/* Softmax-weighted sum over positions [p0, p1):
 *   m = max s, l = sum exp(s - m), o = sum exp(s - m) v / l.  */
static void attend_range(double *o, double *m_out, double *l_out, const uint16_t *q_ih,
                         const uint16_t *k_pool, const uint16_t *v_pool, const int32_t *table_i,
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
        const uint16_t *v = token_row(v_pool, table_i, p0 + t, kv, num_kv_heads, block_size, head_dim);
        for (int x = 0; x < head_dim; ++x) o[x] += w * widen(v[x], dtype);
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

/* out[num_seqs][num_q_heads][head_dim] (double).  If seq_subset is not NULL,
 * only the listed sequences are computed and the other rows are left as they
 * are.  Returns 0 on success, 1 on bad dimensions. */
int pa_oracle_decode(double *out, const uint16_t *q, const uint16_t *k_pool, const uint16_t *v_pool,
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
        attend_range(o, &m, &l, q_ih, k_pool, v_pool, table_i, 0, seq_lens[i], kv, num_kv_heads,
                     block_size, head_dim, scale, dtype);
    }
    return 0;
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
        attend_range(o_out + w * head_dim, &m_out[w], &l_out[w], q_ih, k_pool, v_pool, table_i, p0,
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
