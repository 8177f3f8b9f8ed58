/*
 * Float64 CPU oracle for chunked-prefill extend attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the package smoke check and
 * the CPU-baseline leg of the benchmark may load this library.  The CUDA path
 * shares no code, header, table or helper with it; neither side includes or
 * links the other.
 *
 * What it computes, and where the pages define it:
 *
 *  - extend attention, direct form.  SGLang chunked-prefill article
 *    (zdszero.github.io/chunked_prefill.html), section on splitting one prefill
 *    into resumable extends, the equation for o_i: query i of the chunk, at
 *    global position P+i, attends to every key j in [0, P+i] with weights
 *    exp(q_i . k_j / sqrt(d)), normalised by their sum.  Keys j < P come from
 *    the cache, keys j >= P from this round's new K/V.  Both live in the paged
 *    cache here (the KV-append step writes the new rows before attention).
 *
 *  - extend attention, two-stage form.  Same section: Stage 1 is the unmasked
 *    prefix rectangle, Stage 2 the causal triangle inside the chunk, each with
 *    its log-sum-exp statistics (m, l), merged by the online-softmax formula
 *    m = max(m1, m2),
 *    o = (e^{m1-m} l1 o1 + e^{m2-m} l2 o2) / (e^{m1-m} l1 + e^{m2-m} l2).
 *
 *  - one-shot causal attention on contiguous Q/K/V: the reference point for
 *    the statement (same section, and its closing summary) that chunked extend
 *    equals one-shot prefill up to floating-point summation order.
 *
 *  - KV append: the chunk's K/V rows are written into pages at positions
 *    [P, P+E).  Same article, section on where the half-finished request's KV
 *    lives (the request's req_to_token row keeps its page slots across chunks);
 *    mini-infer article (smarter.xin/posts/c9e9b85f), write_prefill_kv.
 *
 * Conventions (readings where the pages are silent):
 *  - query head h uses KV head floor(h / G), G = H_q / H_kv;
 *  - scale = 1/sqrt(d) unless given, natural exponential, lse = m + ln(l)
 *    with m taken over the scaled scores;
 *  - inputs are raw fp32 or bf16 element arrays, widened exactly to double.
 *
 * Layouts (row-major, last dimension contiguous):
 *  q, out      [total_q, H_q, d]
 *  k/v cache   [num_pages, page_size, H_kv, d]
 *  page_table  [n_seqs, max_pages] int32
 *  qo_indptr   [n_seqs + 1] int32, prefix_len [n_seqs] int32
 *  lse         [total_q, H_q]
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_F32 0
#define ORC_BF16 1

/* Deliberate mistakes, switched on only by the test that checks the pins
 * catch them.  0 = none.  See oracle_set_fault(). */
static int g_fault = 0;

void oracle_set_fault(int code) { g_fault = code; }

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

static double widen(const void* base, int dtype, int64_t idx) {
    if (dtype == ORC_F32) return (double)((const float*)base)[idx];
    uint32_t bits = (uint32_t)((const uint16_t*)base)[idx] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* Sequence that owns global query row r: the s with indptr[s] <= r < indptr[s+1]. */
static int seq_of_row(const int32_t* qo_indptr, int n_seqs, int64_t r) {
    int lo = 0, hi = n_seqs - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) / 2;
        if (qo_indptr[mid] <= r) lo = mid; else hi = mid - 1;
    }
    return lo;
}

/* Element offset of (position j of sequence s, KV head g, dim 0) in the cache. */
static int64_t cache_off(const int32_t* page_table, int max_pages, int s, int64_t j,
                         int page_size, int h_kv, int g, int d) {
    int64_t page = page_table[(int64_t)s * max_pages + j / page_size];
    int64_t slot = j % page_size;
    return ((page * page_size + slot) * h_kv + g) * (int64_t)d;
}

/* Softmax-weighted sum over keys [j0, j1) for one (query row, head).
 * Returns the partial statistics (m, l) and the normalised partial output o
 * (o = sum_j e^{s_j - m} v_j / l).  An empty range gives m = -inf, l = 0, o = 0. */
static void attend_range(const void* q, const void* kc, const void* vc, int dtype,
                         const int32_t* page_table, int max_pages, int s, int64_t qrow,
                         int h, int g, int64_t j0, int64_t j1, int h_q, int h_kv, int d,
                         int page_size, double scale, double* m_out, double* l_out,
                         double* o, double* scores) {
    for (int c = 0; c < d; ++c) o[c] = 0.0;
    if (j1 <= j0) { *m_out = -INFINITY; *l_out = 0.0; return; }
    int64_t qoff = (qrow * h_q + h) * (int64_t)d;
    double m = -INFINITY;
    for (int64_t j = j0; j < j1; ++j) {
        int64_t ko = cache_off(page_table, max_pages, s, j, page_size, h_kv, g, d);
        double dot = 0.0;
        for (int c = 0; c < d; ++c) dot += widen(q, dtype, qoff + c) * widen(kc, dtype, ko + c);
        double sc = dot * scale;
        scores[j - j0] = sc;
        if (sc > m) m = sc;
    }
    double l = 0.0;
    for (int64_t j = j0; j < j1; ++j) {
        double p = exp(scores[j - j0] - m);
        l += p;
        int64_t vo = cache_off(page_table, max_pages, s, j, page_size, h_kv, g, d);
        for (int c = 0; c < d; ++c) o[c] += p * widen(vc, dtype, vo + c);
    }
    for (int c = 0; c < d; ++c) o[c] /= l;
    *m_out = m;
    *l_out = l;
}

/*
 * Direct form.  rows == NULL computes every query row; otherwise only the
 * n_rows listed global rows, written densely to out[n_rows, H_q, d] and
 * lse[n_rows, H_q] (lse may be NULL).
 */
int oracle_extend_attention(const void* q, const void* k_cache, const void* v_cache, int dtype,
                            const int32_t* page_table, int max_pages, const int32_t* qo_indptr,
                            const int32_t* prefix_len, int n_seqs, int64_t total_q, int h_q,
                            int h_kv, int d, int page_size, double scale, const int64_t* rows,
                            int64_t n_rows, double* out, double* lse) {
    if (h_kv <= 0 || h_q % h_kv != 0 || d <= 0 || page_size <= 0 || n_seqs <= 0) return 1;
    int G = h_q / h_kv;
    int64_t nr = rows ? n_rows : total_q;
    int64_t max_keys = 0;
    for (int s = 0; s < n_seqs; ++s) {
        int64_t kv = (int64_t)prefix_len[s] + (qo_indptr[s + 1] - qo_indptr[s]);
        if (kv > max_keys) max_keys = kv;
    }
    int err = 0;
#pragma omp parallel
    {
        double* scores = (double*)malloc(sizeof(double) * (size_t)(max_keys + 1));
        double* o = (double*)malloc(sizeof(double) * (size_t)d);
        if (!scores || !o) {
#pragma omp atomic write
            err = 2;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (int64_t t = 0; t < nr * h_q; ++t) {
                int64_t ri = t / h_q;
                int h = (int)(t % h_q);
                int64_t r = rows ? rows[ri] : ri;
                int s = seq_of_row(qo_indptr, n_seqs, r);
                int64_t i = r - qo_indptr[s];
                int g = h / G;
                if (g_fault == 3) g = h % h_kv;            /* planted: wrong GQA map */
                int64_t last = (int64_t)prefix_len[s] + i; /* key P+i included */
                if (g_fault == 1) last -= 1;               /* planted: diagonal dropped */
                double sc = scale;
                if (g_fault == 2) sc = 1.0 / (double)d;    /* planted: wrong scale */
                double m, l;
                attend_range(q, k_cache, v_cache, dtype, page_table, max_pages, s, r, h, g, 0,
                             last + 1, h_q, h_kv, d, page_size, sc, &m, &l, o, scores);
                double* dst = out + (ri * h_q + h) * (int64_t)d;
                for (int c = 0; c < d; ++c) dst[c] = o[c];
                if (lse) lse[ri * h_q + h] = m + log(l);
            }
        }
        free(scores);
        free(o);
    }
    return err;
}

/* Online-softmax merge of two normalised partials (P5, the merge equation).
 * An empty partial (l = 0) contributes nothing. */
static void lse_merge(double m1, double l1, const double* o1, double m2, double l2,
                      const double* o2, int d, double* m_out, double* l_out, double* o) {
    double m = m1 > m2 ? m1 : m2;
    double w1 = (l1 > 0.0) ? exp(m1 - m) * l1 : 0.0;
    double w2 = (l2 > 0.0) ? exp(m2 - m) * l2 : 0.0;
    for (int c = 0; c < d; ++c) {
        double a = (l1 > 0.0) ? w1 * o1[c] : 0.0;
        double b = (l2 > 0.0) ? w2 * o2[c] : 0.0;
        o[c] = (a + b) / (w1 + w2);
    }
    *m_out = m;
    *l_out = w1 + w2;
}

/* Two-stage form: Stage 1 over the prefix [0, P), Stage 2 over [P, P+i], then
 * the merge.  Same arguments as the direct form. */
int oracle_extend_attention_two_stage(const void* q, const void* k_cache, const void* v_cache,
                                      int dtype, const int32_t* page_table, int max_pages,
                                      const int32_t* qo_indptr, const int32_t* prefix_len,
                                      int n_seqs, int64_t total_q, int h_q, int h_kv, int d,
                                      int page_size, double scale, const int64_t* rows,
                                      int64_t n_rows, double* out, double* lse) {
    if (h_kv <= 0 || h_q % h_kv != 0 || d <= 0 || page_size <= 0 || n_seqs <= 0) return 1;
    int G = h_q / h_kv;
    int64_t nr = rows ? n_rows : total_q;
    int64_t max_keys = 0;
    for (int s = 0; s < n_seqs; ++s) {
        int64_t kv = (int64_t)prefix_len[s] + (qo_indptr[s + 1] - qo_indptr[s]);
        if (kv > max_keys) max_keys = kv;
    }
    int err = 0;
#pragma omp parallel
    {
        double* scores = (double*)malloc(sizeof(double) * (size_t)(max_keys + 1));
        double* o1 = (double*)malloc(sizeof(double) * (size_t)d * 3);
        if (!scores || !o1) {
#pragma omp atomic write
            err = 2;
        } else {
            double* o2 = o1 + d;
            double* o = o2 + d;
#pragma omp for schedule(dynamic, 4)
            for (int64_t t = 0; t < nr * h_q; ++t) {
                int64_t ri = t / h_q;
                int h = (int)(t % h_q);
                int64_t r = rows ? rows[ri] : ri;
                int s = seq_of_row(qo_indptr, n_seqs, r);
                int64_t i = r - qo_indptr[s];
                int g = h / G;
                int64_t P = prefix_len[s];
                double m1, l1, m2, l2, m, l;
                attend_range(q, k_cache, v_cache, dtype, page_table, max_pages, s, r, h, g, 0, P,
                             h_q, h_kv, d, page_size, scale, &m1, &l1, o1, scores);
                attend_range(q, k_cache, v_cache, dtype, page_table, max_pages, s, r, h, g, P,
                             P + i + 1, h_q, h_kv, d, page_size, scale, &m2, &l2, o2, scores);
                lse_merge(m1, l1, o1, m2, l2, o2, d, &m, &l, o);
                double* dst = out + (ri * h_q + h) * (int64_t)d;
                for (int c = 0; c < d; ++c) dst[c] = o[c];
                if (lse) lse[ri * h_q + h] = m + log(l);
            }
        }
        free(scores);
        free(o1);
    }
    return err;
}

/* One-shot causal attention over contiguous q [N, H_q, d], k/v [N, H_kv, d]:
 * row i attends to keys [0, i].  Independent of pages and chunking. */
int oracle_causal_attention(const void* q, const void* k, const void* v, int dtype, int64_t n,
                            int h_q, int h_kv, int d, double scale, double* out, double* lse) {
    if (h_kv <= 0 || h_q % h_kv != 0 || d <= 0 || n <= 0) return 1;
    int G = h_q / h_kv;
    int err = 0;
#pragma omp parallel
    {
        double* scores = (double*)malloc(sizeof(double) * (size_t)n);
        if (!scores) {
#pragma omp atomic write
            err = 2;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (int64_t t = 0; t < n * h_q; ++t) {
                int64_t i = t / h_q;
                int h = (int)(t % h_q);
                int g = h / G;
                int64_t qo = (i * h_q + h) * (int64_t)d;
                double m = -INFINITY;
                for (int64_t j = 0; j <= i; ++j) {
                    int64_t ko = (j * h_kv + g) * (int64_t)d;
                    double dot = 0.0;
                    for (int c = 0; c < d; ++c) dot += widen(q, dtype, qo + c) * widen(k, dtype, ko + c);
                    scores[j] = dot * scale;
                    if (scores[j] > m) m = scores[j];
                }
                double l = 0.0;
                double* dst = out + qo;
                for (int c = 0; c < d; ++c) dst[c] = 0.0;
                for (int64_t j = 0; j <= i; ++j) {
                    double p = exp(scores[j] - m);
                    l += p;
                    int64_t vo = (j * h_kv + g) * (int64_t)d;
                    for (int c = 0; c < d; ++c) dst[c] += p * widen(v, dtype, vo + c);
                }
                for (int c = 0; c < d; ++c) dst[c] /= l;
                if (lse) lse[i * h_q + h] = m + log(l);
            }
        }
        free(scores);
    }
    return err;
}

/*
 * KV append as a plain byte scatter: new row r of sequence s (r in
 * [indptr[s], indptr[s+1])) goes to position P_s + (r - indptr[s]) of that
 * sequence, i.e. page page_table[s][pos / page_size], slot pos % page_size.
 * One token's [H_kv, d] block is contiguous on both sides.
 */
int oracle_kv_append(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                     int64_t num_pages, const int32_t* page_table, int max_pages,
                     const int32_t* qo_indptr, const int32_t* prefix_len, int n_seqs, int h_kv,
                     int d, int page_size, int elem_bytes) {
    int64_t row_bytes = (int64_t)h_kv * d * elem_bytes;
    for (int s = 0; s < n_seqs; ++s) {
        for (int64_t r = qo_indptr[s]; r < qo_indptr[s + 1]; ++r) {
            int64_t pos = (int64_t)prefix_len[s] + (r - qo_indptr[s]);
            if (pos / page_size >= max_pages) return 1;
            int64_t page = page_table[(int64_t)s * max_pages + pos / page_size];
            if (page < 0 || page >= num_pages) return 1;
            int64_t dst = (page * page_size + pos % page_size) * row_bytes;
            memcpy((char*)k_cache + dst, (const char*)k_new + r * row_bytes, (size_t)row_bytes);
            memcpy((char*)v_cache + dst, (const char*)v_new + r * row_bytes, (size_t)row_bytes);
        }
    }
    return 0;
}
