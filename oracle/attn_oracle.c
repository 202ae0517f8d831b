/*
 * attn_oracle.c -- plain, slow, fp64 CPU oracle for grouped-query causal
 * prefill attention, single-query decode attention and the K/V cache append.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: it exists so that the tests, the smoke check and the CPU
 * baseline leg of the benchmark can compare the CUDA kernels against a
 * definition a reader can check by eye.  It shares no code, header, constant
 * or helper with the CUDA library.
 *
 * Every function materialises the whole score row, applies the mask, takes a
 * two-pass softmax (max, then exp/sum) and forms the weighted sum of V rows in
 * double precision.  Inputs are the fp32 tensors the GPU sees, promoted to
 * double on read; outputs are double.  OpenMP splits independent (head, row)
 * problems across threads; the arithmetic inside one problem runs in the
 * plain order written here.
 *
 * Sources (web pages, cited by title and section):
 *  [P1] "aprender-gpu 0.32.0 -- src/kernels/attention/flash/prefill_fused.rs",
 *       module doc (Algorithm, steps 1-3), `build_ptx` (parameter list, head
 *       bounds check, GQA map, packed-stride address arithmetic, causal
 *       column limit j <= i, online softmax, normalise and store).
 *  [P2] "soft3/glia/run/backend/honeycrisp/kernels/attention.rs", module doc
 *       (inputs, per-head formula, sliding window), `kmain` decode kernel
 *       (window start, -1e4 mask, softmax, normalise), KV_APPEND_TEMPLATE and
 *       KV_APPEND_BOTH_TEMPLATE (cache write at `position`),
 *       FUSED_ROPE_KV_ATTN_TEMPLATE (rotate-half RoPE of the new key and the
 *       query, append, decode).
 *
 * Parity pins: every function below is pinned by the `-m "not gpu"` tests
 * (closed forms, invariants, brute force, a library cross-check); none is
 * "parity unpinned".
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static void set_threads(int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Softmax-weighted sum over one materialised score row.
 * scores[0..n) already hold the masked scores; the weights are written back
 * into scores (so a caller may inspect them) and out[0..d) receives
 * sum_j w_j * V_j where row j of V starts at v + j * v_row_pitch.
 * Two-pass softmax: m = max_j s_j; w_j = exp(s_j - m) / sum_k exp(s_k - m).
 * A score of -INFINITY contributes weight exactly 0.
 */
static void softmax_weighted_sum(double *scores, size_t n, const float *v,
                                 size_t v_row_pitch, uint32_t d, double *out) {
    double m = -INFINITY;
    for (size_t j = 0; j < n; ++j)
        if (scores[j] > m) m = scores[j];
    double l = 0.0;
    for (size_t j = 0; j < n; ++j) {
        double p = (scores[j] == -INFINITY) ? 0.0 : exp(scores[j] - m);
        scores[j] = p;
        l += p;
    }
    for (size_t j = 0; j < n; ++j) scores[j] /= l;
    for (uint32_t e = 0; e < d; ++e) out[e] = 0.0;
    for (size_t j = 0; j < n; ++j) {
        if (scores[j] == 0.0) continue;
        const float *vr = v + j * v_row_pitch;
        for (uint32_t e = 0; e < d; ++e) out[e] += scores[j] * (double)vr[e];
    }
}

/*
 * Causal grouped-query prefill [P1 module doc, Algorithm; `build_ptx`].
 *
 *   Q, O : [m, q_stride] row pitch; head h occupies columns [h*d, (h+1)*d)
 *   K, V : [m, kv_stride] row pitch; KV head g occupies columns [g*d, (g+1)*d)
 *   kv head of query head h = h / (num_q_heads / num_kv_heads)   [P1 GQA map]
 *   s_ij = scale * sum_e Q[i,h,e] K[j,kvh,e]   for j <= i   (causal limit)
 *   s_ij = -inf                                 for j >  i   (never attended)
 *   O[i,h,:] = softmax_j(s_i.) . V[., kvh, :]
 *
 * rows: the query rows to evaluate (NULL = all rows 0..m-1, n_rows ignored).
 * o:    [n_rows or m, num_q_heads, d] doubles, dense (row r of the list at
 *       o + r * num_q_heads * d).
 * weights (optional, may be NULL): [n_rows, num_q_heads, m] doubles receiving
 *       the materialised softmax weights, zero for j > i.
 * Returns 0, or -1 on an argument the definition cannot take.
 */
int oracle_prefill_causal(const float *q, const float *k, const float *v,
                          uint32_t m, uint32_t num_q_heads, uint32_t num_kv_heads,
                          uint32_t d, uint32_t q_stride, uint32_t kv_stride,
                          double scale, const uint32_t *rows, uint32_t n_rows,
                          double *o, double *weights, int nthreads) {
    if (num_kv_heads == 0 || num_q_heads % num_kv_heads != 0 || d == 0) return -1;
    if (q_stride < num_q_heads * d || kv_stride < num_kv_heads * d) return -1;
    const uint32_t heads_per_kv = num_q_heads / num_kv_heads;
    const uint32_t nr = rows ? n_rows : m;
    for (uint32_t r = 0; r < nr; ++r)
        if (rows && rows[r] >= m) return -1;
    set_threads(nthreads);
    int bad = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (m ? m : 1));
        if (!s) {
#pragma omp atomic write
            bad = 1;
        }
#pragma omp for collapse(2) schedule(dynamic, 4)
        for (uint32_t r = 0; r < nr; ++r) {
            for (uint32_t h = 0; h < num_q_heads; ++h) {
                if (!s) continue;
                const uint32_t i = rows ? rows[r] : r;
                const uint32_t kvh = h / heads_per_kv;
                const float *qi = q + (size_t)i * q_stride + (size_t)h * d;
                for (uint32_t j = 0; j < m; ++j) {
                    if (j > i) { s[j] = -INFINITY; continue; }
                    const float *kj = k + (size_t)j * kv_stride + (size_t)kvh * d;
                    double dot = 0.0;
                    for (uint32_t e = 0; e < d; ++e) dot += (double)qi[e] * (double)kj[e];
                    s[j] = scale * dot;
                }
                double *out = o + ((size_t)r * num_q_heads + h) * d;
                softmax_weighted_sum(s, m, v + (size_t)kvh * d, kv_stride, d, out);
                if (weights)
                    memcpy(weights + ((size_t)r * num_q_heads + h) * m, s, sizeof(double) * m);
            }
        }
        free(s);
    }
    return bad ? -1 : 0;
}

/*
 * Single-query grouped-query decode against a [kv_heads, max_seq, d] cache
 * [P2 module doc; `kmain`].
 *
 *   q    : [num_heads, d]
 *   K, V : [kv_heads, max_seq, d]; rows 0..total_seq-1 are valid
 *   kvh  = h / (num_heads / kv_heads)
 *   s_s  = scale * q[h] . K[kvh, s]     for s in [0, total_seq)
 *   ws   = (window > 0 && total_seq > window) ? total_seq - window : 0
 *   s_s  = -1e4 (replacing the score) for s < ws
 *   out[h] = softmax(s) . V[kvh, 0..total_seq)
 *
 * out: [num_heads, d] doubles.  weights (optional): [num_heads, total_seq].
 * Returns 0, or -1 on an argument the definition cannot take (total_seq == 0
 * has no softmax; total_seq > max_seq reads outside the cache).
 */
static int decode_impl(const double *qd, const float *k_cache, const float *v_cache,
                       uint32_t num_heads, uint32_t kv_heads, uint32_t d, uint32_t max_seq,
                       uint32_t total_seq, uint32_t window, double scale, double *out,
                       double *weights, int nthreads) {
    if (kv_heads == 0 || num_heads % kv_heads != 0 || d == 0) return -1;
    if (total_seq == 0 || total_seq > max_seq) return -1;
    const uint32_t repeat = num_heads / kv_heads;
    const uint32_t ws = (window > 0 && total_seq > window) ? total_seq - window : 0;
    set_threads(nthreads);
    int bad = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * total_seq);
        if (!s) {
#pragma omp atomic write
            bad = 1;
        }
#pragma omp for schedule(static)
        for (uint32_t h = 0; h < num_heads; ++h) {
            if (!s) continue;
            const uint32_t kvh = h / repeat;
            const double *qh = qd + (size_t)h * d;
            const float *kb = k_cache + (size_t)kvh * max_seq * d;
            const float *vb = v_cache + (size_t)kvh * max_seq * d;
            for (uint32_t t = 0; t < total_seq; ++t) {
                const float *kr = kb + (size_t)t * d;
                double dot = 0.0;
                for (uint32_t e = 0; e < d; ++e) dot += qh[e] * (double)kr[e];
                s[t] = scale * dot;
                if (t < ws) s[t] = -1.0e4;
            }
            softmax_weighted_sum(s, total_seq, vb, d, d, out + (size_t)h * d);
            if (weights) memcpy(weights + (size_t)h * total_seq, s, sizeof(double) * total_seq);
        }
        free(s);
    }
    return bad ? -1 : 0;
}

int oracle_decode(const float *q, const float *k_cache, const float *v_cache,
                  uint32_t num_heads, uint32_t kv_heads, uint32_t d,
                  uint32_t max_seq, uint32_t total_seq, uint32_t window,
                  double scale, double *out, double *weights, int nthreads) {
    double *qd = (double *)malloc(sizeof(double) * (size_t)num_heads * (d ? d : 1));
    if (!qd) return -1;
    for (size_t i = 0; i < (size_t)num_heads * d; ++i) qd[i] = (double)q[i];
    const int rc = decode_impl(qd, k_cache, v_cache, num_heads, kv_heads, d, max_seq, total_seq,
                               window, scale, out, weights, nthreads);
    free(qd);
    return rc;
}

/*
 * K/V cache append [P2 KV_APPEND_TEMPLATE, KV_APPEND_BOTH_TEMPLATE]:
 *   cache[g, position, e] = src[g, e]   for every KV head g and element e.
 * v_src/v_cache may both be NULL (append to one cache only).
 * Returns 0, or -1 when position >= max_seq (outside the cache).
 */
int oracle_kv_append(const float *k_src, const float *v_src, float *k_cache,
                     float *v_cache, uint32_t kv_heads, uint32_t d,
                     uint32_t max_seq, uint32_t position) {
    if (position >= max_seq) return -1;
    if ((v_src == NULL) != (v_cache == NULL)) return -1;
    for (uint32_t g = 0; g < kv_heads; ++g) {
        for (uint32_t e = 0; e < d; ++e) {
            const size_t src = (size_t)g * d + e;
            const size_t dst = ((size_t)g * max_seq + position) * d + e;
            k_cache[dst] = k_src[src];
            if (v_cache) v_cache[dst] = v_src[src];
        }
    }
    return 0;
}

/*
 * Rotate-half RoPE of one vector [P2 FUSED_ROPE_KV_ATTN_TEMPLATE]: with
 * h = d / 2, element i pairs with i + h and
 *   y[i]     = x[i] cos[i] - x[i+h] sin[i]
 *   y[i + h] = x[i] sin[i] + x[i+h] cos[i]      for i in [0, h).
 * (The page fixes d = 128, h = 64; the same rule is applied to any even d.)
 */
static void rope(const double *x, const float *cosv, const float *sinv, uint32_t d, double *y) {
    const uint32_t h = d / 2;
    for (uint32_t i = 0; i < h; ++i) {
        const double c = (double)cosv[i], sn = (double)sinv[i];
        y[i] = x[i] * c - x[i + h] * sn;
        y[i + h] = x[i] * sn + x[i + h] * c;
    }
}

/*
 * Fused RoPE + append + decode [P2 FUSED_ROPE_KV_ATTN_TEMPLATE]:
 *   k_cache[g, position] = rope(k_new[g])   (rounded to the fp32 cache)
 *   v_cache[g, position] = v_new[g]
 *   q'[h] = rope(q[h])                      (kept in double)
 *   out = decode(q', caches, total_seq, window, scale)   (as oracle_decode)
 * rope_cos/rope_sin = NULL: no rotation (plain append + decode).
 * The caches are updated in place.  Returns 0, or -1 on a bad argument.
 */
int oracle_decode_append(const float *q, const float *k_new, const float *v_new,
                         const float *rope_cos, const float *rope_sin, float *k_cache,
                         float *v_cache, uint32_t num_heads, uint32_t kv_heads, uint32_t d,
                         uint32_t max_seq, uint32_t total_seq, uint32_t position,
                         uint32_t window, double scale, double *out, int nthreads) {
    if (position >= max_seq || d == 0 || (d % 2) != 0) return -1;
    if ((rope_cos == NULL) != (rope_sin == NULL)) return -1;
    double *tmp = (double *)malloc(sizeof(double) * d * 2);
    double *qd = (double *)malloc(sizeof(double) * (size_t)num_heads * d);
    if (!tmp || !qd) {
        free(tmp);
        free(qd);
        return -1;
    }
    for (uint32_t g = 0; g < kv_heads; ++g) {
        for (uint32_t e = 0; e < d; ++e) tmp[e] = (double)k_new[(size_t)g * d + e];
        if (rope_cos) rope(tmp, rope_cos, rope_sin, d, tmp + d);
        else memcpy(tmp + d, tmp, sizeof(double) * d);
        for (uint32_t e = 0; e < d; ++e) {
            const size_t dst = ((size_t)g * max_seq + position) * d + e;
            k_cache[dst] = (float)tmp[d + e];
            v_cache[dst] = v_new[(size_t)g * d + e];
        }
    }
    for (uint32_t h = 0; h < num_heads; ++h) {
        for (uint32_t e = 0; e < d; ++e) tmp[e] = (double)q[(size_t)h * d + e];
        if (rope_cos) rope(tmp, rope_cos, rope_sin, d, qd + (size_t)h * d);
        else memcpy(qd + (size_t)h * d, tmp, sizeof(double) * d);
    }
    const int rc = decode_impl(qd, k_cache, v_cache, num_heads, kv_heads, d, max_seq, total_seq,
                               window, scale, out, NULL, nthreads);
    free(tmp);
    free(qd);
    return rc;
}
