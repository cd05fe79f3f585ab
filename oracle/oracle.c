/*
 * oracle.c -- plain fp64 CPU oracle for the scaled-dot-product attention forward
 * (prefill with an optional causal mask, and single-token decode against a KV cache),
 * with grouped-query attention.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's CPU-baseline
 * leg load this file. The CUDA library never links, includes or calls it, and it shares
 * no code, header, table or helper with the CUDA library.
 *
 * What it computes is the plain definition the fused kernels must reach (up to rounding):
 *
 *   "Attention three-op fusion" (xdnf.cn/news/349386), section 1.1:
 *       S = Q K^T * scale;  P = row-softmax(S);  O = P V        (one head)
 *   same page, section 3.2 (second remark): the scale multiplies the scores before softmax.
 *   same page, section 4.3 / section 6.1 (first item): a masked score is -infinity, so that
 *       exp() gives it weight 0; causal: query i sees key j only when j <= i; keys at or
 *       beyond the valid length are masked the same way.
 *   "CS336 Lecture 6: kernels and Triton" (semidirectx.com), section 6: the row softmax is
 *       subtract-the-row-max, exponentiate, divide by the row sum (two passes over the row);
 *       masked entries must be -infinity, not 0.
 *   "Hand-written Triton decoder" (m.nlpx.cn/news/28229), section 2.1: 2 KV heads are
 *       broadcast to 8 query heads (grouped-query attention). Reading taken here: contiguous
 *       groups, kv head = query head / (Hq / Hkv).
 *   "triton-optimization" skill (skillsmp.com), section 3.5: log-sum-exp of a row = m + log(d).
 *
 * Every value is fp64; inputs are the exact fp64 widening of what the GPU reads. The score
 * row is materialised in full, the mask is applied, then a two-pass softmax (max, then sum)
 * and the weighted sum of V rows. No blocking, fusion or reordering beyond that.
 *
 * The online-softmax recurrence and the block merge (the method the kernels use) are here
 * too, written from:
 *   "Attention three-op fusion", section 2.2 (running max m, running sum l, correction
 *       factor exp(m - m_new); merge order does not matter) and section 2.3 (the
 *       accumulated output is corrected with the same factor and divided by l at the end);
 *   same page, section 4.4 (keys split into chunks, partial results merged across blocks).
 * They are checked against the two-pass definition by the tests.
 *
 * Layouts (row-major, D innermost):
 *   prefill  q [B, Hq, S, D], k/v [B, Hkv, S, D], o [B, Hq, S, D], lse [B, Hq, S]
 *   decode   q [B, Hq, D], k/v cache [B, Hkv, max_len, D], seqlens [B], o [B, Hq, D], lse [B, Hq]
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* One query row against n_keys keys (rows of k and v, kv_stride doubles apart).
 * visible[j] != 0 marks an unmasked key. Writes o[0..D) and *lse.
 * A row with no visible key gets o = 0 and lse = -infinity (no NaN). */
static void attend_row(const double *q, const double *k, const double *v, int64_t kv_stride,
                       int n_keys, const unsigned char *visible, int D, double scale,
                       double *s, double *o, double *lse)
{
    /* scores, masked entries set to -infinity */
    for (int j = 0; j < n_keys; ++j) {
        if (!visible[j]) { s[j] = -INFINITY; continue; }
        const double *kj = k + (int64_t)j * kv_stride;
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += q[d] * kj[d];
        s[j] = scale * dot;
    }
    /* pass 1: row max */
    double m = -INFINITY;
    for (int j = 0; j < n_keys; ++j) if (s[j] > m) m = s[j];
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    if (m == -INFINITY) { *lse = -INFINITY; return; }
    /* pass 2: exponentials and their sum */
    double l = 0.0;
    for (int j = 0; j < n_keys; ++j) { s[j] = exp(s[j] - m); l += s[j]; }
    /* P = e / l, O = P V */
    for (int j = 0; j < n_keys; ++j) {
        double p = s[j] / l;
        if (p == 0.0) continue;
        const double *vj = v + (int64_t)j * kv_stride;
        for (int d = 0; d < D; ++d) o[d] += p * vj[d];
    }
    *lse = m + log(l);
}

static void set_threads(int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Prefill rows listed in rows[] (flat ids r = (b*Hq + h)*S + i), or every row when rows is NULL.
 * o_out/lse_out are indexed by the position in rows[] (or by r when rows is NULL). */
int oracle_prefill_rows(const double *q, const double *k, const double *v,
                        int B, int S, int Hq, int Hkv, int D, double scale, int causal,
                        const int64_t *rows, int64_t n_rows, double *o_out, double *lse_out,
                        int nthreads)
{
    if (B < 0 || S < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || Hq % Hkv != 0) return 1;
    const int G = Hq / Hkv;
    const int64_t total = (int64_t)B * Hq * S;
    const int64_t n = rows ? n_rows : total;
    set_threads(nthreads);
    int bad = 0;
#pragma omp parallel reduction(| : bad)
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(S > 0 ? S : 1));
        unsigned char *vis = (unsigned char *)malloc((size_t)(S > 0 ? S : 1));
        if (!s || !vis) bad = 1;
#pragma omp for schedule(dynamic, 8)
        for (int64_t t = 0; t < n; ++t) {
            if (!s || !vis) continue;
            const int64_t r = rows ? rows[t] : t;
            if (r < 0 || r >= total) { bad = 1; continue; }
            const int i = (int)(r % S);
            const int h = (int)((r / S) % Hq);
            const int b = (int)(r / ((int64_t)S * Hq));
            const int g = h / G; /* contiguous query-head groups share one kv head */
            for (int j = 0; j < S; ++j) vis[j] = causal ? (j <= i) : 1;
            const double *qi = q + r * D;
            const double *kb = k + ((int64_t)b * Hkv + g) * S * D;
            const double *vb = v + ((int64_t)b * Hkv + g) * S * D;
            attend_row(qi, kb, vb, D, S, vis, D, scale, s, o_out + t * D, lse_out + t);
        }
        free(s);
        free(vis);
    }
    return bad;
}

int oracle_prefill(const double *q, const double *k, const double *v, double *o, double *lse,
                   int B, int S, int Hq, int Hkv, int D, double scale, int causal, int nthreads)
{
    return oracle_prefill_rows(q, k, v, B, S, Hq, Hkv, D, scale, causal, NULL, 0, o, lse, nthreads);
}

/* Decode: one query per (b, h) against the first seqlens[b] rows of the cache.
 * The cache position of the newest token is seqlens[b]-1 (it was written before attention). */
int oracle_decode(const double *q, const double *kc, const double *vc, const int32_t *seqlens,
                  double *o, double *lse, int B, int Hq, int Hkv, int D, int max_len,
                  double scale, int nthreads)
{
    if (B < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || max_len < 0 || Hq % Hkv != 0) return 1;
    for (int b = 0; b < B; ++b)
        if (seqlens[b] < 0 || seqlens[b] > max_len) return 1;
    const int G = Hq / Hkv;
    set_threads(nthreads);
    int bad = 0;
#pragma omp parallel reduction(| : bad)
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(max_len > 0 ? max_len : 1));
        unsigned char *vis = (unsigned char *)malloc((size_t)(max_len > 0 ? max_len : 1));
        if (!s || !vis) bad = 1;
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < (int64_t)B * Hq; ++r) {
            if (!s || !vis) continue;
            const int b = (int)(r / Hq), h = (int)(r % Hq), g = h / G;
            const int L = seqlens[b];
            for (int j = 0; j < L; ++j) vis[j] = 1;
            const double *kb = kc + ((int64_t)b * Hkv + g) * max_len * D;
            const double *vb = vc + ((int64_t)b * Hkv + g) * max_len * D;
            attend_row(q + r * D, kb, vb, D, L, vis, D, scale, s, o + r * D, lse + r);
        }
        free(s);
        free(vis);
    }
    return bad;
}

/* A chunk of Sq new queries against a KV cache: query i of sequence b sits at position
 * p = L_b - Sq + i (the chunk is the last Sq tokens, already written to the cache), sees keys
 * j < L_b, and with the causal mask only j <= p. Queries at p < 0 see nothing (O = 0, LSE = -inf).
 * With Sq = L_b this is prefill; with Sq = 1 it is decode.
 *   q [B, Hq, Sq, D], k/v cache [B, Hkv, max_len, D], seqlens [B], o [B, Hq, Sq, D], lse [B, Hq, Sq]
 * ("Hand-written Triton decoder", section 1.4: speculative decoding and beam search reuse the
 * same attention with several new tokens; "Attention three-op fusion", section 4.3: the causal
 * mask as -infinity.) */
int oracle_chunk(const double *q, const double *kc, const double *vc, const int32_t *seqlens,
                 double *o, double *lse, int B, int Sq, int Hq, int Hkv, int D, int max_len,
                 double scale, int causal, int nthreads)
{
    if (B < 0 || Sq < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || max_len < 0 || Hq % Hkv != 0) return 1;
    for (int b = 0; b < B; ++b)
        if (seqlens[b] < 0 || seqlens[b] > max_len) return 1;
    const int G = Hq / Hkv;
    set_threads(nthreads);
    int bad = 0;
#pragma omp parallel reduction(| : bad)
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(max_len > 0 ? max_len : 1));
        unsigned char *vis = (unsigned char *)malloc((size_t)(max_len > 0 ? max_len : 1));
        if (!s || !vis) bad = 1;
#pragma omp for schedule(dynamic, 4)
        for (int64_t r = 0; r < (int64_t)B * Hq * Sq; ++r) {
            if (!s || !vis) continue;
            const int i = (int)(r % Sq);
            const int h = (int)((r / Sq) % Hq);
            const int b = (int)(r / ((int64_t)Sq * Hq));
            const int g = h / G;
            const int L = seqlens[b];
            const long long p = (long long)L - Sq + i;
            for (int j = 0; j < L; ++j) vis[j] = causal ? ((long long)j <= p) : 1;
            const double *kb = kc + ((int64_t)b * Hkv + g) * max_len * D;
            const double *vb = vc + ((int64_t)b * Hkv + g) * max_len * D;
            attend_row(q + r * D, kb, vb, D, L, vis, D, scale, s, o + r * D, lse + r);
        }
        free(s);
        free(vis);
    }
    return bad;
}

/* Batched prefill of sequences padded to S tokens: sequence b holds seqlens[b] valid tokens at
 * positions 0 .. seqlens[b]-1. Row i < L_b sees keys j < L_b (and j <= i when causal); padding
 * rows i >= L_b see nothing (O = 0, LSE = -inf). Layouts as oracle_prefill.
 * ("Attention three-op fusion", section 4.3: padding positions get score -infinity.) */
int oracle_prefill_varlen(const double *q, const double *k, const double *v, const int32_t *seqlens,
                          double *o, double *lse, int B, int S, int Hq, int Hkv, int D,
                          double scale, int causal, int nthreads)
{
    if (B < 0 || S < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || Hq % Hkv != 0) return 1;
    for (int b = 0; b < B; ++b)
        if (seqlens[b] < 0 || seqlens[b] > S) return 1;
    const int G = Hq / Hkv;
    set_threads(nthreads);
    int bad = 0;
#pragma omp parallel reduction(| : bad)
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(S > 0 ? S : 1));
        unsigned char *vis = (unsigned char *)malloc((size_t)(S > 0 ? S : 1));
        if (!s || !vis) bad = 1;
#pragma omp for schedule(dynamic, 8)
        for (int64_t r = 0; r < (int64_t)B * Hq * S; ++r) {
            if (!s || !vis) continue;
            const int i = (int)(r % S);
            const int h = (int)((r / S) % Hq);
            const int b = (int)(r / ((int64_t)S * Hq));
            const int g = h / G;
            const int L = seqlens[b];
            for (int j = 0; j < L; ++j) vis[j] = (i < L) && (causal ? (j <= i) : 1);
            const double *kb = k + ((int64_t)b * Hkv + g) * S * D;
            const double *vb = v + ((int64_t)b * Hkv + g) * S * D;
            attend_row(q + r * D, kb, vb, D, L, vis, D, scale, s, o + r * D, lse + r);
        }
        free(s);
        free(vis);
    }
    return bad;
}

/* Rotary position embedding, rotate-half form, on n rows of D values (D even): with
 * x = [x1 | x2] (halves of D/2), out = [x1*cos - x2*sin | x1*sin + x2*cos], cos and sin given per
 * row as tables of D/2 values ("triton-optimization" skill, section 3.4: RoPE on the two halves
 * of each head with precomputed cos/sin tables; "Hand-written Triton decoder", section 1.2: RoPE
 * computed in floating point while loading q and k). */
void oracle_rope_rows(const double *x, const double *cosv, const double *sinv, double *out,
                      int64_t n, int D)
{
    const int H = D / 2;
    for (int64_t r = 0; r < n; ++r) {
        const double *xr = x + r * D;
        const double *c = cosv + r * H;
        const double *sn = sinv + r * H;
        double *o = out + r * D;
        for (int d = 0; d < H; ++d) {
            o[d] = xr[d] * c[d] - xr[d + H] * sn[d];
            o[d + H] = xr[d] * sn[d] + xr[d + H] * c[d];
        }
    }
}

/* ---- the method: online softmax over key blocks, and the merge of block partials ---- */

/* Partial state of one query row over n keys (one block): m = max score, l = sum of
 * exp(s - m), o_un = sum of exp(s - m) v (not divided by l). Empty block: m = -inf, l = 0. */
void oracle_row_partial(const double *q, const double *k, const double *v, int n, int D,
                        double scale, double *m_out, double *l_out, double *o_un)
{
    double m = -INFINITY;
    double *s = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    for (int j = 0; j < n; ++j) {
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += q[d] * k[(int64_t)j * D + d];
        s[j] = scale * dot;
        if (s[j] > m) m = s[j];
    }
    double l = 0.0;
    for (int d = 0; d < D; ++d) o_un[d] = 0.0;
    if (m != -INFINITY) {
        for (int j = 0; j < n; ++j) {
            double e = exp(s[j] - m);
            l += e;
            for (int d = 0; d < D; ++d) o_un[d] += e * v[(int64_t)j * D + d];
        }
    }
    free(s);
    *m_out = m;
    *l_out = l;
}

/* Merge nb partial states (m[i], l[i], o_un[i*D..]) of one row, in the order given:
 *   M = max_i m_i;  L = sum_i l_i exp(m_i - M);  O = sum_i exp(m_i - M) o_un_i / L;
 *   lse = M + log L.  All blocks empty: O = 0, lse = -inf. */
void oracle_merge(const double *m, const double *l, const double *o_un, int nb, int D,
                  double *o, double *lse)
{
    double M = -INFINITY;
    for (int i = 0; i < nb; ++i) if (m[i] > M) M = m[i];
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    if (M == -INFINITY) { *lse = -INFINITY; return; }
    double L = 0.0;
    for (int i = 0; i < nb; ++i) {
        if (m[i] == -INFINITY) continue;
        double w = exp(m[i] - M);
        L += l[i] * w;
        for (int d = 0; d < D; ++d) o[d] += w * o_un[(int64_t)i * D + d];
    }
    for (int d = 0; d < D; ++d) o[d] /= L;
    *lse = M + log(L);
}

/* The recurrence itself, one row, keys visited in blocks of `block` in index order:
 *   m_new = max(m, max(s_blk)); c = exp(m - m_new);
 *   l = l c + sum exp(s_blk - m_new);  acc = acc c + sum exp(s_blk - m_new) v;
 * and at the end O = acc / l, lse = m + log l. Starts from m = -inf, l = 0, acc = 0. */
void oracle_online_row(const double *q, const double *k, const double *v, int n, int D,
                       double scale, int block, double *o, double *lse)
{
    double m = -INFINITY, l = 0.0;
    double *acc = (double *)calloc((size_t)(D > 0 ? D : 1), sizeof(double));
    double *s = (double *)malloc(sizeof(double) * (size_t)(block > 0 ? block : 1));
    if (block <= 0) block = 1;
    for (int j0 = 0; j0 < n; j0 += block) {
        const int nb = (n - j0 < block) ? (n - j0) : block;
        double mb = -INFINITY;
        for (int j = 0; j < nb; ++j) {
            double dot = 0.0;
            for (int d = 0; d < D; ++d) dot += q[d] * k[(int64_t)(j0 + j) * D + d];
            s[j] = scale * dot;
            if (s[j] > mb) mb = s[j];
        }
        const double m_new = (mb > m) ? mb : m;
        const double c = (m == -INFINITY) ? 0.0 : exp(m - m_new);
        l *= c;
        for (int d = 0; d < D; ++d) acc[d] *= c;
        for (int j = 0; j < nb; ++j) {
            const double e = exp(s[j] - m_new);
            l += e;
            for (int d = 0; d < D; ++d) acc[d] += e * v[(int64_t)(j0 + j) * D + d];
        }
        m = m_new;
    }
    for (int d = 0; d < D; ++d) o[d] = (l > 0.0) ? acc[d] / l : 0.0;
    *lse = (l > 0.0) ? m + log(l) : -INFINITY;
    free(acc);
    free(s);
}
