/*
 * pkv_oracle.c -- CPU oracle for paged decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously correct
 * statement of what the decode step computes.  It is compiled and called only
 * by the tests, by the package's smoke check and by the benchmark's CPU
 * baseline leg.  It shares no code, header or constant with the CUDA library
 * and must never be linked into it.
 *
 * What it computes (decode attention for one new token per sequence):
 *   "KV cache & PagedAttention -- vi sao chatbot AI ton bo nho" (aiwiki.vn),
 *   second paragraph: the query of the current position interacts with the
 *   keys of every position it may see, and the resulting attention weights
 *   are used to combine the values.  Third paragraph: those keys and values
 *   come from the cache instead of being recomputed.
 *   "PagedAttention (vLLM) -- Virtual memory cho AI", section "Y tuong cot
 *   loi": attention does not depend on where a token's K/V sit physically.
 *   Paging therefore changes only addresses, and the oracle works on plain
 *   contiguous per-sequence K/V with no block table at all.
 *
 * For sequence s, query head h, kv head g = h / (Hq / Hkv)  (consecutive
 * grouping of query heads onto the reduced set of KV heads):
 *   score_t = scale * sum_d q[s,h,d] * K_s[t,g,d]          t = 0 .. L_s-1
 *   p_t     = exp(score_t - max_u score_u) / sum_u exp(score_u - max_u score_u)
 *   out[s,h,d] = sum_t p_t * V_s[t,g,d]
 * An empty context (L_s == 0) yields an all-zero output row.
 *
 * Everything is IEEE double precision, step for step as written above.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Number of threads the parallel loop below will use. */
int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* One (sequence, query head) pair.  k_s / v_s point at row 0 of the
 * sequence's contiguous [L, Hkv, D] slab.  Returns |sum_t p_t - 1|. */
static double attend_one(const double *q_sh, const double *k_s, const double *v_s,
                         int64_t L, int64_t Hkv, int64_t D, int64_t g, double scale,
                         double *out_sh, double *scores)
{
    int64_t t, d;
    double m, denom, wsum;

    for (d = 0; d < D; ++d) out_sh[d] = 0.0;
    if (L <= 0) return 0.0;

    /* scores: scaled dot products of the query with every cached key */
    for (t = 0; t < L; ++t) {
        const double *k_t = k_s + (t * Hkv + g) * D;
        double acc = 0.0;
        for (d = 0; d < D; ++d) acc += q_sh[d] * k_t[d];
        scores[t] = scale * acc;
    }

    /* softmax over the L scores, shifted by their maximum */
    m = scores[0];
    for (t = 1; t < L; ++t)
        if (scores[t] > m) m = scores[t];
    denom = 0.0;
    for (t = 0; t < L; ++t) {
        scores[t] = exp(scores[t] - m);
        denom += scores[t];
    }
    wsum = 0.0;
    for (t = 0; t < L; ++t) {
        scores[t] = scores[t] / denom; /* p_t */
        wsum += scores[t];
    }

    /* weighted sum of the cached values */
    for (t = 0; t < L; ++t) {
        const double *v_t = v_s + (t * Hkv + g) * D;
        const double p = scores[t];
        for (d = 0; d < D; ++d) out_sh[d] += p * v_t[d];
    }
    return fabs(wsum - 1.0);
}

/*
 * q        [S, Hq, D]
 * k, v     [sum_s L_s, Hkv, D]  sequences stored one after another;
 *          sequence s starts at row tok_start[s]
 * seq_lens [S]
 * out      [S, Hq, D]
 * wsum_err [S, Hq] or NULL: |sum of softmax weights - 1| per pair
 * Returns 0 on success, -1 on bad arguments or allocation failure.
 */
int oracle_decode_attention(const double *q, const double *k, const double *v,
                            const int64_t *tok_start, const int64_t *seq_lens,
                            int64_t S, int64_t Hq, int64_t Hkv, int64_t D, double scale,
                            double *out, double *wsum_err)
{
    int64_t s, maxL = 0;
    int failed = 0;

    if (S < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || Hq % Hkv != 0) return -1;
    for (s = 0; s < S; ++s) {
        if (seq_lens[s] < 0) return -1;
        if (seq_lens[s] > maxL) maxL = seq_lens[s];
    }

#pragma omp parallel reduction(|| : failed)
    {
        double *scores = (double *)malloc((size_t)(maxL > 0 ? maxL : 1) * sizeof(double));
        int64_t i;
        if (!scores) failed = 1;
#pragma omp for schedule(dynamic, 1)
        for (i = 0; i < S * Hq; ++i) {
            const int64_t si = i / Hq, h = i % Hq;
            const int64_t g = h / (Hq / Hkv);
            const double *k_s = k + tok_start[si] * Hkv * D;
            const double *v_s = v + tok_start[si] * Hkv * D;
            double err;
            if (!scores) continue;
            err = attend_one(q + i * D, k_s, v_s, seq_lens[si], Hkv, D, g, scale,
                             out + i * D, scores);
            if (wsum_err) wsum_err[i] = err;
        }
        free(scores);
    }
    return failed ? -1 : 0;
}
