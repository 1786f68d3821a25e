/*
 * kvr_regions_oracle.c -- plain, slow CPU oracle of the four cache regions:
 * sink, retrieval, local and update buffer.
 *
 * TEST INFRASTRUCTURE, like kvr_oracle.c: only the test suite, the package
 * smoke check and the benchmark's CPU legs load it; the CUDA library shares
 * nothing with it. Built with -O2 -ffp-contract=off.
 *
 * Source: ParisKV, "Meccanismo di Aggiornamento a Finestra Scorrevole": for
 * unbounded generation the cache is kept in four regions -- Sink (the first
 * tokens, kept on the GPU), Local (the recent tokens, on the GPU), Retrieval
 * (the older tokens, searched and offloaded) and an Update Buffer. When the
 * buffer fills up, the oldest local tokens move to Retrieval and the buffer's
 * tokens become Local, so the retrieval metadata stays current while both the
 * recent context and the long-range history stay reachable.
 *
 * Readings (the pages give no sizes and no positions):
 *   - regions by position, for a unit of length N: Sink [0, S), Retrieval
 *     [S, R), Local followed by the buffer [R, N); the attention reads the
 *     Sink, the top-k of Retrieval and all of [R, N);
 *   - set-up: R = max(min(S, N), N - L) (Local holds the L newest tokens and
 *     the buffer is empty);
 *   - after appends: the sink first takes the positions below S (R =
 *     max(R, min(S, N))); then while N - R >= L + U, R += U (the buffer holds
 *     N - R - L tokens; when it reaches U, the U oldest local tokens move to
 *     Retrieval and the buffer becomes the newest part of Local);
 *   - clamps for short units: S' = min(S, N), R' = min(max(R, S'), N).
 * Selection over [S', R') follows the steps of orc_select_unit (coarse
 * scores, first C' by (score desc, index asc), exact q_bar . k, first k' by
 * (score desc, index asc), output ascending); only the pool's lower end
 * moves from 0 to S'.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define RG_M 8
#define RG_MAXD 128

/* from kvr_oracle.c / kvr_rsq_oracle.c (the same oracle library) */
void orc_fwht_f32(float *x, int d);
void orc_group_mean(const float *q, int G, int d, float *qbar);
int orc_encode(const float *x, int64_t n, int d, const int8_t *sgn, uint8_t *codes);
void orc_coarse_scores(const uint8_t *codes, int64_t n, int nb, const uint8_t *qcode,
                       const int32_t *lut, int32_t *score);
int64_t orc_top_by_int(const int32_t *score, int64_t n, int64_t c, int64_t *out);
int64_t orc_top_by_float(const float *score, const int64_t *index, int64_t n, int64_t c,
                         int64_t *out);
float orc_exact_score(const float *qbar, const float *k, int d);
int64_t orc_rsq_record_bytes(int d);
float orc_rsq_score(const uint8_t *rec, const float *zq, int d);

/* ------------------------------------------------------------------------ */
/* Region boundaries.                                                        */
/* ------------------------------------------------------------------------ */

int64_t orc_region_init(int64_t N, int64_t S, int64_t L)
{
    const int64_t s_eff = S < N ? S : N;
    const int64_t r = N - L;
    return r > s_eff ? r : s_eff;
}

/* Retrieval end after appends up to length N (U >= 1). */
int64_t orc_region_advance(int64_t N, int64_t R, int64_t S, int64_t L, int64_t U)
{
    const int64_t s_eff = S < N ? S : N;
    if (R < s_eff)
        R = s_eff;
    while (N - R >= L + U)
        R += U;
    return R;
}

static void clamp_regions(int64_t N, int64_t S, int64_t R, int64_t *lo, int64_t *hi)
{
    int64_t s = S < N ? S : N;
    if (s < 0)
        s = 0;
    int64_t r = R < s ? s : R;
    if (r > N)
        r = N;
    *lo = s;
    *hi = r;
}

/* ------------------------------------------------------------------------ */
/* Selection over the retrieval region.                                      */
/* ------------------------------------------------------------------------ */

/*
 * As orc_select_unit, with the pool [S', R') instead of [0, N - W). rec is
 * NULL for exact rescoring, else the units' reranker records (the estimate
 * replaces q_bar . k). cand / cand_S (optional, C' entries) and coarse
 * (optional, one per pool key from S') as in orc_select_unit.
 */
int orc_select_unit_regions(const float *q, int G, const float *K, const uint8_t *codes,
                            const uint8_t *rec, int64_t N, int d, const int8_t *sgn, int64_t C,
                            int64_t k, int64_t S, int64_t R, const int32_t *lut,
                            int32_t *out_idx, int32_t *out_count, int32_t *cand, float *cand_S,
                            int32_t *coarse)
{
    if (d % 16 != 0 || d > RG_MAXD || G < 1)
        return -1;
    const int nb = d / RG_M;
    int64_t lo, hi;
    clamp_regions(N, S, R, &lo, &hi);
    const int64_t pool = hi - lo;
    for (int64_t j = 0; j < k; j++)
        out_idx[j] = -1;
    *out_count = 0;

    float qbar[RG_MAXD], zq[RG_MAXD];
    uint8_t qcode[RG_MAXD / RG_M];
    orc_group_mean(q, G, d, qbar);
    orc_encode(qbar, 1, d, sgn, qcode);
    for (int j = 0; j < d; j++)
        zq[j] = qbar[j] * (float)sgn[j];
    orc_fwht_f32(zq, d);
    if (pool == 0)
        return 0;

    int32_t *s = (int32_t *)malloc(sizeof(int32_t) * (size_t)pool);
    orc_coarse_scores(codes + lo * nb, pool, nb, qcode, lut, s);
    if (coarse)
        memcpy(coarse, s, sizeof(int32_t) * (size_t)pool);
    int64_t *cset = (int64_t *)malloc(sizeof(int64_t) * (size_t)(C > 0 ? C : 1));
    const int64_t nc = orc_top_by_int(s, pool, C, cset);
    free(s);
    for (int64_t j = 0; j < nc; j++)
        cset[j] += lo;  /* positions in the unit */

    float *Sc = (float *)malloc(sizeof(float) * (size_t)(nc > 0 ? nc : 1));
    const int64_t rb = orc_rsq_record_bytes(d);
    for (int64_t j = 0; j < nc; j++) {
        Sc[j] = rec ? orc_rsq_score(rec + cset[j] * rb, zq, d)
                    : orc_exact_score(qbar, K + cset[j] * (int64_t)d, d);
        if (cand)
            cand[j] = (int32_t)cset[j];
        if (cand_S)
            cand_S[j] = Sc[j];
    }
    int64_t *top = (int64_t *)malloc(sizeof(int64_t) * (size_t)(k > 0 ? k : 1));
    int64_t nk = orc_top_by_float(Sc, cset, nc, k, top);
    int rc = 0;
    if (nk < 0) {
        rc = -1;
        nk = 0;
    }
    for (int64_t j = 0; j < nk; j++)
        out_idx[j] = (int32_t)top[j];
    *out_count = (int32_t)nk;
    free(top);
    free(Sc);
    free(cset);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* Attention over sink, selected retrieval tokens, local and buffer.        */
/* ------------------------------------------------------------------------ */

/*
 * Attention of the G query heads of one unit over T = [0, S') U idx U
 * [R', N), in fp64 from the fp32 values (as orc_attend_unit: two-pass
 * softmax of (q_h . k_t) * scale). Indices in idx must lie in [S', R');
 * returns -1 otherwise. An empty T gives zeros.
 */
int orc_attend_unit_regions(const float *q, int G, const float *K, const float *V, int64_t N,
                            int d, int64_t S, int64_t R, const int32_t *idx, int64_t count,
                            float scale, double *out)
{
    int64_t lo, hi;
    clamp_regions(N, S, R, &lo, &hi);
    for (int64_t j = 0; j < count; j++)
        if (idx[j] < lo || idx[j] >= hi)
            return -1;
    memset(out, 0, sizeof(double) * (size_t)G * (size_t)d);
    const int64_t nt = lo + count + (N - hi);
    if (nt == 0)
        return 0;
    int64_t *tok = (int64_t *)malloc(sizeof(int64_t) * (size_t)nt);
    int64_t n = 0;
    for (int64_t t = 0; t < lo; t++)
        tok[n++] = t;
    for (int64_t j = 0; j < count; j++)
        tok[n++] = idx[j];
    for (int64_t t = hi; t < N; t++)
        tok[n++] = t;
    double *s = (double *)malloc(sizeof(double) * (size_t)nt);
    for (int h = 0; h < G; h++) {
        const float *qh = q + (int64_t)h * d;
        double mx = -INFINITY;
        for (int64_t j = 0; j < nt; j++) {
            const float *kt = K + tok[j] * (int64_t)d;
            double acc = 0.0;
            for (int c = 0; c < d; c++)
                acc += (double)qh[c] * (double)kt[c];
            s[j] = acc * (double)scale;
            if (s[j] > mx)
                mx = s[j];
        }
        double den = 0.0;
        for (int64_t j = 0; j < nt; j++) {
            s[j] = exp(s[j] - mx);
            den += s[j];
        }
        double *oh = out + (int64_t)h * d;
        for (int64_t j = 0; j < nt; j++) {
            const float *vt = V + tok[j] * (int64_t)d;
            const double p = s[j] / den;
            for (int c = 0; c < d; c++)
                oh[c] += p * (double)vt[c];
        }
    }
    free(s);
    free(tok);
    return 0;
}
