/*
 * kvr_rsq_oracle.c -- plain, slow CPU oracle for the calibrated inner-product
 * reranker of the candidates (RSQ-IP).
 *
 * TEST INFRASTRUCTURE, like kvr_oracle.c: only the test suite, the package
 * smoke check and the benchmark's CPU legs load it; the CUDA library shares
 * nothing with it. Built with -O2 -ffp-contract=off: each fp32 operation below
 * is one IEEE round-to-nearest-even operation in the order written.
 *
 * Source: ParisKV, "Pipeline di Recupero Nativa su GPU in Due Stadi",
 * candidate reranking: each sub-space direction of a rotated key is coded
 * with 4 bits (a sign bit and 3 magnitude bits) from the Beta prior the
 * rotation induces; a per-key, per-sub-space scale w is fixed at prefill to
 * correct the quantisation misalignment; the score <k, q> is estimated as
 * ||q|| sum_b w_b <v_b, q~_b> from the dequantised directions v_b and the
 * rotated query q~, without reading the full-precision keys.
 *
 * Readings (the pages give neither levels nor the calibration):
 *   - 4 bits per coordinate of a sub-block direction u_b = z_b / ||z_b||
 *     (z = FWHT(D k), sub-blocks of m = 8): the sign bit is the analytic
 *     centroid's, the 3 magnitude bits pick one of 8 levels for |u_j|;
 *   - the prior: a coordinate of a uniformly random unit vector in R^m has
 *     u_j^2 ~ Beta(1/2, (m-1)/2); the 8 magnitude bins have equal probability
 *     under it and each level is the conditional mean of |u_j| in its bin;
 *   - calibration: w_b = ||z_b|| / <u_b, v_b> with v_b the dequantised
 *     direction (signs and levels), so the estimate is exact when v_b is
 *     parallel to u_b; in fp32: s_b = sum_j z_j^2, c_b = sum_j |z_j| lev_j,
 *     w_b = bf16(s_b / c_b) (0 for an all-zero sub-block);
 *   - the estimate, ranking-equivalent to q_bar . k: sum_b w_b <v_b, zq_b>
 *     with zq = FWHT(D q_bar), in a canonical fp32 order (fma chain over the
 *     8 coordinates of a block from +0, times w_b, then butterfly sums over
 *     16 block slots with spans 8, 4, 2, 1, empty slots +0).
 *
 * Record of one key (6 * d/8 bytes): d/8 little-endian 32-bit block words,
 * nibble j (bits 4j .. 4j+3) of word b holding coordinate 8b + j as
 * magnitude | sign << 3, then d/8 bf16 scales w_b.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define RSQ_M 8
#define RSQ_MAXD 128
#define RSQ_LEVELS 8

/* from kvr_oracle.c / kvr_tiers_oracle.c (the same oracle library) */
void orc_fwht_f32(float *x, int d);
void orc_group_mean(const float *q, int G, int d, float *qbar);
int orc_encode(const float *x, int64_t n, int d, const int8_t *sgn, uint8_t *codes);
void orc_coarse_scores(const uint8_t *codes, int64_t n, int nb, const uint8_t *qcode,
                       const int32_t *lut, int32_t *score);
int64_t orc_top_by_int(const int32_t *score, int64_t n, int64_t c, int64_t *out);
int64_t orc_top_by_float(const float *score, const int64_t *index, int64_t n, int64_t c,
                         int64_t *out);
float orc_bf16_round(float x);

/* ------------------------------------------------------------------------ */
/* The magnitude quantiser from the Beta prior.                              */
/* ------------------------------------------------------------------------ */

/* Density of t = |u_j| on [0, 1] for a uniformly random unit vector in R^m:
   u_j^2 ~ Beta(1/2, (m-1)/2) gives f(t) = 2 (1 - t^2)^((m-3)/2) / B(1/2, (m-1)/2). */
static double mag_density(double t, int m)
{
    const double a = 0.5, b = 0.5 * (m - 1);
    const double lbeta = lgamma(a) + lgamma(b) - lgamma(a + b);
    if (t >= 1.0)
        return 0.0;
    return 2.0 * pow(1.0 - t * t, b - 1.0) * exp(-lbeta);
}

/* integral of t^power f(t) over [lo, hi], composite Simpson */
static double mag_integral(double lo, double hi, int m, int power)
{
    const int n = 20000;
    const double h = (hi - lo) / n;
    double s = 0.0;
    for (int i = 0; i <= n; i++) {
        const double t = lo + h * i;
        const double g = (power ? t : 1.0) * mag_density(t, m);
        s += g * ((i == 0 || i == n) ? 1.0 : ((i & 1) ? 4.0 : 2.0));
    }
    return s * h / 3.0;
}

/*
 * Edges bound[0..8] (bound[0] = 0, bound[8] = 1) of the 8 equal-probability
 * bins of |u_j| and the conditional mean level[0..7] of each bin, in fp64.
 * Returns -1 for m < 3 (the density is then unbounded at 1).
 */
int orc_rsq_table(int m, double *bound, double *level)
{
    if (m < 3)
        return -1;
    bound[0] = 0.0;
    bound[RSQ_LEVELS] = 1.0;
    for (int i = 1; i < RSQ_LEVELS; i++) {
        const double target = (double)i / RSQ_LEVELS;
        double lo = bound[i - 1], hi = 1.0;
        const double base = mag_integral(0.0, bound[i - 1], m, 0);  /* CDF at the previous edge */
        for (int it = 0; it < 60; it++) {
            const double mid = 0.5 * (lo + hi);
            if (base + mag_integral(bound[i - 1], mid, m, 0) < target)
                lo = mid;
            else
                hi = mid;
        }
        bound[i] = 0.5 * (lo + hi);
    }
    for (int i = 0; i < RSQ_LEVELS; i++)
        level[i] = mag_integral(bound[i], bound[i + 1], m, 1) * RSQ_LEVELS;
    return 0;
}

/* The fp32 tables the codes are decided with: bsq[i] = fl(bound[i]^2)
   (bsq[0] = 0) and lev[i] = fl(level[i]). */
int orc_rsq_float_tables(int m, float *bsq, float *lev)
{
    double bound[RSQ_LEVELS + 1], level[RSQ_LEVELS];
    if (orc_rsq_table(m, bound, level))
        return -1;
    for (int i = 0; i < RSQ_LEVELS; i++) {
        bsq[i] = (float)(bound[i] * bound[i]);
        lev[i] = (float)level[i];
    }
    return 0;
}

/* The m = 8 fp32 tables, computed once (the oracle is single-threaded). */
static const float *rsq_tables8(int which)
{
    static float bsq[RSQ_LEVELS], lev[RSQ_LEVELS];
    static int done = 0;
    if (!done) {
        orc_rsq_float_tables(RSQ_M, bsq, lev);
        done = 1;
    }
    return which ? lev : bsq;
}

/* ------------------------------------------------------------------------ */
/* Records and the estimate.                                                 */
/* ------------------------------------------------------------------------ */

int64_t orc_rsq_record_bytes(int d) { return 6 * (int64_t)(d / RSQ_M); }

static uint16_t bf16_bits(float x)
{
    const float r = orc_bf16_round(x);
    uint32_t u;
    memcpy(&u, &r, 4);
    return (uint16_t)(u >> 16);
}

static float bf16_value(uint16_t h)
{
    const uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/*
 * Records rec[n][6 d/8] of the rows x[n][d]: z = FWHT(D x) (the codes'
 * rotation), then per block b of 8 coordinates:
 *   s = fma chain of z_j * z_j over j ascending from +0;
 *   mag_j = #{i in 1..7 : fl(z_j * z_j) >= fl(bsq[i] * s)};
 *   c = fma chain of |z_j| * lev[mag_j] over j ascending from +0;
 *   w = bf16(s / c), 0 when c == 0 (an all-zero sub-block: every
 *   coordinate lands in the top bin, 0 >= edge * 0, and weighs nothing).
 */
int orc_rsq_encode(const float *x, int64_t n, int d, const int8_t *sgn, uint8_t *rec)
{
    if (d % RSQ_M != 0 || d > RSQ_MAXD)
        return -1;
    const float *bsq = rsq_tables8(0), *lev = rsq_tables8(1);
    const int nb = d / RSQ_M;
    const int64_t rb = orc_rsq_record_bytes(d);
    float z[RSQ_MAXD];
    for (int64_t r = 0; r < n; r++) {
        const float *xr = x + r * (int64_t)d;
        uint8_t *out = rec + r * rb;
        for (int j = 0; j < d; j++)
            z[j] = xr[j] * (float)sgn[j];
        orc_fwht_f32(z, d);
        for (int b = 0; b < nb; b++) {
            const float *zb = z + b * RSQ_M;
            float s = 0.0f;
            for (int j = 0; j < RSQ_M; j++)
                s = fmaf(zb[j], zb[j], s);
            uint32_t word = 0;
            float c = 0.0f;
            for (int j = 0; j < RSQ_M; j++) {
                const float a = zb[j] * zb[j];
                int mag = 0;
                for (int i = 1; i < RSQ_LEVELS; i++)
                    if (a >= bsq[i] * s)
                        mag = i;
                const uint32_t neg = zb[j] < 0.0f ? 1u : 0u;
                word |= ((uint32_t)mag | neg << 3) << (4 * j);
                c = fmaf(fabsf(zb[j]), lev[mag], c);
            }
            const float w = (c > 0.0f) ? s / c : 0.0f;
            const uint16_t wb = bf16_bits(w);
            for (int i = 0; i < 4; i++)
                out[4 * b + i] = (uint8_t)(word >> (8 * i));
            out[4 * nb + 2 * b] = (uint8_t)(wb & 0xff);
            out[4 * nb + 2 * b + 1] = (uint8_t)(wb >> 8);
        }
    }
    return 0;
}

/* The estimate of one record against the rotated query zq[d] (canonical order above). */
float orc_rsq_score(const uint8_t *rec, const float *zq, int d)
{
    const float *lev = rsq_tables8(1);
    const int nb = d / RSQ_M;
    float t[16];
    for (int b = 0; b < 16; b++) {
        t[b] = 0.0f;
        if (b >= nb)
            continue;
        const uint32_t word = (uint32_t)rec[4 * b] | (uint32_t)rec[4 * b + 1] << 8 |
                              (uint32_t)rec[4 * b + 2] << 16 | (uint32_t)rec[4 * b + 3] << 24;
        float e = 0.0f;
        for (int j = 0; j < RSQ_M; j++) {
            const uint32_t nib = (word >> (4 * j)) & 15u;
            const float v = (nib & 8u) ? -lev[nib & 7u] : lev[nib & 7u];
            e = fmaf(v, zq[b * RSQ_M + j], e);
        }
        const uint16_t wb = (uint16_t)(rec[4 * nb + 2 * b] | (rec[4 * nb + 2 * b + 1] << 8));
        t[b] = bf16_value(wb) * e;
    }
    for (int span = 8; span >= 1; span >>= 1)
        for (int b = 0; b < span; b++)
            t[b] = t[b] + t[b + span];
    return t[0];
}

/*
 * Selection of one unit with the RSQ-IP estimate in place of the exact
 * rescoring: the coarse stage and the candidate set are those of
 * orc_select_unit; the candidates are then ranked by (estimate desc, index
 * asc) and the first k' kept, emitted ascending. rec[N][6 d/8] are the
 * pool keys' records. cand / cand_S (optional) receive the candidates and
 * their estimates. Returns 0, or -1 on a NaN estimate or a bad shape.
 */
int orc_select_unit_rsq(const float *q, int G, const uint8_t *codes, const uint8_t *rec,
                        int64_t N, int d, const int8_t *sgn, int64_t C, int64_t k, int64_t W,
                        const int32_t *lut, int32_t *out_idx, int32_t *out_count, int32_t *cand,
                        float *cand_S)
{
    if (d % 16 != 0 || d > RSQ_MAXD || G < 1)
        return -1;
    const int nb = d / RSQ_M;
    const int64_t rb = orc_rsq_record_bytes(d);
    int64_t pool = N - W;
    if (pool < 0)
        pool = 0;
    for (int64_t j = 0; j < k; j++)
        out_idx[j] = -1;
    *out_count = 0;
    float qbar[RSQ_MAXD], zq[RSQ_MAXD];
    uint8_t qcode[RSQ_MAXD / RSQ_M];
    orc_group_mean(q, G, d, qbar);
    orc_encode(qbar, 1, d, sgn, qcode);
    for (int j = 0; j < d; j++)
        zq[j] = qbar[j] * (float)sgn[j];
    orc_fwht_f32(zq, d);
    if (pool == 0)
        return 0;
    int32_t *s = (int32_t *)malloc(sizeof(int32_t) * (size_t)pool);
    orc_coarse_scores(codes, pool, nb, qcode, lut, s);
    int64_t *cset = (int64_t *)malloc(sizeof(int64_t) * (size_t)(C > 0 ? C : 1));
    const int64_t nc = orc_top_by_int(s, pool, C, cset);
    free(s);
    float *S = (float *)malloc(sizeof(float) * (size_t)(nc > 0 ? nc : 1));
    for (int64_t j = 0; j < nc; j++) {
        S[j] = orc_rsq_score(rec + cset[j] * rb, zq, d);
        if (cand)
            cand[j] = (int32_t)cset[j];
        if (cand_S)
            cand_S[j] = S[j];
    }
    int64_t *top = (int64_t *)malloc(sizeof(int64_t) * (size_t)(k > 0 ? k : 1));
    int64_t nk = orc_top_by_float(S, cset, nc, k, top);
    int rc = 0;
    if (nk < 0) {
        rc = -1;
        nk = 0;
    }
    for (int64_t j = 0; j < nk; j++)
        out_idx[j] = (int32_t)top[j];
    *out_count = (int32_t)nk;
    free(top);
    free(S);
    free(cset);
    return rc;
}
