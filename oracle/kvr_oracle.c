/*
 * kvr_oracle.c -- plain, slow CPU oracle for retrieval-based sparse decode
 * attention.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the package smoke check and the
 * benchmark's CPU-baseline / reference leg load this file's library. The CUDA
 * library neither links nor calls it, and the two share no source, header,
 * table or helper.
 *
 * Every function follows the method in the order the pages give it, one
 * (b, kv-head) unit at a time, with single-threaded loops and no blocking or
 * fusion. Floating point: compiled with -O2 -ffp-contract=off and no
 * fast-math, so every fp32 operation below is one IEEE-754 round-to-nearest-
 * even operation, evaluated in the order written. Where an fp32 result
 * decides an integer (a sign bit, a rank), the order written here is the
 * canonical order that the GPU path must reproduce; each function states the
 * reading of the pages that fixes its order.
 *
 * Sources (page title, section):
 *   [P-rot]   ParisKV, "Centroidi Analitici Robusti al Drift": l2
 *             normalisation, shared random orthogonal rotation (SRHT), fixed
 *             sign-pattern centroids +-1/sqrt(m) on the unit sphere.
 *   [P-pipe]  ParisKV, "Pipeline di Recupero Nativa su GPU in Due Stadi":
 *             split into B sub-blocks, nearest analytic centroid per
 *             sub-block, top-rho query centroids per sub-block, tiered votes
 *             summed into an integer coarse score, pruning to a candidate set.
 *   [P-prob]  ParisKV, "Problematica": attention over a top-k subset of past
 *             tokens only.
 *   [Q-meth]  QEvict, "Metodologia: QEvict": three tiers (full precision,
 *             recoverable low-bit INT2, evicted) over contiguous windows under
 *             a fixed memory budget.
 *   [Q-mech]  QEvict, "Meccanismi Chiave": window-level routing, cumulative
 *             attention scores, demotion / promotion, write-once quantisation
 *             ledger, GQA.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_MAX_D 128
#define ORC_M 8 /* sub-block width m: 8 dims per analytic-centroid sub-block */

/* ------------------------------------------------------------------------ */
/* Step 1 [P-rot]: the rotation.                                             */
/* ------------------------------------------------------------------------ */

/*
 * In-place fast Walsh-Hadamard transform in natural (Sylvester) order:
 * on return x = H_d x with H_d[i][j] = (-1)^popcount(i & j). Stages run with
 * the butterfly span h ascending 1, 2, 4, ..., d/2; each butterfly replaces
 * (x_i, x_{i+h}) by (x_i + x_{i+h}, x_i - x_{i+h}).
 */
void orc_fwht_f32(float *x, int d)
{
    for (int h = 1; h < d; h <<= 1) {
        for (int i = 0; i < d; i++) {
            if (i & h)
                continue;
            float a = x[i];
            float b = x[i + h];
            x[i] = a + b;
            x[i + h] = a - b;
        }
    }
}

/*
 * The SRHT of [P-rot] with its dimension equal to the head dimension: the
 * sampling step is the identity, so the rotation is R = (1/sqrt(d)) H_d D,
 * D = diag(sgn), sgn_j in {+1, -1}. Writes the rotated unit vector
 * y = R x / ||x||_2 in fp64 (used by the tests of the rotation; the codes
 * below need only signs, see orc_encode).
 */
int orc_srht_unit_f64(const float *x, int d, const int8_t *sgn, double *y)
{
    double nrm = 0.0;
    for (int j = 0; j < d; j++)
        nrm += (double)x[j] * (double)x[j];
    nrm = sqrt(nrm);
    for (int i = 0; i < d; i++) {
        double acc = 0.0;
        for (int j = 0; j < d; j++) {
            int neg = __builtin_popcount((unsigned)(i & j)) & 1;
            double hij = neg ? -1.0 : 1.0;
            acc += hij * (double)sgn[j] * (double)x[j];
        }
        y[i] = (nrm > 0.0) ? acc / (sqrt((double)d) * nrm) : 0.0;
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Step 2 [P-rot], [P-pipe]: nearest analytic centroid = sign code.          */
/* ------------------------------------------------------------------------ */

/*
 * Code of n vectors x[n][d] (fp32 values; bf16 inputs are widened exactly).
 * Per vector: z = fl32 FWHT(D x). The rotated unit vector is a positive
 * multiple of z (by 1/(sqrt(d)||x||)), and a positive scale changes neither
 * the sign of a coordinate nor which centroid is nearest, so the code is read
 * off z directly. Sub-block b covers dims 8b..8b+7; its nearest centroid in
 * {+-1/sqrt(8)}^8 is the one whose signs agree with z (ties at z_j == 0 go to
 * the '+' centroid, the lowest byte value). Byte b of the code has bit j set
 * iff z[8b + j] < 0. codes is [n][d/8].
 */
int orc_encode(const float *x, int64_t n, int d, const int8_t *sgn, uint8_t *codes)
{
    if (d % ORC_M != 0 || d > ORC_MAX_D)
        return -1;
    float z[ORC_MAX_D];
    int nb = d / ORC_M;
    for (int64_t r = 0; r < n; r++) {
        const float *xr = x + r * (int64_t)d;
        for (int j = 0; j < d; j++)
            z[j] = xr[j] * (float)sgn[j];
        orc_fwht_f32(z, d);
        for (int b = 0; b < nb; b++) {
            unsigned byte = 0;
            for (int j = 0; j < ORC_M; j++)
                if (z[b * ORC_M + j] < 0.0f)
                    byte |= 1u << j;
            codes[r * nb + b] = (uint8_t)byte;
        }
    }
    return 0;
}

/*
 * The query of a KV head: the mean of its G query heads q[G][d], summed left
 * to right in fp32 and divided by G (IEEE division). One selection serves the
 * whole GQA group; q_bar . k is the group's summed logit divided by G.
 */
void orc_group_mean(const float *q, int G, int d, float *qbar)
{
    for (int j = 0; j < d; j++) {
        float acc = q[j];
        for (int g = 1; g < G; g++)
            acc = acc + q[(int64_t)g * d + j];
        qbar[j] = acc / (float)G;
    }
}

/* ------------------------------------------------------------------------ */
/* Step 3 [P-pipe]: coarse collision votes.                                  */
/* ------------------------------------------------------------------------ */

static int popcount8(unsigned v)
{
    int c = 0;
    for (int j = 0; j < 8; j++)
        c += (v >> j) & 1u;
    return c;
}

/*
 * Coarse score of n keys against one query code: per sub-block b the query
 * votes for the centroids at Hamming distance r from its own nearest centroid
 * with weight lut[r] (r = 0..8); a key collects the vote of the bucket it sits
 * in; votes are summed over the nb sub-blocks into an integer.
 */
void orc_coarse_scores(const uint8_t *codes, int64_t n, int nb, const uint8_t *qcode,
                       const int32_t *lut, int32_t *score)
{
    for (int64_t i = 0; i < n; i++) {
        int32_t s = 0;
        for (int b = 0; b < nb; b++)
            s += lut[popcount8((unsigned)(codes[i * nb + b] ^ qcode[b]))];
        score[i] = s;
    }
}

/* ------------------------------------------------------------------------ */
/* Selection orders.                                                         */
/* ------------------------------------------------------------------------ */

typedef struct {
    int32_t s;
    int64_t i;
} orc_int_key;

static int cmp_int_desc_idx_asc(const void *pa, const void *pb)
{
    const orc_int_key *a = (const orc_int_key *)pa, *b = (const orc_int_key *)pb;
    if (a->s != b->s)
        return (a->s > b->s) ? -1 : 1;
    return (a->i < b->i) ? -1 : (a->i > b->i);
}

typedef struct {
    float s;
    int64_t i;
} orc_flt_key;

/* fp32 comparison: -0.0 and +0.0 compare equal and fall to the index. */
static int cmp_flt_desc_idx_asc(const void *pa, const void *pb)
{
    const orc_flt_key *a = (const orc_flt_key *)pa, *b = (const orc_flt_key *)pb;
    if (a->s > b->s)
        return -1;
    if (a->s < b->s)
        return 1;
    return (a->i < b->i) ? -1 : (a->i > b->i);
}

static int cmp_i64_asc(const void *pa, const void *pb)
{
    int64_t a = *(const int64_t *)pa, b = *(const int64_t *)pb;
    return (a < b) ? -1 : (a > b);
}

/*
 * First c of n integer scores in the order (score descending, index
 * ascending); the chosen indices are written ascending. Returns min(c, n).
 */
int64_t orc_top_by_int(const int32_t *score, int64_t n, int64_t c, int64_t *out)
{
    if (c > n)
        c = n;
    if (c <= 0)
        return 0;
    orc_int_key *v = (orc_int_key *)malloc(sizeof(orc_int_key) * (size_t)n);
    for (int64_t i = 0; i < n; i++) {
        v[i].s = score[i];
        v[i].i = i;
    }
    qsort(v, (size_t)n, sizeof(orc_int_key), cmp_int_desc_idx_asc);
    for (int64_t j = 0; j < c; j++)
        out[j] = v[j].i;
    free(v);
    qsort(out, (size_t)c, sizeof(int64_t), cmp_i64_asc);
    return c;
}

/*
 * First c of n (score, index) pairs in the order (fp32 score descending,
 * index ascending); the chosen indices are written ascending. Returns
 * min(c, n), or -1 when a score is NaN.
 */
int64_t orc_top_by_float(const float *score, const int64_t *index, int64_t n, int64_t c,
                         int64_t *out)
{
    for (int64_t j = 0; j < n; j++)
        if (score[j] != score[j])
            return -1;
    if (c > n)
        c = n;
    if (c <= 0)
        return 0;
    orc_flt_key *v = (orc_flt_key *)malloc(sizeof(orc_flt_key) * (size_t)n);
    for (int64_t j = 0; j < n; j++) {
        v[j].s = score[j];
        v[j].i = index[j];
    }
    qsort(v, (size_t)n, sizeof(orc_flt_key), cmp_flt_desc_idx_asc);
    for (int64_t j = 0; j < c; j++)
        out[j] = v[j].i;
    free(v);
    qsort(out, (size_t)c, sizeof(int64_t), cmp_i64_asc);
    return c;
}

/* ------------------------------------------------------------------------ */
/* Step 4: exact rescoring of the candidates.                                */
/* ------------------------------------------------------------------------ */

/*
 * Exact logit of one candidate, q_bar . k, in the canonical fp32 order: the d
 * dims are cut into 16 contiguous chunks of d/16; chunk c accumulates
 * p_c = fma(q_j, k_j, p_c) over its dims j ascending from +0.0f; then four
 * butterfly rounds with span 8, 4, 2, 1 replace every p_c by p_c + p_{c^span};
 * the result is p_0.
 */
float orc_exact_score(const float *qbar, const float *k, int d)
{
    float p[16];
    int w = d / 16;
    for (int c = 0; c < 16; c++) {
        float acc = 0.0f;
        for (int j = c * w; j < (c + 1) * w; j++)
            acc = fmaf(qbar[j], k[j], acc);
        p[c] = acc;
    }
    for (int span = 8; span >= 1; span >>= 1) {
        float nxt[16];
        for (int c = 0; c < 16; c++)
            nxt[c] = p[c] + p[c ^ span];
        memcpy(p, nxt, sizeof(p));
    }
    return p[0];
}

/* ------------------------------------------------------------------------ */
/* Steps 1-4 for one (b, kv-head) unit.                                      */
/* ------------------------------------------------------------------------ */

/*
 * Selection for one unit at current length N (tokens 0..N-1 of K[N][d] and
 * codes[N][nb] are valid). The newest W tokens form the local window and are
 * never candidates; the pool is [0, N - W). Outputs:
 *   out_idx[0..k-1]: the final top-k' pool indices ascending, padded with -1;
 *   *out_count = k' = min(k, C'), C' = min(C, pool);
 *   cand[0..C'-1] (optional): the coarse candidate set, ascending;
 *   cand_S[0..C'-1] (optional): exact scores of cand[] in that order;
 *   coarse[0..pool-1] (optional): the coarse score of every pool key;
 *   qcode_out[0..nb-1] (optional): the query code.
 * Returns 0, or -1 on a NaN exact score or a bad shape.
 */
int orc_select_unit(const float *q, int G, const float *K, const uint8_t *codes, int64_t N,
                    int d, const int8_t *sgn, int64_t C, int64_t k, int64_t W,
                    const int32_t *lut, int32_t *out_idx, int32_t *out_count, int32_t *cand,
                    float *cand_S, int32_t *coarse, uint8_t *qcode_out)
{
    if (d % 16 != 0 || d > ORC_MAX_D || G < 1)
        return -1;
    int nb = d / ORC_M;
    int64_t pool = N - W;
    if (pool < 0)
        pool = 0;
    for (int64_t j = 0; j < k; j++)
        out_idx[j] = -1;
    *out_count = 0;

    float qbar[ORC_MAX_D];
    uint8_t qcode[ORC_MAX_D / ORC_M];
    orc_group_mean(q, G, d, qbar);
    orc_encode(qbar, 1, d, sgn, qcode);
    if (qcode_out)
        memcpy(qcode_out, qcode, (size_t)nb);
    if (pool == 0)
        return 0;

    int32_t *s = (int32_t *)malloc(sizeof(int32_t) * (size_t)pool);
    orc_coarse_scores(codes, pool, nb, qcode, lut, s);
    if (coarse)
        memcpy(coarse, s, sizeof(int32_t) * (size_t)pool);

    int64_t *cset = (int64_t *)malloc(sizeof(int64_t) * (size_t)(C > 0 ? C : 1));
    int64_t nc = orc_top_by_int(s, pool, C, cset);
    free(s);

    float *S = (float *)malloc(sizeof(float) * (size_t)(nc > 0 ? nc : 1));
    for (int64_t j = 0; j < nc; j++) {
        S[j] = orc_exact_score(qbar, K + cset[j] * (int64_t)d, d);
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

/* ------------------------------------------------------------------------ */
/* Step 5 [P-prob]: attention over the selected tokens plus the window.      */
/* ------------------------------------------------------------------------ */

/*
 * Attention of the G query heads q[G][d] of one unit over the token set
 * T = {idx[0..count-1]} U [max(0, N-W), N), in fp64 from the fp32 values of
 * q, K, V: s_t = (q_h . k_t) * scale, two-pass softmax (max, then
 * normalised sum). out[G][d]; an empty T gives zeros. Indices in idx must lie
 * in the pool [0, N-W); returns -1 otherwise.
 */
int orc_attend_unit(const float *q, int G, const float *K, const float *V, int64_t N, int d,
                    const int32_t *idx, int64_t count, int64_t W, float scale, double *out)
{
    int64_t w0 = N - W;
    if (w0 < 0)
        w0 = 0;
    int64_t nt = count + (N - w0);
    for (int64_t j = 0; j < count; j++)
        if (idx[j] < 0 || idx[j] >= w0)
            return -1;
    memset(out, 0, sizeof(double) * (size_t)G * (size_t)d);
    if (nt == 0)
        return 0;
    int64_t *tok = (int64_t *)malloc(sizeof(int64_t) * (size_t)nt);
    for (int64_t j = 0; j < count; j++)
        tok[j] = idx[j];
    for (int64_t t = w0; t < N; t++)
        tok[count + (t - w0)] = t;
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
            double p = s[j] / den;
            for (int c = 0; c < d; c++)
                oh[c] += p * (double)vt[c];
        }
    }
    free(s);
    free(tok);
    return 0;
}
