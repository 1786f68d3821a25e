/*
 * kvr_votes_oracle.c -- plain, slow CPU oracle of the magnitude-aware
 * reading of the coarse votes.
 *
 * TEST INFRASTRUCTURE, like kvr_oracle.c: only the test suite, the package
 * smoke check and the benchmark's CPU legs load it; the CUDA library shares
 * nothing with it. Built with -O2 -ffp-contract=off.
 *
 * Source: ParisKV, "Pipeline di Recupero Nativa su GPU in Due Stadi": per
 * sub-space the query selects its top-rho most similar centroids; keys in
 * those buckets receive tiered votes, summed over the sub-spaces into an
 * integer coarse score.
 *
 * Readings (the literal one: centroids ranked by their similarity to the
 * rotated query sub-vector, magnitudes included):
 *   - zq = FWHT(D q_bar) (the codes' rotation, fp32 canonical order); per
 *     sub-block b of 8 coordinates, a_j = |zq_{8b+j}| and the query code bit
 *     s_j = (zq_{8b+j} < 0);
 *   - a centroid c (a sign pattern) differs from the query code in the flip
 *     set x = c XOR qcode_b; <zq_b, c> = (sum_j a_j - 2 sum_{j in x} a_j)/sqrt(8),
 *     so ranking by similarity is ranking by the flip cost
 *     f(x) = sum over set bits j of x, ascending, of a_j (fp32 from +0);
 *   - order: (f(x) ascending, x ascending); rank r(x) in 0..255;
 *   - tiers: the ring sizes of the Hamming reading, in rank order: ranks
 *     0 | 1..8 | 9..36 | 37..92 | 93..162 | 163..218 | 219..246 | 247..254 |
 *     255 are tiers 0..8, and the vote of x is lut[tier(r(x))];
 *   - coarse score of a key = sum over sub-blocks of vote_b(code_b XOR
 *     qcode_b); everything after it (candidates by (score desc, index asc),
 *     exact rescoring, top-k) as in orc_select_unit.
 * With all a_j of a sub-block equal, f(x) = popcount(x) a_j exactly for the
 * sums involved, the order is by popcount then x, and the votes are the
 * Hamming-ring votes lut[popcount(x)].
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define VT_M 8
#define VT_MAXD 128

/* from kvr_oracle.c (the same oracle library) */
void orc_fwht_f32(float *x, int d);
void orc_group_mean(const float *q, int G, int d, float *qbar);
int orc_encode(const float *x, int64_t n, int d, const int8_t *sgn, uint8_t *codes);
int64_t orc_top_by_int(const int32_t *score, int64_t n, int64_t c, int64_t *out);
int64_t orc_top_by_float(const float *score, const int64_t *index, int64_t n, int64_t c,
                         int64_t *out);
float orc_exact_score(const float *qbar, const float *k, int d);

static const int ring_end[9] = {1, 9, 37, 93, 163, 219, 247, 255, 256};

float orc_flip_cost(const float *a, unsigned x)
{
    float f = 0.0f;
    for (int j = 0; j < VT_M; j++)
        if ((x >> j) & 1u)
            f = f + a[j];
    return f;
}

/* Vote tables T[nb][256] of the rotated query zq[d]. */
int orc_mag_vote_table(const float *zq, int d, const int32_t *lut, int32_t *T)
{
    if (d % VT_M != 0 || d > VT_MAXD)
        return -1;
    const int nb = d / VT_M;
    for (int b = 0; b < nb; b++) {
        float a[VT_M], f[256];
        for (int j = 0; j < VT_M; j++) {
            const float z = zq[b * VT_M + j];
            a[j] = z < 0.0f ? -z : z;
        }
        for (unsigned x = 0; x < 256; x++)
            f[x] = orc_flip_cost(a, x);
        for (unsigned x = 0; x < 256; x++) {
            int r = 0;  /* patterns before x in the order */
            for (unsigned y = 0; y < 256; y++)
                if (f[y] < f[x] || (f[y] == f[x] && y < x))
                    r++;
            int tier = 0;
            while (r >= ring_end[tier])
                tier++;
            T[b * 256 + x] = lut[tier];
        }
    }
    return 0;
}

/*
 * Selection of one unit with magnitude-aware votes: as orc_select_unit, the
 * coarse score of each pool key from the vote tables. coarse (optional,
 * pool entries) and table (optional, nb * 256) receive the coarse scores and
 * the vote tables.
 */
int orc_select_unit_mag(const float *q, int G, const float *K, const uint8_t *codes, int64_t N,
                        int d, const int8_t *sgn, int64_t C, int64_t k, int64_t W,
                        const int32_t *lut, int32_t *out_idx, int32_t *out_count, int32_t *cand,
                        float *cand_S, int32_t *coarse, int32_t *table)
{
    if (d % 16 != 0 || d > VT_MAXD || G < 1)
        return -1;
    const int nb = d / VT_M;
    int64_t pool = N - W;
    if (pool < 0)
        pool = 0;
    for (int64_t j = 0; j < k; j++)
        out_idx[j] = -1;
    *out_count = 0;
    float qbar[VT_MAXD], zq[VT_MAXD];
    uint8_t qcode[VT_MAXD / VT_M];
    orc_group_mean(q, G, d, qbar);
    orc_encode(qbar, 1, d, sgn, qcode);
    for (int j = 0; j < d; j++)
        zq[j] = qbar[j] * (float)sgn[j];
    orc_fwht_f32(zq, d);
    int32_t *T = (int32_t *)malloc(sizeof(int32_t) * (size_t)nb * 256);
    orc_mag_vote_table(zq, d, lut, T);
    if (table)
        memcpy(table, T, sizeof(int32_t) * (size_t)nb * 256);
    if (pool == 0) {
        free(T);
        return 0;
    }
    int32_t *s = (int32_t *)malloc(sizeof(int32_t) * (size_t)pool);
    for (int64_t i = 0; i < pool; i++) {
        int32_t v = 0;
        for (int b = 0; b < nb; b++)
            v += T[b * 256 + (codes[i * nb + b] ^ qcode[b])];
        s[i] = v;
    }
    free(T);
    if (coarse)
        memcpy(coarse, s, sizeof(int32_t) * (size_t)pool);
    int64_t *cset = (int64_t *)malloc(sizeof(int64_t) * (size_t)(C > 0 ? C : 1));
    const int64_t nc = orc_top_by_int(s, pool, C, cset);
    free(s);
    float *Sc = (float *)malloc(sizeof(float) * (size_t)(nc > 0 ? nc : 1));
    for (int64_t j = 0; j < nc; j++) {
        Sc[j] = orc_exact_score(qbar, K + cset[j] * (int64_t)d, d);
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
