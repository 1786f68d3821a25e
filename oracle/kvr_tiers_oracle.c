/*
 * kvr_tiers_oracle.c -- plain, slow CPU oracle for the tiered window cache:
 * INT2 quantisation with a write-once ledger, attention over bf16 and INT2
 * windows with per-window attention mass, and the cumulative-score routing
 * of windows between the bf16, INT2 and evicted tiers.
 *
 * TEST INFRASTRUCTURE, like kvr_oracle.c: only the test suite, the package
 * smoke check and the benchmark's CPU legs load it; the CUDA library shares
 * nothing with it. Built with -O2 -ffp-contract=off and no fast-math: each
 * fp32 operation is one IEEE round-to-nearest-even operation in the order
 * written.
 *
 * Sources (page title, section):
 *   [Q-meth]  QEvict, "Metodologia: QEvict": the cache is split into
 *             contiguous windows, each kept at full precision, in a
 *             recoverable low-bit (INT2) form, or evicted, under a fixed
 *             memory budget.
 *   [Q-mech]  QEvict, "Meccanismi Chiave": routing per window; a window's
 *             importance is its attention mass accumulated over decode steps;
 *             demotion to the quantised tier, promotion back by
 *             dequantisation; a window is quantised once, at its first
 *             demotion, into a persistent ledger reused by every later move;
 *             GQA support.
 *
 * Readings (the pages give no constants and no quantiser):
 *   - windows of 64 tokens; window w holds tokens [64w, 64w + 64); windows
 *     below floor(N/64) are closed and routed, the newest partial window is
 *     open, always bf16 and always attended;
 *   - INT2 is asymmetric per token and per group of 32 contiguous channels of
 *     the head dimension, for K and V alike, with an fp16 scale and zero:
 *     z = fp16 rounded down from the group minimum, s = the smallest fp16 at
 *     or above fl((max - z) / 3) with fl(3 s + z) >= max, code =
 *     clamp(rint((x - z) / s), 0, 3) (code 0 when s = 0), value =
 *     fl(code * s + z) with one rounding; a promoted window stores the bf16
 *     nearest to each value;
 *   - the mass of window w for one KV head is the softmax probability of its
 *     tokens summed over the tokens and over the G query heads of the group;
 *     the score adds llrint(mass * 2^32) each step (int64), evicted windows
 *     keep their score and get no mass;
 *   - each step ranks the live closed windows by (score desc, window asc);
 *     the first quota (the initial bf16 count) are bf16, the others INT2;
 *     while the tier bytes exceed the budget (initial bf16 count * 64 tokens *
 *     2 rows * 2d bytes + initial INT2 count * ledger bytes), the lowest-ranked
 *     INT2 window is evicted, for good. A bf16 window that leaves the bf16
 *     tier writes its ledger only if it has none.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_WIN 64   /* tokens per routed window */
#define ORC_QG 32    /* channels per INT2 group */

enum { ORC_BF16 = 0, ORC_INT2 = 1, ORC_EVICTED = 2 };

/* ------------------------------------------------------------------------ */
/* IEEE binary16 and bfloat16 from their definitions.                        */
/* ------------------------------------------------------------------------ */

/* Exact value of an fp16 bit pattern (1 sign, 5 exponent, 10 fraction bits). */
static double f16_value(uint16_t h)
{
    const int e = (h >> 10) & 31, m = h & 1023;
    double v;
    if (e == 31)
        v = m ? NAN : INFINITY;
    else if (e == 0)
        v = ldexp((double)m, -24);
    else
        v = ldexp((double)(1024 + m), e - 25);
    return (h & 0x8000) ? -v : v;
}

float orc_f16_to_f32(uint16_t h) { return (float)f16_value(h); }

/* Ordered key of a non-NaN fp16: monotone in the value (both zeros -> 0). */
static int f16_key(uint16_t h) { return (h & 0x8000) ? -(int)(h & 0x7fff) : (int)h; }
static uint16_t f16_of_key(int k) { return k < 0 ? (uint16_t)(0x8000 | -k) : (uint16_t)k; }

/*
 * fp16 rounded toward -inf (dir < 0) or +inf (dir > 0): the largest (smallest)
 * fp16 value, infinities included, that is <= x (>= x). An exact zero keeps
 * its sign; a result of zero from a nonzero x takes the sign of x, as IEEE
 * directed rounding does. NaN gives the canonical fp16 NaN.
 */
static uint16_t f16_directed(float xf, int dir)
{
    if (xf != xf)
        return 0x7e00;
    const double x = (double)xf;
    if (x == 0.0)
        return signbit(xf) ? 0x8000 : 0x0000;
    /* binary search over keys [-0x7c00, 0x7c00] (-inf .. +inf) */
    int lo = -0x7c00, hi = 0x7c00;
    if (dir < 0) {
        /* largest key with value <= x; value(-inf) <= x always */
        while (lo < hi) {
            const int mid = lo + (hi - lo + 1) / 2;
            if (f16_value(f16_of_key(mid)) <= x)
                lo = mid;
            else
                hi = mid - 1;
        }
    } else {
        /* smallest key with value >= x; value(+inf) >= x always */
        while (lo < hi) {
            const int mid = lo + (hi - lo) / 2;
            if (f16_value(f16_of_key(mid)) >= x)
                hi = mid;
            else
                lo = mid + 1;
        }
    }
    uint16_t h = f16_of_key(lo);
    if ((h & 0x7fff) == 0)
        h = (x < 0) ? 0x8000 : 0x0000;
    return h;
}

uint16_t orc_f32_to_f16_rd(float x) { return f16_directed(x, -1); }
uint16_t orc_f32_to_f16_ru(float x) { return f16_directed(x, +1); }

/* The next fp16 above a finite non-NaN h (+0 after -0 is skipped: -0 -> smallest subnormal). */
uint16_t orc_f16_next_up(uint16_t h)
{
    int k = f16_key(h);
    if (k >= 0x7c00)
        return h;
    return f16_of_key(k + 1);
}

/*
 * bfloat16 nearest to x (ties to even), returned as the fp32 with the same
 * value: bfloat16 keeps the top 16 bits of the fp32 encoding, so rounding
 * adds half of the dropped range, minus one unless the kept part is odd, and
 * truncates. NaN stays NaN.
 */
float orc_bf16_round(float x)
{
    uint32_t u;
    memcpy(&u, &x, 4);
    if ((u & 0x7fffffffu) > 0x7f800000u) {
        u |= 0x00400000u;
    } else {
        const uint32_t keep_odd = (u >> 16) & 1u;
        u += 0x7fffu + keep_odd;
    }
    u &= 0xffff0000u;
    float r;
    memcpy(&r, &u, 4);
    return r;
}

/* ------------------------------------------------------------------------ */
/* INT2 with an fp16 scale and zero per group of 32 channels [Q-meth].       */
/* ------------------------------------------------------------------------ */

/*
 * Quantise x[0..31]: codes[8] (element j at byte j/4, bits 2*(j%4)),
 * scale and zero as fp16 bit patterns. Returns -1 if the range does not fit
 * fp16 (z or s not finite), 0 otherwise.
 */
int orc_int2_quantize_group(const float *x, uint8_t *codes, uint16_t *scale, uint16_t *zero)
{
    float mn = x[0], mx = x[0];
    for (int j = 1; j < ORC_QG; j++) {
        if (x[j] < mn)
            mn = x[j];
        if (x[j] > mx)
            mx = x[j];
    }
    const uint16_t z16 = orc_f32_to_f16_rd(mn);
    const float z = orc_f16_to_f32(z16);
    const float r = (mx - z) / 3.0f;
    uint16_t s16 = orc_f32_to_f16_ru(r);
    int bad = !isfinite(z) || !isfinite(orc_f16_to_f32(s16));
    while (!bad && fmaf(3.0f, orc_f16_to_f32(s16), z) < mx) {
        s16 = orc_f16_next_up(s16);
        bad = !isfinite(orc_f16_to_f32(s16));
    }
    const float s = orc_f16_to_f32(s16);
    memset(codes, 0, ORC_QG / 4);
    for (int j = 0; j < ORC_QG; j++) {
        int c = 0;
        if (s != 0.0f && !bad) {
            const float t = rintf((x[j] - z) / s);
            c = t < 0.0f ? 0 : (t > 3.0f ? 3 : (int)t);
        }
        codes[j >> 2] |= (uint8_t)(c << (2 * (j & 3)));
    }
    *scale = s16;
    *zero = z16;
    return bad ? -1 : 0;
}

/* Values of one group: out[j] = fl(code_j * s + z). */
void orc_int2_dequantize_group(const uint8_t *codes, uint16_t scale, uint16_t zero, float *out)
{
    const float s = orc_f16_to_f32(scale), z = orc_f16_to_f32(zero);
    for (int j = 0; j < ORC_QG; j++) {
        const int c = (codes[j >> 2] >> (2 * (j & 3))) & 3;
        out[j] = fmaf((float)c, s, z);
    }
}

/* Bytes of one window's ledger: K codes, K params, V codes, V params. */
int64_t orc_ledger_bytes(int d) { return 2 * (int64_t)ORC_WIN * (d / ORC_QG) * (8 + 4); }

/*
 * Ledger of one window from its 64 K rows and 64 V rows (fp32 values, [64][d]).
 * Layout: [K codes: token, group, 8 B][K params: token, group, (fp16 scale,
 * fp16 zero) little-endian][V codes][V params]. Returns the number of groups
 * whose range did not fit fp16.
 */
int orc_ledger_write_window(const float *Kw, const float *Vw, int d, uint8_t *ledger)
{
    const int ng = d / ORC_QG;
    const int64_t cbytes = (int64_t)ORC_WIN * ng * 8, pbytes = (int64_t)ORC_WIN * ng * 4;
    int bad = 0;
    for (int kv = 0; kv < 2; kv++) {
        const float *X = kv ? Vw : Kw;
        uint8_t *codes = ledger + kv * (cbytes + pbytes);
        uint8_t *params = codes + cbytes;
        for (int t = 0; t < ORC_WIN; t++)
            for (int g = 0; g < ng; g++) {
                uint16_t s, z;
                bad += orc_int2_quantize_group(X + (int64_t)t * d + g * ORC_QG,
                                               codes + ((int64_t)t * ng + g) * 8, &s, &z) != 0;
                uint8_t *p = params + ((int64_t)t * ng + g) * 4;
                p[0] = (uint8_t)(s & 0xff);
                p[1] = (uint8_t)(s >> 8);
                p[2] = (uint8_t)(z & 0xff);
                p[3] = (uint8_t)(z >> 8);
            }
    }
    return bad;
}

/* The window's dequantised fp32 K and V rows, [64][d] each. */
void orc_ledger_read_window(const uint8_t *ledger, int d, float *Kw, float *Vw)
{
    const int ng = d / ORC_QG;
    const int64_t cbytes = (int64_t)ORC_WIN * ng * 8, pbytes = (int64_t)ORC_WIN * ng * 4;
    for (int kv = 0; kv < 2; kv++) {
        float *X = kv ? Vw : Kw;
        const uint8_t *codes = ledger + kv * (cbytes + pbytes);
        const uint8_t *params = codes + cbytes;
        for (int t = 0; t < ORC_WIN; t++)
            for (int g = 0; g < ng; g++) {
                const uint8_t *p = params + ((int64_t)t * ng + g) * 4;
                const uint16_t s = (uint16_t)(p[0] | (p[1] << 8));
                const uint16_t z = (uint16_t)(p[2] | (p[3] << 8));
                orc_int2_dequantize_group(codes + ((int64_t)t * ng + g) * 8, s, z,
                                          X + (int64_t)t * d + g * ORC_QG);
            }
    }
}

/* ------------------------------------------------------------------------ */
/* Attention over the tiers, with window mass [Q-meth], [Q-mech].            */
/* ------------------------------------------------------------------------ */

/*
 * One unit (batch entry, KV head) of length N: G query heads q[G][d]; K, V
 * [cap][d] fp32 values of the bf16 cache; ledger [n_win][ledger bytes];
 * tier[n_win]. Tokens attended: closed windows (w < N/64) of tier bf16 from
 * K, V; closed windows of tier INT2 from their dequantised ledger; the open
 * window [64 floor(N/64), N) from K, V; evicted windows not at all. fp64
 * two-pass softmax of s = (q_h . k_t) * scale. out[G][d]; mass[w] for
 * w < ceil(N/64): the probability of the window's tokens summed over tokens
 * and heads (0 for evicted windows). Returns -1 on a bad tier value.
 */
int orc_tiered_attend_unit(const float *q, int G, const float *K, const float *V,
                           const uint8_t *ledger, const int8_t *tier, int64_t N, int d,
                           float scale, double *out, double *mass)
{
    const int64_t closed = N / ORC_WIN, nw = (N + ORC_WIN - 1) / ORC_WIN;
    const int64_t lb = orc_ledger_bytes(d);
    for (int64_t w = 0; w < closed; w++)
        if (tier[w] < ORC_BF16 || tier[w] > ORC_EVICTED)
            return -1;
    /* gather the attended rows (dequantising INT2 windows) */
    int64_t nt = 0;
    for (int64_t w = 0; w < nw; w++)
        if (w >= closed || tier[w] != ORC_EVICTED)
            nt += (w < closed) ? ORC_WIN : N - w * ORC_WIN;
    memset(out, 0, sizeof(double) * (size_t)G * (size_t)d);
    for (int64_t w = 0; w < nw; w++)
        mass[w] = 0.0;
    if (nt == 0)
        return 0;
    float *Kt = (float *)malloc(sizeof(float) * (size_t)nt * (size_t)d);
    float *Vt = (float *)malloc(sizeof(float) * (size_t)nt * (size_t)d);
    int64_t *win = (int64_t *)malloc(sizeof(int64_t) * (size_t)nt);
    int64_t j = 0;
    for (int64_t w = 0; w < nw; w++) {
        if (w < closed && tier[w] == ORC_EVICTED)
            continue;
        const int64_t t0 = w * ORC_WIN, n = (w < closed) ? ORC_WIN : N - t0;
        if (w < closed && tier[w] == ORC_INT2) {
            orc_ledger_read_window(ledger + w * lb, d, Kt + j * d, Vt + j * d);
        } else {
            memcpy(Kt + j * d, K + t0 * d, sizeof(float) * (size_t)(n * d));
            memcpy(Vt + j * d, V + t0 * d, sizeof(float) * (size_t)(n * d));
        }
        for (int64_t i = 0; i < n; i++)
            win[j + i] = w;
        j += n;
    }
    double *s = (double *)malloc(sizeof(double) * (size_t)nt);
    for (int h = 0; h < G; h++) {
        const float *qh = q + (int64_t)h * d;
        double mx = -INFINITY;
        for (int64_t t = 0; t < nt; t++) {
            double acc = 0.0;
            for (int c = 0; c < d; c++)
                acc += (double)qh[c] * (double)Kt[t * d + c];
            s[t] = acc * (double)scale;
            if (s[t] > mx)
                mx = s[t];
        }
        double den = 0.0;
        for (int64_t t = 0; t < nt; t++) {
            s[t] = exp(s[t] - mx);
            den += s[t];
        }
        double *oh = out + (int64_t)h * d;
        for (int64_t t = 0; t < nt; t++) {
            const double p = s[t] / den;
            mass[win[t]] += p;
            for (int c = 0; c < d; c++)
                oh[c] += p * (double)Vt[t * d + c];
        }
    }
    free(s);
    free(win);
    free(Vt);
    free(Kt);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Tier set-up and routing [Q-meth], [Q-mech].                               */
/* ------------------------------------------------------------------------ */

/* Bytes a window costs in the budget: bf16 K and V rows, or its ledger. */
static int64_t bf16_window_bytes(int d) { return (int64_t)ORC_WIN * 2 * 2 * d; }

/*
 * Set-up of one unit of length N over n_win windows: tiers of the closed
 * windows from init[] (0 bf16, 1 INT2, 2 evicted), windows at and after the
 * open one bf16; INT2 windows get their ledger quantised from K, V; scores 0.
 * quota = the number of bf16 closed windows, budget = the bytes of the
 * initial tiers. Returns -1 on a bad tier value, else the number of groups
 * whose range did not fit fp16.
 */
int orc_tier_init_unit(const int8_t *init, const float *K, const float *V, int64_t N, int d,
                       int64_t n_win, int8_t *tier, int64_t *score, uint8_t *has_ledger,
                       uint8_t *ledger, int32_t *quota, int64_t *budget)
{
    const int64_t closed = N / ORC_WIN, lb = orc_ledger_bytes(d);
    int64_t n_bf = 0, n_q = 0;
    int bad = 0;
    for (int64_t w = 0; w < n_win; w++) {
        const int8_t t = (w < closed) ? init[w] : ORC_BF16;
        if (t < ORC_BF16 || t > ORC_EVICTED)
            return -1;
        tier[w] = t;
        score[w] = 0;
        has_ledger[w] = 0;
        if (w < closed && t == ORC_BF16)
            n_bf++;
        if (w < closed && t == ORC_INT2) {
            n_q++;
            bad += orc_ledger_write_window(K + w * ORC_WIN * d, V + w * ORC_WIN * d, d,
                                           ledger + w * lb);
            has_ledger[w] = 1;
        }
    }
    *quota = (int32_t)n_bf;
    *budget = n_bf * bf16_window_bytes(d) + n_q * lb;
    return bad;
}

typedef struct {
    int64_t score;
    int64_t w;
} rank_entry;

static int cmp_rank(const void *pa, const void *pb)
{
    const rank_entry *a = (const rank_entry *)pa, *b = (const rank_entry *)pb;
    if (a->score != b->score)
        return a->score > b->score ? -1 : 1;
    return a->w < b->w ? -1 : (a->w > b->w);
}

/*
 * One routing step of one unit after attention over length N: mass[w]
 * (fp32, w < ceil(N/64)) is added to the score of every non-evicted window
 * as llrint(mass * 2^32); the live closed windows are ranked and re-tiered
 * (see the readings above); data moves: bf16 -> INT2 writes the ledger if the
 * window has none, INT2 -> bf16 writes the bf16-rounded dequantised rows into
 * K, V; evictions move nothing. stats = {promotions, demotions, evictions}.
 * Returns -1 on a bad tier value, else the number of groups whose range did
 * not fit fp16 in ledgers written by this step.
 */
int orc_tier_update_unit(int8_t *tier, int64_t *score, uint8_t *has_ledger, uint8_t *ledger,
                         float *K, float *V, const float *mass, int64_t N, int d, int32_t quota,
                         int64_t budget, int32_t *stats)
{
    const int64_t closed = N / ORC_WIN, nw = (N + ORC_WIN - 1) / ORC_WIN;
    const int64_t lb = orc_ledger_bytes(d);
    stats[0] = stats[1] = stats[2] = 0;
    for (int64_t w = 0; w < nw; w++)
        if (tier[w] < ORC_BF16 || tier[w] > ORC_EVICTED)
            return -1;
    for (int64_t w = 0; w < nw; w++)
        if (tier[w] != ORC_EVICTED)
            score[w] += llrint((double)mass[w] * 4294967296.0);

    rank_entry *r = (rank_entry *)malloc(sizeof(rank_entry) * (size_t)(closed + 1));
    int64_t live = 0;
    for (int64_t w = 0; w < closed; w++)
        if (tier[w] != ORC_EVICTED) {
            r[live].score = score[w];
            r[live].w = w;
            live++;
        }
    qsort(r, (size_t)live, sizeof(rank_entry), cmp_rank);
    int8_t *nt = (int8_t *)malloc((size_t)(live + 1));
    int64_t bytes = 0;
    for (int64_t i = 0; i < live; i++) {
        nt[i] = (i < quota) ? ORC_BF16 : ORC_INT2;
        bytes += (nt[i] == ORC_BF16) ? bf16_window_bytes(d) : lb;
    }
    for (int64_t i = live - 1; i >= 0 && bytes > budget; i--)
        if (nt[i] == ORC_INT2) {
            nt[i] = ORC_EVICTED;
            bytes -= lb;
        }
    int bad = 0;
    float *Kw = (float *)malloc(sizeof(float) * ORC_WIN * (size_t)d);
    float *Vw = (float *)malloc(sizeof(float) * ORC_WIN * (size_t)d);
    for (int64_t i = 0; i < live; i++) {
        const int64_t w = r[i].w;
        const int8_t from = tier[w], to = nt[i];
        if (from == ORC_BF16 && to == ORC_INT2) {
            if (!has_ledger[w]) {
                bad += orc_ledger_write_window(K + w * ORC_WIN * d, V + w * ORC_WIN * d, d,
                                               ledger + w * lb);
                has_ledger[w] = 1;
            }
            stats[1]++;
        } else if (from == ORC_INT2 && to == ORC_BF16) {
            orc_ledger_read_window(ledger + w * lb, d, Kw, Vw);
            for (int64_t e = 0; e < ORC_WIN * (int64_t)d; e++) {
                K[w * ORC_WIN * d + e] = orc_bf16_round(Kw[e]);
                V[w * ORC_WIN * d + e] = orc_bf16_round(Vw[e]);
            }
            stats[0]++;
        } else if (to == ORC_EVICTED) {
            stats[2]++;
        }
        tier[w] = to;
    }
    free(Vw);
    free(Kw);
    free(nt);
    free(r);
    return bad;
}

/* ------------------------------------------------------------------------ */
/* Array forms of the conversions (for tests over many samples).             */
/* ------------------------------------------------------------------------ */

void orc_f32_to_f16_array(const float *x, int64_t n, int dir, uint16_t *out)
{
    for (int64_t i = 0; i < n; i++)
        out[i] = f16_directed(x[i], dir);
}

void orc_bf16_round_array(const float *x, int64_t n, float *out)
{
    for (int64_t i = 0; i < n; i++)
        out[i] = orc_bf16_round(x[i]);
}
