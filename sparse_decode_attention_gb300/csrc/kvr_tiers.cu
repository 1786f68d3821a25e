// kvr_tiers.cu -- the tiered window cache: INT2 quantisation into a
// write-once ledger, attention over bf16 and INT2 windows with the attention
// mass of every window, and the cumulative-score routing between the bf16,
// INT2 and evicted tiers.
//
// Source: QEvict, "Metodologia: QEvict" (contiguous windows in a
// full-precision, a recoverable INT2 or an evicted tier under a fixed memory
// budget) and "Meccanismi Chiave" (routing per window, cumulative attention
// scores, demotion / promotion, write-once ledger, GQA).
//
// Kernels:
//   tier_init_kernel     grid (kInitX, U): tiers, scores, ledgers of the
//                        initially INT2 windows (one CTA per window at a time)
//   tier_count_kernel    grid U: quota and budget from the initial tiers
//   tiered_attend_kernel grid (S, U): each CTA streams a contiguous range of
//                        its unit's windows through shared memory (cp.async,
//                        double-buffered: 64 K + 64 V rows of a bf16 window,
//                        or the window's ledger), scores them for the G heads,
//                        keeps an online softmax and writes its partial
//                        (m, l, o) plus the log2-sum-exp of every window
//   tiered_combine_kernel grid U: merges the S partials into the output and
//                        turns the window log2-sum-exps into window masses
//   tier_rank_kernel     grid U: score update, bitonic ranking of the live
//                        closed windows, new tiers, list of data moves
//   tier_move_kernel     grid (kMoveX, U): quantise demoted windows without a
//                        ledger, dequantise promoted windows into K, V
#include <algorithm>

#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math_constants.h>

#include "kvr_device.cuh"
#include "kvr_launch.h"

namespace kvr {

namespace {

constexpr int kWin = 64;        // tokens per window
constexpr int kQG = 32;         // channels per INT2 group
constexpr int kThreads = 256;   // threads of the init / attend / move kernels
constexpr int kRankThreads = 1024;
constexpr int kInitX = 64;      // init CTAs per unit
constexpr int kMoveX = 16;      // move CTAs per unit
constexpr int kMaxWin = 16384;  // windows per unit the ranking holds in shared memory

__host__ __device__ constexpr int ledger_bytes_of(int d) { return 2 * kWin * (d / kQG) * 12; }

// ---------------------------------------------------------------- INT2 groups

// The fp16 value one step above a non-negative, finite fp16 bit pattern.
__device__ __forceinline__ unsigned short f16_next_up_pos(unsigned short h)
{
    return (h & 0x8000u) ? (unsigned short)0x0001u : (unsigned short)(h + 1u);
}

// Quantise one group of 32 values: codes (element j at byte j/4, bits
// 2 (j%4)), params = fp16 scale | fp16 zero << 16. Returns false when the
// range does not fit fp16. The scan order of min / max (strict compares from
// element 0) fixes the sign of a zero extreme.
__device__ __forceinline__ bool quant_group(const float (&x)[kQG], uint2 &codes, uint32_t &params)
{
    float mn = x[0], mx = x[0];
#pragma unroll
    for (int j = 1; j < kQG; j++) {
        if (x[j] < mn) mn = x[j];
        if (x[j] > mx) mx = x[j];
    }
    const __half zh = __float2half_rd(mn);
    const float z = __half2float(zh);
    const float r = __fdiv_rn(__fsub_rn(mx, z), 3.0f);
    unsigned short sb = __half_as_ushort(__float2half_ru(r));
    bool ok = isfinite(z) && isfinite(__half2float(__ushort_as_half(sb)));
    // one step up always suffices (the shortfall is a few fp32 ulps of the
    // range, one fp16 step is 2^-10 of the scale); the bound is a guard
    for (int it = 0; it < 4 && ok && fmaf(3.0f, __half2float(__ushort_as_half(sb)), z) < mx;
         it++) {
        sb = f16_next_up_pos(sb);
        ok = isfinite(__half2float(__ushort_as_half(sb)));
    }
    const float s = __half2float(__ushort_as_half(sb));
    uint32_t lo = 0, hi = 0;
#pragma unroll
    for (int j = 0; j < kQG; j++) {
        uint32_t c = 0;
        if (ok && s != 0.0f) {
            const float t = rintf(__fdiv_rn(__fsub_rn(x[j], z), s));
            c = t < 0.0f ? 0u : (t > 3.0f ? 3u : (uint32_t)t);
        }
        if (j < 16) lo |= c << (2 * j);
        else hi |= c << (2 * (j - 16));
    }
    codes = make_uint2(lo, hi);
    params = (uint32_t)sb | ((uint32_t)__half_as_ushort(zh) << 16);
    return ok;
}

__device__ __forceinline__ void load_group_bf16(const __nv_bfloat16 *src, float (&x)[kQG])
{
    const uint4 *p = reinterpret_cast<const uint4 *>(src);
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const uint4 v = p[i];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; k++) {
            x[8 * i + 2 * k] = bf16_lo(w[k]);
            x[8 * i + 2 * k + 1] = bf16_hi(w[k]);
        }
    }
}

// Ledger of one window from its 64 K rows and 64 V rows (row stride D), by the
// whole CTA.
template <int D>
__device__ void quantize_window(const __nv_bfloat16 *Kw, const __nv_bfloat16 *Vw,
                                uint8_t *ledger, int32_t *err)
{
    constexpr int NG = D / kQG, GROUPS = kWin * NG, CB = kWin * NG * 8, PB = kWin * NG * 4;
    for (int i = threadIdx.x; i < 2 * GROUPS; i += blockDim.x) {
        const int kv = i >= GROUPS, gi = kv ? i - GROUPS : i;
        float x[kQG];
        load_group_bf16((kv ? Vw : Kw) + (size_t)gi * kQG, x);
        uint2 codes;
        uint32_t params;
        if (!quant_group(x, codes, params)) set_err(err, KVR_DEVERR_RANGE);
        uint8_t *base = ledger + kv * (CB + PB);
        *reinterpret_cast<uint2 *>(base + gi * 8) = codes;
        *reinterpret_cast<uint32_t *>(base + CB + gi * 4) = params;
    }
}

// bf16 rows of one window from its ledger, by the whole CTA.
template <int D>
__device__ void dequantize_window(const uint8_t *ledger, __nv_bfloat16 *Kw, __nv_bfloat16 *Vw)
{
    constexpr int NG = D / kQG, GROUPS = kWin * NG, CB = kWin * NG * 8, PB = kWin * NG * 4;
    for (int i = threadIdx.x; i < 2 * GROUPS; i += blockDim.x) {
        const int kv = i >= GROUPS, gi = kv ? i - GROUPS : i;
        const uint8_t *base = ledger + kv * (CB + PB);
        const uint2 codes = *reinterpret_cast<const uint2 *>(base + gi * 8);
        const uint32_t params = *reinterpret_cast<const uint32_t *>(base + CB + gi * 4);
        const float s = __half2float(__ushort_as_half((unsigned short)(params & 0xffffu)));
        const float z = __half2float(__ushort_as_half((unsigned short)(params >> 16)));
        uint32_t out[16];
#pragma unroll
        for (int j = 0; j < kQG; j += 2) {
            const uint32_t w = j < 16 ? codes.x : codes.y;
            const int sh = 2 * (j & 15);
            const float a = fmaf((float)((w >> sh) & 3u), s, z);
            const float b = fmaf((float)((w >> (sh + 2)) & 3u), s, z);
            const __nv_bfloat162 p = __floats2bfloat162_rn(a, b);
            out[j / 2] = *reinterpret_cast<const uint32_t *>(&p);
        }
        uint4 *dst = reinterpret_cast<uint4 *>((kv ? Vw : Kw) + (size_t)gi * kQG);
#pragma unroll
        for (int i4 = 0; i4 < 4; i4++)
            dst[i4] = make_uint4(out[4 * i4], out[4 * i4 + 1], out[4 * i4 + 2], out[4 * i4 + 3]);
    }
}

// Length of unit u's batch entry, or -1 (error flagged) when outside [0, cap].
__device__ __forceinline__ int64_t unit_len(const int32_t *seq_len, int b, int64_t cap,
                                            int32_t *err)
{
    const int64_t N = seq_len[b];
    if (N < 0 || N > cap) {
        if (threadIdx.x == 0) set_err(err, KVR_DEVERR_SEQ_LEN);
        return -1;
    }
    return N;
}

__device__ __forceinline__ int8_t checked_tier(int8_t t, int32_t *err)
{
    if (t < KVR_TIER_BF16 || t > KVR_TIER_EVICTED) {
        set_err(err, KVR_DEVERR_TIER);
        return KVR_TIER_EVICTED;
    }
    return t;
}

// ---------------------------------------------------------------- init

struct TierArgs {
    int Hkv, d;
    int64_t cap, n_win;
    int8_t *tier;
    int64_t *score;
    uint8_t *has_ledger, *ledger;
    int32_t *quota;
    int64_t *budget;
};

template <int D>
__global__ void __launch_bounds__(kThreads) tier_init_kernel(TierArgs a, const int8_t *init,
                                                             const __nv_bfloat16 *K,
                                                             const __nv_bfloat16 *V,
                                                             const int32_t *seq_len, int32_t *err)
{
    const int u = blockIdx.y, b = u / a.Hkv;
    int64_t N = unit_len(seq_len, b, a.cap, err);
    const bool bad_len = N < 0;
    if (bad_len) N = 0;
    const int64_t closed = N / kWin;
    const size_t uw = (size_t)u * a.n_win;
    for (int64_t w = blockIdx.x; w < a.n_win; w += gridDim.x) {
        int8_t t = KVR_TIER_BF16;
        if (w < closed) t = checked_tier(init[uw + w], threadIdx.x == 0 ? err : nullptr);
        if (threadIdx.x == 0) {
            a.tier[uw + w] = t;
            a.score[uw + w] = 0;
            a.has_ledger[uw + w] = (t == KVR_TIER_INT2) ? 1 : 0;
        }
        if (t == KVR_TIER_INT2) {
            const size_t row = (size_t)u * a.cap + (size_t)w * kWin;
            quantize_window<D>(K + row * D, V + row * D,
                               a.ledger + (uw + w) * (size_t)ledger_bytes_of(D), err);
        }
    }
}

__global__ void __launch_bounds__(kThreads) tier_count_kernel(TierArgs a, const int32_t *seq_len)
{
    __shared__ int64_t sh[2];
    const int u = blockIdx.x, b = u / a.Hkv;
    int64_t N = seq_len[b];
    if (N < 0 || N > a.cap) N = 0;
    const int64_t closed = N / kWin;
    if (threadIdx.x < 2) sh[threadIdx.x] = 0;
    __syncthreads();
    int nb = 0, nq = 0;
    for (int64_t w = threadIdx.x; w < closed; w += blockDim.x) {
        const int8_t t = a.tier[(size_t)u * a.n_win + w];
        nb += t == KVR_TIER_BF16;
        nq += t == KVR_TIER_INT2;
    }
    nb = warp_sum(nb);
    nq = warp_sum(nq);
    if ((threadIdx.x & 31) == 0) {
        atomicAdd(reinterpret_cast<unsigned long long *>(&sh[0]), (unsigned long long)nb);
        atomicAdd(reinterpret_cast<unsigned long long *>(&sh[1]), (unsigned long long)nq);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        a.quota[u] = (int32_t)sh[0];
        a.budget[u] = sh[0] * (int64_t)kWin * 4 * a.d + sh[1] * (int64_t)ledger_bytes_of(a.d);
    }
}

// ---------------------------------------------------------------- attention

struct TieredArgs {
    int Hkv, G;
    int64_t cap, n_win;
    int S;  // CTAs per unit
    const int8_t *tier;
    const uint8_t *ledger;
    const __nv_bfloat16 *q, *K, *V;
    const int32_t *seq_len;
    float scale_log2;  // scale * log2(e)
    float *part;       // [U, S, 2G + G*D]: m[G], l[G], o[G][D]
    float *lse;        // [U, n_win, G] log2-sum-exp of each window's scores (-inf: none)
    int32_t *err;
    uint64_t wait_ns;  // limit of each wait for a copy
    int withhold_last; // test hook: each CTA never issues its last copy (its wait runs out)
};

// Two 2-bit codes at bits 0-1 and 16-17 of t (the other bits ignored) as the
// bf16 pair (128 + c0, 128 + c1): 128 is 0x4300 in bf16 and its mantissa step
// is 1, so OR-ing a code into the low bits is exact (one LOP3). A product
// over such values carries 128 times the sum of the other operand, which the
// caller subtracts.
__device__ __forceinline__ uint32_t codes_off128(uint32_t t)
{
    return (t & 0x00030003u) | 0x43004300u;
}

// 2-D tensor-map copy of one box into shared memory, completing on `bar`
// (x: innermost coordinate in elements, a multiple of 8 for 2-byte elements).
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y,
                                            uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, "
        "{%2, %3}], [%4];\n" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

template <int D, int G> struct TieredCfg {
    static constexpr int RB = 2 * D;                   // bf16 row bytes
    static constexpr int NG = D / kQG;                 // INT2 groups per row
    static constexpr int LB = ledger_bytes_of(D);
    static constexpr int CB = kWin * NG * 8, PB = kWin * NG * 4;
    // staging ring: a slot holds the 64 K (or V) rows of a bf16 window as
    // 128-byte-swizzled boxes of 64 rows x 64 dims (TMA), or an INT2 window's
    // ledger (bulk copy); slots are filled ahead in window order
    static constexpr int SLOT = kWin * RB;
    static constexpr int NS = (D >= 128) ? 5 : 8;
    static constexpr int BOXES = D / 64;               // 128-byte column boxes per row
    static_assert(LB <= SLOT, "a ledger fits a slot");
    static constexpr int KS = D / 16;                  // k-steps of the score product
    static constexpr int MT = D / 16;                  // 16-dim tiles of the output
    static constexpr int NSTR = 2;                     // softmax streams: even / odd windows
    // P, and the scale-weighted P of each INT2 group, are kept as [token][8
    // heads] bf16 rows of 16 bytes (a hi and a lo array each): the output's B
    // operand for 16 tokens is one ldmatrix.x4.trans (hi and lo)
    static constexpr int PT = kWin * 8 * 2;                      // bytes of a [64][8] bf16 array
    static constexpr int oBar = NS * SLOT;                       // uint64 [NS]
    static constexpr int oP = oBar + 64;                         // [NSTR][hi, lo][64][8] bf16
    static constexpr int oSP = oP + NSTR * 2 * PT;               // [NSTR][NG][hi, lo][64][8] bf16
    static constexpr int oQp = oSP + NSTR * NG * 2 * PT;         // uint32 [KS][32 lanes][2]
    static constexpr int oMx = oQp + KS * 32 * 8;                // float [NSTR][4 tiles][8]
    static constexpr int oLs = oMx + NSTR * 4 * 8 * 4;           // float [NSTR][4 tiles][8]
    static constexpr int oZc = oLs + NSTR * 4 * 8 * 4;           // float [NSTR][4 tiles][NG][8]
    static constexpr int oQs = oZc + NSTR * 4 * NG * 8 * 4;      // float [NG][8]
    static constexpr int oSt = oQs + NG * 8 * 4;                 // float [NSTR][m, l, alpha, m_new][8]
    static constexpr int LMAX = 1024;                            // windows per listing pass
    static constexpr int oLive = oSt + NSTR * 4 * 8 * 4;         // int32 [LMAX]
    static constexpr int oCnt = oLive + LMAX * 4;                // int [8]
    static constexpr int bytes = oCnt + 8 * 4 + 1024;            // + alignment of the ring
    static_assert(G <= 8, "one 8-column tile of heads");
    static_assert(NS >= 4, "a pair of bf16 windows takes four slots");
    static_assert(8 * 32 * 4 * 4 <= NS * SLOT, "the d=64 stream merge fits the ring");
};

// Per pair of windows (stream 0 takes window ci, stream 1 window ci + 1) and
// three block barriers:
//   1. warp (stream, tile) scores its 16 tokens against the G heads on the
//      tensor cores (mma.sync m16n8k16, fp32 accumulate) and reduces their
//      maximum per head;
//   2. the same warp turns its scores into softmax weights against the
//      stream's running maximum, writes them (bf16 hi + lo) as the output's B
//      operand, and its partial sums per head; for an INT2 window also the
//      weights times each group's V scale and the group's zero and offset
//      terms;
//   3. warp (dim tile) accumulates O^T += V^T P^T for both streams; one warp
//      commits the streams' states and the windows' log2-sum-exps.
// INT2 codes enter the products as the bf16 values 128 + code (one shift and
// one LOP3 per pair of codes); the 128 times the other operand's sum is
// subtracted with the group's scale: a key's score over group g is
// s (codes . q) + z sum(q) = s (mma - 128 sum(q)) + z sum(q), and V's share
// is (s p) . codes + sum_t p z = mma(s p) - 128 sum_t (s p) + sum_t p z, with
// s p as the tensor core sees it (hi + lo). For the scores the k order inside
// each 16-channel step is permuted (k = 2c, 2c+1, 2c+8, 2c+9 of lane c are
// channels c, c+8, c+4, c+12: the code bits 2c and 2c+16 of one word), with
// the query permuted alike.
template <int D, int G>
__global__ void __launch_bounds__(kThreads, 2)
    tiered_attend_kernel(TieredArgs a, const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV)
{
    using C = TieredCfg<D, G>;
    extern __shared__ __align__(16) uint8_t smem_raw[];
    // the ring's 128-byte swizzle repeats every 1 KB: align its base to 1 KB
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *sBar = reinterpret_cast<uint64_t *>(smem + C::oBar);
    uint8_t *sP = smem + C::oP;
    uint8_t *sSP = smem + C::oSP;
    uint2 *sQp = reinterpret_cast<uint2 *>(smem + C::oQp);
    float *sMx = reinterpret_cast<float *>(smem + C::oMx);
    float *sLs = reinterpret_cast<float *>(smem + C::oLs);
    float *sZc = reinterpret_cast<float *>(smem + C::oZc);
    float *sQs = reinterpret_cast<float *>(smem + C::oQs);
    float *sSt = reinterpret_cast<float *>(smem + C::oSt);  // stream st: m at 32 st, l +8, alpha +16, m_new +24
    int32_t *sLive = reinterpret_cast<int32_t *>(smem + C::oLive);
    int *sCnt = reinterpret_cast<int *>(smem + C::oCnt);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int gq = lane >> 2, cq = lane & 3;  // fragment row group, column pair
    const int lm = lane >> 3, lr = lane & 7;  // ldmatrix: matrix, row
    const int x = blockIdx.x, u = blockIdx.y, b = u / a.Hkv, h = u % a.Hkv;
    int64_t N = a.seq_len[b];
    if (N < 0 || N > a.cap) {
        if (tid == 0 && x == 0) set_err(a.err, KVR_DEVERR_SEQ_LEN);
        N = 0;
    }
    const int64_t closed = N / kWin, nw = (N + kWin - 1) / kWin;
    const int64_t w_begin = nw * x / a.S, w_end = nw * (x + 1) / a.S;
    const size_t uw = (size_t)u * a.n_win;
    const int8_t *tier = a.tier + uw;
    const __nv_bfloat16 *qg = a.q + ((size_t)b * a.Hkv * G + (size_t)h * G) * D;
    const uint8_t *Lu = a.ledger + uw * (size_t)C::LB;

    // q as B fragments (column n = head gq; heads >= G are zero): in the
    // natural k order in registers (bf16 windows), in the permuted order of
    // the INT2 scores in shared memory
    uint32_t qf[C::KS][2];
#pragma unroll
    for (int ks = 0; ks < C::KS; ks++) {
        qf[ks][0] = qf[ks][1] = 0u;
        if (gq < G) {
            const uint32_t *row = reinterpret_cast<const uint32_t *>(qg + (size_t)gq * D);
            qf[ks][0] = row[(16 * ks + 2 * cq) / 2];
            qf[ks][1] = row[(16 * ks + 8 + 2 * cq) / 2];
        }
    }
    for (int i = tid; i < C::KS * 32; i += kThreads) {
        const int ks = i / 32, n = (i % 32) >> 2, c = i & 3;
        uint32_t v0 = 0u, v1 = 0u;
        if (n < G) {
            const uint16_t *row = reinterpret_cast<const uint16_t *>(qg + (size_t)n * D) + 16 * ks;
            v0 = (uint32_t)row[c] | ((uint32_t)row[c + 8] << 16);
            v1 = (uint32_t)row[c + 4] | ((uint32_t)row[c + 12] << 16);
        }
        sQp[i] = make_uint2(v0, v1);
    }
    // per-group sums of q (the zero's share of an INT2 score); stream states
    if (tid < C::NG * 8) {
        const int g = tid / 8, hh = tid % 8;
        float sum = 0.0f;
        if (hh < G)
            for (int j = 0; j < kQG; j++) sum += __bfloat162float(qg[(size_t)hh * D + g * kQG + j]);
        sQs[tid] = sum;
    }
    if (tid < C::NSTR * 8) {
        sSt[(tid / 8) * 32 + tid % 8] = -CUDART_INF_F;
        sSt[(tid / 8) * 32 + 8 + tid % 8] = 0.0f;
    }
    // set when a wait for a copy ran out: the CTA then stops after the
    // current pair of windows, waits (bounded) for the copies it issued and
    // leaves its (invalid) partial behind, KVR_DEVERR_TIMEOUT set
    __shared__ int s_dead;
    if (tid == 0) {
        for (int i = 0; i < C::NS; i++) mbar_init(&sBar[i], 1);
        mbar_fence_init();
        s_dead = 0;
    }
    __syncthreads();

    // output accumulators O^T (16 dims x 8 heads) per stream: d=128, warp w
    // owns dims 16w.. of both streams; d=64, warp w owns dims 16(w%4).. of
    // stream w/4
    constexpr bool BOTH = C::MT >= 8;
    const int mt_d = BOTH ? warp : (warp & 3);
    const int my_st = BOTH ? 0 : (warp >> 2);
    float acc[2][4] = {{0.0f, 0.0f, 0.0f, 0.0f}, {0.0f, 0.0f, 0.0f, 0.0f}};

    int li = 0, lc = 0;  // loads issued, loads consumed (block-uniform, across passes)
    bool dead = false;   // s_dead as read after a barrier (block-uniform)
    for (int64_t p0 = w_begin; p0 < w_end; p0 += C::LMAX) {
        const int64_t p1 = (p0 + C::LMAX < w_end) ? p0 + C::LMAX : w_end;
        // the live windows of [p0, p1) in order, bit 30 set for INT2 ones;
        // evicted windows get no mass (log2-sum-exp -inf)
        int nlive = 0;
        for (int64_t r0 = p0; r0 < p1; r0 += kThreads) {
            const int64_t w = r0 + tid;
            int code = -1;
            if (w < p1) {
                if (w >= closed) {
                    code = 0;  // the open window: bf16
                } else {
                    const int8_t t = checked_tier(tier[w], a.err);
                    if (t == KVR_TIER_EVICTED) {
#pragma unroll
                        for (int g = 0; g < G; g++) a.lse[(uw + w) * G + g] = -CUDART_INF_F;
                    } else {
                        code = (t == KVR_TIER_INT2) ? 1 : 0;
                    }
                }
            }
            __syncwarp();
            const unsigned bal = __ballot_sync(kFull, code >= 0);
            if (lane == 0) sCnt[warp] = __popc(bal);
            __syncthreads();
            int before = nlive, total = nlive;
#pragma unroll
            for (int ww = 0; ww < kThreads / 32; ww++) {
                before += (ww < warp) ? sCnt[ww] : 0;
                total += sCnt[ww];
            }
            if (code >= 0)
                sLive[before + __popc(bal & ((1u << lane) - 1u))] = (int32_t)w | (code << 30);
            nlive = total;
            __syncthreads();
        }

        // Loads in list order: a bf16 (or the open) window is two loads (its 64
        // K rows, then its 64 V rows, as 128-byte-swizzled tensor-map boxes),
        // an INT2 window one (its ledger, one bulk copy). Load L fills slot
        // L % NS and completes phase (L / NS) & 1 of that slot's barrier; one
        // thread issues, up to NS loads ahead of the consumer.
        int pi = 0, ppart = 0;  // producer: list position, next part (0 K / ledger, 1 V)
        auto issue_ahead = [&]() {
            while (li - lc < C::NS && pi < nlive) {
                const int32_t e = sLive[pi];
                const int64_t pw = e & 0x3fffffff;
                const int slot = li % C::NS;
                uint8_t *dst = smem + slot * C::SLOT;
                const bool q2 = (e >> 30) & 1;
                const bool withheld =
                    a.withhold_last && p1 == w_end && pi == nlive - 1 && (q2 || ppart);
                if (tid == 0 && !withheld) {
                    fence_proxy_async();  // earlier reads of the slot before the async writes
                    if (q2) {
                        mbar_arrive_expect_tx(&sBar[slot], C::LB);
                        bulk_g2s(dst, Lu + (size_t)pw * C::LB, C::LB, &sBar[slot]);
                    } else {
                        mbar_arrive_expect_tx(&sBar[slot], C::SLOT);
                        const int y = (int)((int64_t)u * a.cap + pw * kWin);
#pragma unroll
                        for (int bx = 0; bx < C::BOXES; bx++)
                            tma_load_2d(dst + bx * kWin * 128, ppart ? &tmV : &tmK, 64 * bx, y,
                                        &sBar[slot]);
                    }
                }
                if (q2) {
                    pi++;
                } else if (ppart) {
                    ppart = 0;
                    pi++;
                } else {
                    ppart = 1;
                }
                li++;
            }
        };

        for (int ci = 0; ci < nlive; ci += 2) {
            const bool hasB = ci + 1 < nlive;
            // per window (A: stream 0, B: stream 1) as scalars, picked with
            // selects: an array indexed by a warp-dependent stream would live
            // in local memory
            const int32_t eA = sLive[ci], eB = hasB ? sLive[ci + 1] : 0;
            const bool q2A = ((eA >> 30) & 1) != 0, q2B = hasB && ((eB >> 30) & 1) != 0;
            const int64_t cwA = eA & 0x3fffffff, cwB = eB & 0x3fffffff;
            const int needA = q2A ? 1 : 2;
            const int needB = hasB ? (q2B ? 1 : 2) : 0;
            const int slA = lc, slB = lc + needA;  // first load of each window
            const int nvA = (int)(N - cwA * kWin < kWin ? N - cwA * kWin : kWin);
            const int nvB = (int)(N - cwB * kWin < kWin ? N - cwB * kWin : kWin);
            issue_ahead();
            for (int L = lc; L < lc + needA + needB; L++)
                if (!mbar_wait(&sBar[L % C::NS], (uint32_t)((L / C::NS) & 1), a.err, a.wait_ns))
                    s_dead = 1;
#pragma unroll
            for (int st = 0; st < 2; st++) {
                const bool q2s = st ? q2B : q2A;
                const int nvs = st ? nvB : nvA, sls = st ? slB : slA;
                // rows past the sequence in the open window: whatever the cache
                // holds there must not reach the sum (0 * NaN), so zero them in
                // V (their scores are -inf by index); read after the barrier below
                if ((st == 0 || hasB) && !q2s && nvs < kWin) {
                    uint8_t *vb = smem + ((sls + 1) % C::NS) * C::SLOT;
                    const int nz = kWin - nvs;
                    for (int i = tid; i < C::BOXES * nz * 8; i += kThreads) {
                        const int bx = i / (nz * 8), rem = i % (nz * 8);
                        *reinterpret_cast<uint4 *>(vb + bx * kWin * 128 + (nvs + rem / 8) * 128 +
                                                   (rem % 8) * 16) = make_uint4(0u, 0u, 0u, 0u);
                    }
                }
            }

            // ---- 1. scores: warp -> window (warp / 4), 16 tokens (warp % 4), all dims
            const int st = warp >> 2, mt = warp & 3;
            const bool act = st == 0 || hasB;
            const bool q2s = st ? q2B : q2A;
            const int nvs = st ? nvB : nvA;
            const uint8_t *kbuf = smem + ((st ? slB : slA) % C::NS) * C::SLOT;
            const int t0 = 16 * mt + gq;  // the lane's tokens t0, t0 + 8; heads 2cq, 2cq + 1
            float sc[4] = {-CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F};
            if (act) {
                float c4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                if (!q2s) {
                    // row r, 16-byte chunk c of a box sits at r*128 + ((c ^ (r % 8)) * 16);
                    // even and odd k-steps in two accumulators (two shorter chains)
                    const uint8_t *rowp = kbuf + (16 * mt + lr + ((lm & 1) ? 8 : 0)) * 128;
                    float c4b[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                    for (int ks = 0; ks < C::KS; ks++) {
                        const int ch = 2 * ks + ((lm & 2) ? 1 : 0);
                        uint32_t af[4];
                        ldsm_x4(af, rowp + (ch >> 3) * kWin * 128 + (((ch & 7) ^ lr) << 4));
                        mma16816((ks & 1) ? c4b : c4, af, qf[ks][0], qf[ks][1]);
                    }
#pragma unroll
                    for (int i = 0; i < 4; i++) c4[i] += c4b[i];
                } else {
                    const int r1 = t0 + 8;
#pragma unroll
                    for (int g = 0; g < C::NG; g++) {
                        const uint2 w0 = *reinterpret_cast<const uint2 *>(kbuf + (t0 * C::NG + g) * 8);
                        const uint2 w1 = *reinterpret_cast<const uint2 *>(kbuf + (r1 * C::NG + g) * 8);
                        float cg[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                        for (int j = 0; j < 2; j++) {
                            const uint32_t x0 = j ? w0.y : w0.x, x1 = j ? w1.y : w1.x;
                            uint32_t af[4];
                            af[0] = codes_off128(x0 >> (2 * cq));
                            af[1] = codes_off128(x1 >> (2 * cq));
                            af[2] = codes_off128(x0 >> (2 * cq + 8));
                            af[3] = codes_off128(x1 >> (2 * cq + 8));
                            const uint2 qp = sQp[(2 * g + j) * 32 + lane];
                            mma16816(cg, af, qp.x, qp.y);
                        }
                        const uint32_t pa = *reinterpret_cast<const uint32_t *>(kbuf + C::CB + (t0 * C::NG + g) * 4);
                        const uint32_t pb = *reinterpret_cast<const uint32_t *>(kbuf + C::CB + (r1 * C::NG + g) * 4);
                        const float s0f = __half2float(__ushort_as_half((unsigned short)(pa & 0xffffu)));
                        const float z0f = __half2float(__ushort_as_half((unsigned short)(pa >> 16)));
                        const float s1f = __half2float(__ushort_as_half((unsigned short)(pb & 0xffffu)));
                        const float z1f = __half2float(__ushort_as_half((unsigned short)(pb >> 16)));
                        const float qa = sQs[g * 8 + 2 * cq], qb = sQs[g * 8 + 2 * cq + 1];
                        const float y0 = fmaf(-128.0f, s0f, z0f), y1 = fmaf(-128.0f, s1f, z1f);
                        c4[0] += fmaf(s0f, cg[0], y0 * qa);
                        c4[1] += fmaf(s0f, cg[1], y0 * qb);
                        c4[2] += fmaf(s1f, cg[2], y1 * qa);
                        c4[3] += fmaf(s1f, cg[3], y1 * qb);
                    }
                }
                // log2-domain scores; rows past the sequence (open window) -inf
                if (t0 < nvs) {
                    sc[0] = c4[0] * a.scale_log2;
                    sc[1] = c4[1] * a.scale_log2;
                }
                if (t0 + 8 < nvs) {
                    sc[2] = c4[2] * a.scale_log2;
                    sc[3] = c4[3] * a.scale_log2;
                }
                float ma = fmaxf(sc[0], sc[2]), mb = fmaxf(sc[1], sc[3]);
                __syncwarp();
#pragma unroll
                for (int o = 4; o < 32; o <<= 1) {
                    ma = fmaxf(ma, __shfl_xor_sync(kFull, ma, o));
                    mb = fmaxf(mb, __shfl_xor_sync(kFull, mb, o));
                }
                if (gq == 0) {
                    sMx[(st * 4 + mt) * 8 + 2 * cq] = ma;
                    sMx[(st * 4 + mt) * 8 + 2 * cq + 1] = mb;
                }
            }
            __syncthreads();
            // every write of s_dead (the waits above) precedes this read, every
            // later one follows the pair's last barrier: `dead` is block-uniform
            dead = s_dead != 0;

            // ---- 2. softmax weights of the warp's tokens, B operands of the output
            if (act) {
                const int ha = 2 * cq, hb = ha + 1;
                float *stt = sSt + st * 32;
                float mwa = sMx[st * 32 + ha], mwb = sMx[st * 32 + hb];
#pragma unroll
                for (int m2 = 1; m2 < 4; m2++) {
                    mwa = fmaxf(mwa, sMx[(st * 4 + m2) * 8 + ha]);
                    mwb = fmaxf(mwb, sMx[(st * 4 + m2) * 8 + hb]);
                }
                const float ma_old = stt[ha], mb_old = stt[hb];
                const float ma_new = fmaxf(ma_old, mwa), mb_new = fmaxf(mb_old, mwb);
                // heads past G weigh nothing
                const bool va = ha < G, vb = hb < G;
                float p[4];
                p[0] = (va && sc[0] != -CUDART_INF_F) ? exp2f(sc[0] - ma_new) : 0.0f;
                p[1] = (vb && sc[1] != -CUDART_INF_F) ? exp2f(sc[1] - mb_new) : 0.0f;
                p[2] = (va && sc[2] != -CUDART_INF_F) ? exp2f(sc[2] - ma_new) : 0.0f;
                p[3] = (vb && sc[3] != -CUDART_INF_F) ? exp2f(sc[3] - mb_new) : 0.0f;
                float la = p[0] + p[2], lb = p[1] + p[3];
#pragma unroll
                for (int o = 4; o < 32; o <<= 1) {
                    la += __shfl_xor_sync(kFull, la, o);
                    lb += __shfl_xor_sync(kFull, lb, o);
                }
                if (gq == 0) {
                    sLs[(st * 4 + mt) * 8 + ha] = la;
                    sLs[(st * 4 + mt) * 8 + hb] = lb;
                    if (mt == 0) {  // the stream's new maximum and rescale factor
                        stt[24 + ha] = ma_new;
                        stt[24 + hb] = mb_new;
                        stt[16 + ha] = (ma_old == -CUDART_INF_F) ? 0.0f : exp2f(ma_old - ma_new);
                        stt[16 + hb] = (mb_old == -CUDART_INF_F) ? 0.0f : exp2f(mb_old - mb_new);
                    }
                }
                // P (hi, lo) at [token][head]: this lane's heads ha, hb of t0 and t0 + 8
                uint8_t *pst = sP + st * 2 * C::PT;
                uint32_t hi, lo;
                float r0, r1;
                split_bf16x2(p[0], p[1], hi, lo, r0, r1);
                *reinterpret_cast<uint32_t *>(pst + t0 * 16 + 4 * cq) = hi;
                *reinterpret_cast<uint32_t *>(pst + C::PT + t0 * 16 + 4 * cq) = lo;
                split_bf16x2(p[2], p[3], hi, lo, r0, r1);
                *reinterpret_cast<uint32_t *>(pst + (t0 + 8) * 16 + 4 * cq) = hi;
                *reinterpret_cast<uint32_t *>(pst + C::PT + (t0 + 8) * 16 + 4 * cq) = lo;
                if (q2s) {
                    // V values are code * s + z per (token, group): the output
                    // takes B = s p (hi, lo) per group, and adds this group's
                    // sum_t (p z - 128 (s p as seen))
                    const uint8_t *vp = kbuf + 2 * C::CB + C::PB;  // V params
#pragma unroll
                    for (int g = 0; g < C::NG; g++) {
                        const uint32_t q0 = *reinterpret_cast<const uint32_t *>(vp + (t0 * C::NG + g) * 4);
                        const uint32_t q1 = *reinterpret_cast<const uint32_t *>(vp + ((t0 + 8) * C::NG + g) * 4);
                        const float s0 = __half2float(__ushort_as_half((unsigned short)(q0 & 0xffffu)));
                        const float z0 = __half2float(__ushort_as_half((unsigned short)(q0 >> 16)));
                        const float s1 = __half2float(__ushort_as_half((unsigned short)(q1 & 0xffffu)));
                        const float z1 = __half2float(__ushort_as_half((unsigned short)(q1 >> 16)));
                        uint8_t *spg = sSP + (size_t)(st * C::NG + g) * 2 * C::PT;
                        float e0, e1, e2, e3;
                        split_bf16x2(s0 * p[0], s0 * p[1], hi, lo, e0, e1);
                        *reinterpret_cast<uint32_t *>(spg + t0 * 16 + 4 * cq) = hi;
                        *reinterpret_cast<uint32_t *>(spg + C::PT + t0 * 16 + 4 * cq) = lo;
                        split_bf16x2(s1 * p[2], s1 * p[3], hi, lo, e2, e3);
                        *reinterpret_cast<uint32_t *>(spg + (t0 + 8) * 16 + 4 * cq) = hi;
                        *reinterpret_cast<uint32_t *>(spg + C::PT + (t0 + 8) * 16 + 4 * cq) = lo;
                        float za = fmaf(z0, p[0], fmaf(z1, p[2], -128.0f * (e0 + e2)));
                        float zb = fmaf(z0, p[1], fmaf(z1, p[3], -128.0f * (e1 + e3)));
#pragma unroll
                        for (int o = 4; o < 32; o <<= 1) {
                            za += __shfl_xor_sync(kFull, za, o);
                            zb += __shfl_xor_sync(kFull, zb, o);
                        }
                        if (gq == 0) {
                            sZc[((st * 4 + mt) * C::NG + g) * 8 + ha] = za;
                            sZc[((st * 4 + mt) * C::NG + g) * 8 + hb] = zb;
                        }
                    }
                }
            }
            __syncthreads();

            // ---- 3. output: O^T (dims x heads) += V^T P^T, per stream
#pragma unroll
            for (int so = 0; so < 2; so++) {
                if (!BOTH && so != my_st) continue;
                if (so == 1 && !hasB) continue;
                float *ac = acc[BOTH ? so : 0];
                const float *stt = sSt + so * 32;
                const float al0 = (2 * cq < G) ? stt[16 + 2 * cq] : 0.0f;
                const float al1 = (2 * cq + 1 < G) ? stt[16 + 2 * cq + 1] : 0.0f;
                ac[0] *= al0;
                ac[1] *= al1;
                ac[2] *= al0;
                ac[3] *= al1;
                const int sls = so ? slB : slA;
                // B operand rows: matrices hi t..t+7, hi t+8.., lo t.., lo t+8..
                const int brow = (lm & 1) * 8 + lr, bpart = (lm & 2) ? C::PT : 0;
                if (!(so ? q2B : q2A)) {
                    const uint8_t *pst = sP + so * 2 * C::PT + bpart + brow * 16;
                    const uint8_t *vbuf = smem + ((sls + 1) % C::NS) * C::SLOT;
                    const int ch = 2 * mt_d + ((lm & 1) ? 1 : 0);
                    const uint8_t *vrow = vbuf + (ch >> 3) * kWin * 128 +
                                          (lr + ((lm & 2) ? 8 : 0)) * 128 + (((ch & 7) ^ lr) << 4);
                    // the lo products in their own accumulator: two chains of 4
                    float lo4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                    for (int j = 0; j < 4; j++) {
                        uint32_t af[4], bq[4];
                        ldsm_x4_t(af, vrow + 16 * j * 128);
                        ldsm_x4_t(bq, pst + 16 * j * 16);
                        mma16816(*reinterpret_cast<float(*)[4]>(ac), af, bq[0], bq[1]);
                        mma16816(lo4, af, bq[2], bq[3]);
                    }
#pragma unroll
                    for (int i = 0; i < 4; i++) ac[i] += lo4[i];
                } else {
                    const uint8_t *buf = smem + (sls % C::NS) * C::SLOT;
                    const int g = (16 * mt_d) / kQG, wsel = ((16 * mt_d) % kQG) / 16;
                    const uint8_t *vc = buf + C::CB + C::PB + 4 * wsel;  // V codes of the tile
                    const uint8_t *spg = sSP + (size_t)(so * C::NG + g) * 2 * C::PT + bpart + brow * 16;
                    float lo4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                    for (int j = 0; j < 4; j++) {
                        const int ta = 16 * j + 2 * cq;
                        const uint32_t wa = *reinterpret_cast<const uint32_t *>(vc + (ta * C::NG + g) * 8);
                        const uint32_t wb = *reinterpret_cast<const uint32_t *>(vc + ((ta + 1) * C::NG + g) * 8);
                        const uint32_t wc = *reinterpret_cast<const uint32_t *>(vc + ((ta + 8) * C::NG + g) * 8);
                        const uint32_t wd = *reinterpret_cast<const uint32_t *>(vc + ((ta + 9) * C::NG + g) * 8);
                        // the tile's channels 0-7 of two tokens in the halves of
                        // one word, channels 8-15 in another
                        const uint32_t ab0 = __byte_perm(wa, wb, 0x5410), ab1 = __byte_perm(wa, wb, 0x7632);
                        const uint32_t cd0 = __byte_perm(wc, wd, 0x5410), cd1 = __byte_perm(wc, wd, 0x7632);
                        uint32_t af[4], bq[4];
                        af[0] = codes_off128(ab0 >> (2 * gq));  // dim gq, tokens ta, ta + 1
                        af[1] = codes_off128(ab1 >> (2 * gq));  // dim gq + 8
                        af[2] = codes_off128(cd0 >> (2 * gq));  // dim gq, tokens ta + 8, ta + 9
                        af[3] = codes_off128(cd1 >> (2 * gq));
                        ldsm_x4_t(bq, spg + 16 * j * 16);
                        mma16816(*reinterpret_cast<float(*)[4]>(ac), af, bq[0], bq[1]);
                        mma16816(lo4, af, bq[2], bq[3]);
                    }
                    float za = 0.0f, zb = 0.0f;
#pragma unroll
                    for (int m2 = 0; m2 < 4; m2++) {
                        za += sZc[((so * 4 + m2) * C::NG + g) * 8 + 2 * cq];
                        zb += sZc[((so * 4 + m2) * C::NG + g) * 8 + 2 * cq + 1];
                    }
                    ac[0] += lo4[0] + za;
                    ac[1] += lo4[1] + zb;
                    ac[2] += lo4[2] + za;
                    ac[3] += lo4[3] + zb;
                }
            }
            // the streams' states (the rescale factors above were read from
            // their own slots) and the windows' log2-sum-exps
            if (warp == kThreads / 32 - 1) {
                const int so = lane >> 3, hh = lane & 7;
                if (hh < G && (so == 0 || (so == 1 && hasB))) {
                    float *stt = sSt + so * 32;
                    float ls = 0.0f;
#pragma unroll
                    for (int m2 = 0; m2 < 4; m2++) ls += sLs[(so * 4 + m2) * 8 + hh];
                    const float mn = stt[24 + hh];
                    stt[8 + hh] = stt[8 + hh] * stt[16 + hh] + ls;
                    stt[hh] = mn;
                    a.lse[(uw + (so ? cwB : cwA)) * G + hh] = mn + log2f(ls);
                }
            }
            fence_proxy_async();  // this thread's slot accesses before the next copies into it
            __syncthreads();      // the pair's slots, P and the states are reused next
            lc += needA + needB;
            if (dead) break;
        }
        if (dead) break;
    }
    if (dead)  // copies issued ahead of the pair that timed out
        for (int L = lc; L < li; L++)
            mbar_wait(&sBar[L % C::NS], (uint32_t)((L / C::NS) & 1), a.err, a.wait_ns);
    __syncthreads();

    // ---- merge the two streams into this CTA's partial: o[head][dim]
    // (unnormalised), m, l per head
    float *part = a.part + ((size_t)u * a.S + x) * (2 * G + G * D);
    auto factor = [&](int st2, int hh) {  // weight of stream st2's head hh in the merge
        const float m0 = sSt[hh], m1 = sSt[32 + hh];
        const float M = fmaxf(m0, m1);
        const float m = st2 ? m1 : m0;
        return (m == -CUDART_INF_F) ? 0.0f : exp2f(m - M);
    };
    if (!BOTH) {
        // d = 64: stream 1's warps hand their tiles to stream 0's warps
        float *red = reinterpret_cast<float *>(smem);
        if (my_st == 1)
            *reinterpret_cast<float4 *>(red + (mt_d * 32 + lane) * 4) =
                make_float4(acc[0][0], acc[0][1], acc[0][2], acc[0][3]);
        __syncthreads();
        if (my_st == 0) {
            const float4 o = *reinterpret_cast<const float4 *>(red + (mt_d * 32 + lane) * 4);
            acc[1][0] = o.x;
            acc[1][1] = o.y;
            acc[1][2] = o.z;
            acc[1][3] = o.w;
        }
    }
    if (my_st == 0) {
        const int d0 = 16 * mt_d + gq;
#pragma unroll
        for (int e = 0; e < 2; e++) {
            const int hh = 2 * cq + e;
            if (hh < G) {
                const float f0 = factor(0, hh), f1 = factor(1, hh);
                part[2 * G + hh * D + d0] = acc[0][e] * f0 + acc[1][e] * f1;
                part[2 * G + hh * D + d0 + 8] = acc[0][2 + e] * f0 + acc[1][2 + e] * f1;
            }
        }
    }
    if (tid < G) {
        const float m0 = sSt[tid], m1 = sSt[32 + tid];
        part[tid] = fmaxf(m0, m1);
        part[G + tid] = sSt[8 + tid] * factor(0, tid) + sSt[40 + tid] * factor(1, tid);
    }
}

template <int D, int G>
__global__ void __launch_bounds__(kThreads) tiered_combine_kernel(TieredArgs a, float *out,
                                                                  float *mass)
{
    // the partials' (m, l) are read into shared memory by all threads at
    // once (a chain of dependent global loads per head was the kernel's
    // length), then the weights 2^(m - M) are kept there for the outputs
    extern __shared__ float sDyn[];  // [S][G] m, then weights; [S][G] l
    __shared__ float sM[16], sL[16];
    const int u = blockIdx.x, b = u / a.Hkv, h = u % a.Hkv, tid = threadIdx.x;
    int64_t N = a.seq_len[b];
    if (N < 0 || N > a.cap) N = 0;
    const int64_t nw = (N + kWin - 1) / kWin;
    const float *part = a.part + (size_t)u * a.S * (2 * G + G * D);
    constexpr int PS = 2 * G + G * D;
    float *sF = sDyn, *sLp = sDyn + a.S * G;
    for (int i = tid; i < a.S * G; i += kThreads) {
        const int x = i / G, g = i - x * G;
        sF[i] = part[x * PS + g];
        sLp[i] = part[x * PS + G + g];
    }
    __syncthreads();
    if (tid < G) {
        float M = -CUDART_INF_F;
        for (int x = 0; x < a.S; x++) M = fmaxf(M, sF[x * G + tid]);
        float L = 0.0f;
        if (M != -CUDART_INF_F)
            for (int x = 0; x < a.S; x++) {
                const float m = sF[x * G + tid];
                if (m != -CUDART_INF_F) L += sLp[x * G + tid] * exp2f(m - M);
            }
        sM[tid] = M;
        sL[tid] = L;
    }
    __syncthreads();
    // weights (0 for a split without tokens: its partial output is zero)
    for (int i = tid; i < a.S * G; i += kThreads) {
        const float m = sF[i];
        sF[i] = (m == -CUDART_INF_F) ? 0.0f : exp2f(m - sM[i % G]);
    }
    __syncthreads();
    for (int i = tid; i < G * D; i += kThreads) {
        const int g = i / D;
        const float L = sL[g];
        float o = 0.0f;
        if (L > 0.0f) {
#pragma unroll 4
            for (int x = 0; x < a.S; x++) o += part[x * PS + 2 * G + i] * sF[x * G + g];
            o /= L;
        }
        out[((size_t)b * a.Hkv * G + (size_t)h * G) * D + i] = o;
    }
    const size_t uw = (size_t)u * a.n_win;
#pragma unroll 4
    for (int64_t w = tid; w < a.n_win; w += kThreads) {
        float m = 0.0f;
        if (w < nw) {
#pragma unroll
            for (int g = 0; g < G; g++) {
                const float l = a.lse[(uw + w) * G + g];
                if (sL[g] > 0.0f && l != -CUDART_INF_F) m += exp2f(l - sM[g]) / sL[g];
            }
        }
        mass[uw + w] = m;
    }
}

// ---------------------------------------------------------------- routing

struct RankArgs {
    TierArgs t;
    const float *mass;
    const int32_t *seq_len;
    int32_t *stats;     // [U, 3] or null
    int32_t *moves;     // [U, n_win]: window | kind << 30 (kind 0 quantise, 1 dequantise)
    int32_t *n_moves;   // [U]
    int32_t *err;
    int P;              // sort length: a power of two >= n_win
};

// Rank order: score descending, window ascending.
__device__ __forceinline__ bool before(int64_t sa, int wa, int64_t sb, int wb)
{
    return sa > sb || (sa == sb && wa < wb);
}

__global__ void __launch_bounds__(kRankThreads) tier_rank_kernel(RankArgs r)
{
    extern __shared__ __align__(16) uint8_t smem[];
    int64_t *key = reinterpret_cast<int64_t *>(smem);
    int32_t *win = reinterpret_cast<int32_t *>(smem + (size_t)r.P * 8);
    __shared__ int s_live, s_stat[3], s_moves;
    const TierArgs &a = r.t;
    const int u = blockIdx.x, b = u / a.Hkv, tid = threadIdx.x;
    int64_t N = r.seq_len[b];
    const bool ok = N >= 0 && N <= a.cap;
    if (!ok) {
        if (tid == 0) {
            set_err(r.err, KVR_DEVERR_SEQ_LEN);
            r.n_moves[u] = 0;
            if (r.stats) r.stats[u * 3] = r.stats[u * 3 + 1] = r.stats[u * 3 + 2] = 0;
        }
        return;
    }
    const int64_t closed = N / kWin, nw = (N + kWin - 1) / kWin;
    const size_t uw = (size_t)u * a.n_win;
    if (tid == 0) {
        s_live = 0;
        s_stat[0] = s_stat[1] = s_stat[2] = 0;
        s_moves = 0;
    }
    __syncthreads();
    // 1. scores; 2. collect the live closed windows (one shared-memory
    // atomic per warp and round: ballot, then each lane's rank in the warp)
    const int lane = tid & 31;
    for (int64_t w0 = 0; w0 < nw; w0 += kRankThreads) {
        const int64_t w = w0 + tid;
        bool take = false;
        int64_t sc = 0;
        if (w < nw) {
            const int8_t t = checked_tier(a.tier[uw + w], r.err);
            if (t != KVR_TIER_EVICTED) {
                sc = a.score[uw + w] + __float2ll_rn(r.mass[uw + w] * 4294967296.0f);
                a.score[uw + w] = sc;
                take = w < closed;
            }
        }
        __syncwarp();
        const unsigned bal = __ballot_sync(kFull, take);
        int base = 0;
        if (lane == 0 && bal) base = atomicAdd(&s_live, __popc(bal));
        base = __shfl_sync(kFull, base, 0);
        if (take) {
            const int i = base + __popc(bal & ((1u << lane) - 1u));
            key[i] = sc;
            win[i] = (int32_t)w;
        }
    }
    __syncthreads();
    const int live = s_live;
    int P = 2;  // sort length: the next power of two of the live count
    while (P < live) P <<= 1;
    for (int i = live + tid; i < P; i += kRankThreads) {
        key[i] = INT64_MIN;
        win[i] = INT32_MAX;
    }
    __syncthreads();
    // bitonic sort of [0, P) into rank order; the pair (i, i ^ j) goes to
    // the thread of the lower index, so while consecutive stages have j < 32
    // every element a stage reads was written in the same warp: those stages
    // are separated by a warp barrier only
    for (int k = 2; k <= P; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = tid; i < P; i += kRankThreads) {
                const int l = i ^ j;
                if (l > i) {
                    const bool up = (i & k) == 0;  // this block in rank order
                    const bool lfirst = before(key[l], win[l], key[i], win[i]);
                    if (lfirst == up) {
                        const int64_t tk = key[i];
                        key[i] = key[l];
                        key[l] = tk;
                        const int32_t tw = win[i];
                        win[i] = win[l];
                        win[l] = tw;
                    }
                }
            }
            // the next stage: (k, j / 2), or (2k, k) when j == 1
            const int jn = (j > 1) ? (j >> 1) : k;
            if (j < 32 && jn < 32) __syncwarp();
            else __syncthreads();
        }
    }
    __syncthreads();
    // 3. new tiers and 4. moves
    const int64_t quota = a.quota[u], budget = a.budget[u];
    const int64_t BFB = (int64_t)kWin * 4 * a.d, LBB = ledger_bytes_of(a.d);
    const int64_t n_bf = quota < live ? quota : live, n_q = live - n_bf;
    const int64_t bytes = n_bf * BFB + n_q * LBB;
    int64_t n_ev = 0;
    if (bytes > budget) {
        const int64_t need = (bytes - budget + LBB - 1) / LBB;
        n_ev = need < n_q ? need : n_q;
    }
    for (int i = tid; i < live; i += kRankThreads) {
        const int w = win[i];
        const int8_t to = i < n_bf ? KVR_TIER_BF16
                                   : (i >= live - n_ev ? KVR_TIER_EVICTED : KVR_TIER_INT2);
        const int8_t from = a.tier[uw + w];
        if (from == to) continue;
        a.tier[uw + w] = to;
        if (to == KVR_TIER_EVICTED) {
            atomicAdd(&s_stat[2], 1);
        } else if (to == KVR_TIER_INT2) {
            atomicAdd(&s_stat[1], 1);
            if (!a.has_ledger[uw + w]) {
                a.has_ledger[uw + w] = 1;
                r.moves[uw + atomicAdd(&s_moves, 1)] = w;
            }
        } else {
            atomicAdd(&s_stat[0], 1);
            r.moves[uw + atomicAdd(&s_moves, 1)] = w | (1 << 30);
        }
    }
    __syncthreads();
    if (tid == 0) {
        r.n_moves[u] = s_moves;
        if (r.stats) {
            r.stats[u * 3] = s_stat[0];
            r.stats[u * 3 + 1] = s_stat[1];
            r.stats[u * 3 + 2] = s_stat[2];
        }
    }
}

template <int D>
__global__ void __launch_bounds__(kThreads) tier_move_kernel(TierArgs a, const int32_t *moves,
                                                             const int32_t *n_moves,
                                                             __nv_bfloat16 *K, __nv_bfloat16 *V,
                                                             int32_t *err)
{
    const int u = blockIdx.y;
    const size_t uw = (size_t)u * a.n_win;
    const int n = min(max(n_moves[u], 0), (int)a.n_win);
    for (int i = blockIdx.x; i < n; i += gridDim.x) {
        const int32_t e = moves[uw + i];
        const int64_t w = e & ((1 << 30) - 1);
        if (e < 0 || (w + 1) * kWin > a.cap) {  // never written by the ranking
            if (threadIdx.x == 0) set_err(err, KVR_DEVERR_INDEX);
            continue;
        }
        const size_t row = (size_t)u * a.cap + (size_t)w * kWin;
        uint8_t *lg = a.ledger + (uw + w) * (size_t)ledger_bytes_of(D);
        if (e >> 30) dequantize_window<D>(lg, K + row * D, V + row * D);
        else quantize_window<D>(K + row * D, V + row * D, lg, err);
    }
}

int tiered_splits(int64_t U, int64_t n_win)
{
    const int64_t target = (4 * (int64_t)sm_count() + U - 1) / U;
    const int64_t by_len = (n_win + 7) / 8;
    const int64_t s = target < by_len ? target : by_len;
    return (int)(s < 1 ? 1 : s);
}

TierArgs tier_args(const LaunchCtx &c, const kvr_tier_state &s)
{
    TierArgs a;
    a.Hkv = c.shape.Hkv;
    a.d = c.shape.d;
    a.cap = c.shape.cap;
    a.n_win = s.n_win;
    a.tier = s.tier;
    a.score = s.score;
    a.has_ledger = s.has_ledger;
    a.ledger = s.ledger;
    a.quota = s.quota;
    a.budget = s.budget;
    return a;
}

}  // namespace

size_t tiered_attend_ws_bytes(const kvr_shape &s, int64_t n_win)
{
    const int64_t U = (int64_t)s.B * s.Hkv;
    const int G = s.Hq / s.Hkv;
    const int S = tiered_splits(U, n_win);
    return align_up((size_t)U * S * (2 * G + G * s.d) * 4, 256) +
           align_up((size_t)U * n_win * G * 4, 256);
}

size_t tier_update_ws_bytes(const kvr_shape &s, int64_t n_win)
{
    const int64_t U = (int64_t)s.B * s.Hkv;
    return align_up((size_t)U * n_win * 4, 256) + align_up((size_t)U * 4, 256);
}

kvr_status tier_init_dispatch(const LaunchCtx &c, const kvr_tier_state &s, const int8_t *init,
                              const void *K, const void *V, const int32_t *seq_len, int32_t *err)
{
    const TierArgs a = tier_args(c, s);
    const int U = c.shape.B * c.shape.Hkv;
    const dim3 grid((unsigned)(s.n_win < kInitX ? s.n_win : kInitX), (unsigned)U);
    const auto *Kb = static_cast<const __nv_bfloat16 *>(K);
    const auto *Vb = static_cast<const __nv_bfloat16 *>(V);
    if (c.shape.d == 128)
        tier_init_kernel<128><<<grid, kThreads, 0, c.stream>>>(a, init, Kb, Vb, seq_len, err);
    else
        tier_init_kernel<64><<<grid, kThreads, 0, c.stream>>>(a, init, Kb, Vb, seq_len, err);
    if (check_launch() != KVR_OK) return KVR_ERR_CUDA;
    tier_count_kernel<<<U, kThreads, 0, c.stream>>>(a, seq_len);
    return check_launch();
}

// cuTensorMapEncodeTiled from the driver, looked up once.
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return (PFN_cuTensorMapEncodeTiled_v12000) nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }();
    return fn;
}

// Tensor map of a bf16 cache viewed as rows x d elements: boxes of 64 rows x
// 64 dims (128 bytes) with the 128-byte swizzle; rows past the end read as zero.
static bool rows_map(CUtensorMap *m, const void *base, int d, uint64_t rows)
{
    const PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)d * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)kWin};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, int G>
static kvr_status tiered_launch(const LaunchCtx &c, TieredArgs a, float *out, float *mass)
{
    using C = TieredCfg<D, G>;
    const void *k = reinterpret_cast<const void *>(&tiered_attend_kernel<D, G>);
    kvr_status st = raise_smem_limit(k, C::bytes);
    if (st != KVR_OK) return st;
    const int U = c.shape.B * c.shape.Hkv;
    CUtensorMap tmK, tmV;
    const uint64_t rows = (uint64_t)U * (uint64_t)c.shape.cap;
    if (!rows_map(&tmK, a.K, D, rows) || !rows_map(&tmV, a.V, D, rows)) return KVR_ERR_CUDA;
    tiered_attend_kernel<D, G><<<dim3(a.S, U), kThreads, C::bytes, c.stream>>>(a, tmK, tmV);
    if (check_launch() != KVR_OK) return KVR_ERR_CUDA;  // the combine reads its partials
    const int csmem = 2 * a.S * G * (int)sizeof(float);
    if (raise_smem_limit(reinterpret_cast<const void *>(&tiered_combine_kernel<D, G>), csmem) != KVR_OK)
        return KVR_ERR_CUDA;
    tiered_combine_kernel<D, G><<<U, kThreads, csmem, c.stream>>>(a, out, mass);
    return check_launch();
}

kvr_status tiered_attend_dispatch(const LaunchCtx &c, const kvr_tier_state &s, const void *q,
                                  const void *K, const void *V, const int32_t *seq_len,
                                  float scale, float *out, float *mass, uint8_t *ws, int32_t *err,
                                  uint64_t wait_ns, bool withhold_last)
{
    const kvr_shape &sh = c.shape;
    const int64_t U = (int64_t)sh.B * sh.Hkv;
    const int G = sh.Hq / sh.Hkv;
    TieredArgs a;
    a.Hkv = sh.Hkv;
    a.G = G;
    a.cap = sh.cap;
    a.n_win = s.n_win;
    a.S = tiered_splits(U, s.n_win);
    a.tier = s.tier;
    a.ledger = s.ledger;
    a.q = static_cast<const __nv_bfloat16 *>(q);
    a.K = static_cast<const __nv_bfloat16 *>(K);
    a.V = static_cast<const __nv_bfloat16 *>(V);
    a.seq_len = seq_len;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.part = reinterpret_cast<float *>(ws);
    a.lse = reinterpret_cast<float *>(ws + align_up((size_t)U * a.S * (2 * G + G * sh.d) * 4, 256));
    a.err = err;
    a.wait_ns = wait_ns;
    a.withhold_last = withhold_last ? 1 : 0;
    if (sh.d == 128) {
        switch (G) {
        case 1: return tiered_launch<128, 1>(c, a, out, mass);
        case 2: return tiered_launch<128, 2>(c, a, out, mass);
        case 4: return tiered_launch<128, 4>(c, a, out, mass);
        case 8: return tiered_launch<128, 8>(c, a, out, mass);
        }
    } else {
        switch (G) {
        case 1: return tiered_launch<64, 1>(c, a, out, mass);
        case 2: return tiered_launch<64, 2>(c, a, out, mass);
        case 4: return tiered_launch<64, 4>(c, a, out, mass);
        case 8: return tiered_launch<64, 8>(c, a, out, mass);
        }
    }
    return KVR_ERR_UNSUPPORTED;
}

kvr_status tier_update_dispatch(const LaunchCtx &c, const kvr_tier_state &s, const float *mass,
                                const int32_t *seq_len, void *K, void *V, int32_t *stats,
                                uint8_t *ws, int32_t *err)
{
    const int U = c.shape.B * c.shape.Hkv;
    RankArgs r;
    r.t = tier_args(c, s);
    r.mass = mass;
    r.seq_len = seq_len;
    r.stats = stats;
    r.moves = reinterpret_cast<int32_t *>(ws);
    r.n_moves = reinterpret_cast<int32_t *>(ws + align_up((size_t)U * s.n_win * 4, 256));
    r.err = err;
    int P = 2;
    while (P < s.n_win) P <<= 1;
    r.P = P;
    const int smem = P * 12;
    kvr_status st = raise_smem_limit(reinterpret_cast<const void *>(&tier_rank_kernel), smem);
    if (st != KVR_OK) return st;
    tier_rank_kernel<<<U, kRankThreads, smem, c.stream>>>(r);
    // the move kernel reads the lists the ranking writes: never launch it
    // after a ranking that did not launch
    if (check_launch() != KVR_OK) return KVR_ERR_CUDA;
    const dim3 grid(kMoveX, (unsigned)U);
    auto *Kb = static_cast<__nv_bfloat16 *>(K);
    auto *Vb = static_cast<__nv_bfloat16 *>(V);
    if (c.shape.d == 128)
        tier_move_kernel<128><<<grid, kThreads, 0, c.stream>>>(r.t, r.moves, r.n_moves, Kb, Vb, err);
    else
        tier_move_kernel<64><<<grid, kThreads, 0, c.stream>>>(r.t, r.moves, r.n_moves, Kb, Vb, err);
    return check_launch();
}

bool tier_shape_ok(const kvr_shape &s, int64_t n_win)
{
    const int G = s.Hq / s.Hkv;
    // tensor-map row coordinates are int32
    return s.dtype == KVR_BF16 && G <= 8 && n_win <= kMaxWin && n_win * kWin >= s.cap &&
           (int64_t)s.B * s.Hkv * s.cap < ((int64_t)1 << 31);
}

}  // namespace kvr
