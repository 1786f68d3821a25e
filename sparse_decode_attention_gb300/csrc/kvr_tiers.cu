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
constexpr int kSms = 152;       // GB300 streaming multiprocessors (grid sizing)

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
};

template <int D, int G> struct TieredCfg {
    static constexpr int RB = 2 * D;                   // bf16 row bytes
    static constexpr int RS = RB + 16;                 // padded row stride in shared memory
    static constexpr int NG = D / kQG;                 // INT2 groups per row
    static constexpr int LB = ledger_bytes_of(D);
    static constexpr int CB = kWin * NG * 8, PB = kWin * NG * 4;
    static constexpr int BUF = (2 * kWin * RS > LB ? 2 * kWin * RS : LB);
    static constexpr int DG = D / 4;                   // 4-dim groups (PV)
    static constexpr int TS = kThreads / DG;           // token subsets (PV)
    static constexpr int TPT = kWin / TS;              // tokens per thread per window (PV)
    static constexpr int PART = D / 4;                 // dims per QK part (4 parts)
    static constexpr int GP = G < 4 ? 4 : G;           // padded head count of the P rows
    // shared memory: two staging buffers, then q, partial scores, P, softmax state
    static constexpr int oBuf = 0;
    static constexpr int oQ = 2 * BUF;                       // float [G][D]
    static constexpr int oSp = oQ + G * D * 4;               // float [4][G][kWin]
    static constexpr int oP = oSp + 4 * G * kWin * 4;        // float [kWin][GP]
    static constexpr int oSt = oP + kWin * GP * 4;           // float m[G], l[G], alpha[G]
    static constexpr int oWin = oSt + 3 * 16 * 4;            // int32 [2] window of each buffer
    static constexpr int bytes = oWin + 64;
    static_assert(TS * DG == kThreads && kWin % TS == 0, "PV thread layout");
    static_assert(TS * D * G * 4 <= 2 * BUF, "the final reduction reuses the staging buffers");
};

template <int D, int G>
__global__ void __launch_bounds__(kThreads, 2) tiered_attend_kernel(TieredArgs a)
{
    using C = TieredCfg<D, G>;
    extern __shared__ __align__(16) uint8_t smem[];
    float *q_s = reinterpret_cast<float *>(smem + C::oQ);
    float *sp = reinterpret_cast<float *>(smem + C::oSp);
    float *P = reinterpret_cast<float *>(smem + C::oP);
    float *st_m = reinterpret_cast<float *>(smem + C::oSt);
    float *st_l = st_m + 16, *st_a = st_m + 32;
    int *buf_win = reinterpret_cast<int *>(smem + C::oWin);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
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

    // q of the group, scaled into the log2 domain
    for (int i = tid; i < G * D; i += kThreads)
        q_s[i] = __bfloat162float(a.q[((size_t)b * a.Hkv * G + (size_t)h * G) * D + i]) *
                 a.scale_log2;
    if (tid < G) {
        st_m[tid] = -CUDART_INF_F;
        st_l[tid] = 0.0f;
    }
    // lse of evicted windows in the range: -inf (no mass)
    for (int64_t w = w_begin + tid; w < w_end; w += kThreads) {
        const int8_t t = w < closed ? tier[w] : KVR_TIER_BF16;
        if (w < closed && checked_tier(t, a.err) == KVR_TIER_EVICTED) {
#pragma unroll
            for (int g = 0; g < G; g++) a.lse[(uw + w) * G + g] = -CUDART_INF_F;
        }
    }

    const uint8_t *Ku = reinterpret_cast<const uint8_t *>(a.K + (size_t)u * a.cap * D);
    const uint8_t *Vu = reinterpret_cast<const uint8_t *>(a.V + (size_t)u * a.cap * D);
    const uint8_t *Lu = a.ledger + uw * (size_t)C::LB;

    // next live window at or after w (w_end if none)
    auto next_live = [&](int64_t w) {
        while (w < w_end && w < closed) {
            const int8_t t = tier[w];
            if (t == KVR_TIER_BF16 || t == KVR_TIER_INT2) break;
            w++;
        }
        return w;
    };
    // stage window w into buffer `bi`
    auto issue = [&](int64_t w, int bi) {
        uint8_t *buf = smem + C::oBuf + bi * C::BUF;
        const bool int2 = w < closed && tier[w] == KVR_TIER_INT2;
        if (int2) {
            const uint8_t *src = Lu + (size_t)w * C::LB;
            for (int i = tid; i < C::LB / 16; i += kThreads) cp_async16(buf + i * 16, src + i * 16);
        } else {
            const int64_t t0 = w * kWin;
            const int n = (int)(N - t0 < kWin ? N - t0 : kWin);
            constexpr int PPR = C::RB / 16;  // 16-byte pieces per row
#pragma unroll
            for (int kv = 0; kv < 2; kv++) {
                const uint8_t *base = (kv ? Vu : Ku) + (size_t)t0 * C::RB;
                uint8_t *dst = buf + kv * kWin * C::RS;
                for (int i = tid; i < kWin * PPR; i += kThreads) {
                    const int r = i / PPR, pc = i % PPR;
                    const bool in = r < n;
                    cp_async16(dst + r * C::RS + pc * 16, base + (in ? (size_t)r * C::RB : 0) + pc * 16,
                               in ? 16 : 0);
                }
            }
        }
        if (tid == 0) buf_win[bi] = (int)(int2 ? -(w + 1) : (w + 1));
    };

    // PV accumulators: 4 dims x G heads over the token subset ts
    const int dg = tid % C::DG, ts = tid / C::DG;
    float acc[G][4];
#pragma unroll
    for (int g = 0; g < G; g++)
#pragma unroll
        for (int j = 0; j < 4; j++) acc[g][j] = 0.0f;

    int64_t cur = next_live(w_begin);
    if (cur < w_end) issue(cur, 0);
    cp_async_commit();
    int bi = 0;
    while (cur < w_end) {
        const int64_t nxt = next_live(cur + 1);
        if (nxt < w_end) issue(nxt, bi ^ 1);
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();

        const uint8_t *buf = smem + C::oBuf + bi * C::BUF;
        const bool int2 = buf_win[bi] < 0;
        const int n = (int)(N - cur * kWin < kWin ? N - cur * kWin : kWin);

        // ---- scores: token t = tid % 64, part p = tid / 64 (D/4 dims)
        {
            const int t = tid % kWin, p = tid / kWin;
            float s[G];
#pragma unroll
            for (int g = 0; g < G; g++) s[g] = 0.0f;
            if (!int2) {
                const uint8_t *row = buf + t * C::RS + p * C::PART * 2;
#pragma unroll
                for (int c = 0; c < C::PART; c += 8) {
                    const uint4 kv4 = *reinterpret_cast<const uint4 *>(row + c * 2);
                    const uint32_t w4[4] = {kv4.x, kv4.y, kv4.z, kv4.w};
                    float k8[8];
#pragma unroll
                    for (int i = 0; i < 4; i++) {
                        k8[2 * i] = bf16_lo(w4[i]);
                        k8[2 * i + 1] = bf16_hi(w4[i]);
                    }
#pragma unroll
                    for (int g = 0; g < G; g++) {
                        const float4 qa = *reinterpret_cast<const float4 *>(q_s + g * D + p * C::PART + c);
                        const float4 qb = *reinterpret_cast<const float4 *>(q_s + g * D + p * C::PART + c + 4);
                        s[g] = fmaf(qa.x, k8[0], s[g]);
                        s[g] = fmaf(qa.y, k8[1], s[g]);
                        s[g] = fmaf(qa.z, k8[2], s[g]);
                        s[g] = fmaf(qa.w, k8[3], s[g]);
                        s[g] = fmaf(qb.x, k8[4], s[g]);
                        s[g] = fmaf(qb.y, k8[5], s[g]);
                        s[g] = fmaf(qb.z, k8[6], s[g]);
                        s[g] = fmaf(qb.w, k8[7], s[g]);
                    }
                }
            } else {
                // dims [p*PART, (p+1)*PART) of group (p*PART)/32
                const int d0 = p * C::PART, grp = d0 / kQG, e0 = d0 % kQG;
                const uint8_t *cb = buf + (t * C::NG + grp) * 8;
                const uint32_t params = *reinterpret_cast<const uint32_t *>(buf + C::CB + (t * C::NG + grp) * 4);
                const float sc = __half2float(__ushort_as_half((unsigned short)(params & 0xffffu)));
                const float zz = __half2float(__ushort_as_half((unsigned short)(params >> 16)));
                const uint2 cw = *reinterpret_cast<const uint2 *>(cb);
#pragma unroll
                for (int c = 0; c < C::PART; c++) {
                    const int e = e0 + c;
                    const uint32_t wd = e < 16 ? cw.x : cw.y;
                    const float kx = fmaf((float)((wd >> (2 * (e & 15))) & 3u), sc, zz);
#pragma unroll
                    for (int g = 0; g < G; g++) s[g] = fmaf(q_s[g * D + d0 + c], kx, s[g]);
                }
            }
#pragma unroll
            for (int g = 0; g < G; g++) sp[(p * G + g) * kWin + t] = s[g];
        }
        __syncthreads();

        // ---- softmax state: warp g < G handles head g (two tokens per lane)
        if (warp < G) {
            const int g = warp;
            float s0 = -CUDART_INF_F, s1 = -CUDART_INF_F;
            if (lane < n)
                s0 = ((sp[(0 * G + g) * kWin + lane] + sp[(1 * G + g) * kWin + lane]) +
                      sp[(2 * G + g) * kWin + lane]) + sp[(3 * G + g) * kWin + lane];
            if (lane + 32 < n)
                s1 = ((sp[(0 * G + g) * kWin + lane + 32] + sp[(1 * G + g) * kWin + lane + 32]) +
                      sp[(2 * G + g) * kWin + lane + 32]) + sp[(3 * G + g) * kWin + lane + 32];
            float wm = fmaxf(s0, s1);
#pragma unroll
            for (int o = 16; o; o >>= 1) wm = fmaxf(wm, __shfl_xor_sync(kFull, wm, o));
            const float m_old = st_m[g];
            const float m_new = fmaxf(m_old, wm);
            const float p0 = exp2f(s0 - m_new), p1 = exp2f(s1 - m_new);
            float ls = p0 + p1;
#pragma unroll
            for (int o = 16; o; o >>= 1) ls += __shfl_xor_sync(kFull, ls, o);
            P[lane * C::GP + g] = p0;
            P[(lane + 32) * C::GP + g] = p1;
            if (lane == 0) {
                const float al = exp2f(m_old - m_new);
                st_a[g] = al;
                st_l[g] = st_l[g] * al + ls;
                st_m[g] = m_new;
                a.lse[(uw + cur) * G + g] = m_new + log2f(ls);
            }
        }
        __syncthreads();

        // ---- PV: 4 dims (dg) x G heads over tokens ts, ts + TS, ...
        {
            float al[G];
#pragma unroll
            for (int g = 0; g < G; g++) al[g] = st_a[g];
#pragma unroll
            for (int g = 0; g < G; g++)
#pragma unroll
                for (int j = 0; j < 4; j++) acc[g][j] *= al[g];
            if (!int2) {
                const uint8_t *vbase = buf + kWin * C::RS + dg * 8;
#pragma unroll
                for (int i = 0; i < C::TPT; i++) {
                    const int t = ts + i * C::TS;
                    const uint2 vv = *reinterpret_cast<const uint2 *>(vbase + t * C::RS);
                    const float v4[4] = {bf16_lo(vv.x), bf16_hi(vv.x), bf16_lo(vv.y), bf16_hi(vv.y)};
                    float pg[C::GP];
#pragma unroll
                    for (int g = 0; g < C::GP; g += 4) {
                        const float4 pp = *reinterpret_cast<const float4 *>(P + t * C::GP + g);
                        pg[g] = pp.x;
                        pg[g + 1] = pp.y;
                        pg[g + 2] = pp.z;
                        pg[g + 3] = pp.w;
                    }
#pragma unroll
                    for (int g = 0; g < G; g++)
#pragma unroll
                        for (int j = 0; j < 4; j++) acc[g][j] = fmaf(pg[g], v4[j], acc[g][j]);
                }
            } else {
                const uint8_t *vc = buf + C::CB + C::PB;  // V codes
                const uint8_t *vp = vc + C::CB;           // V params
                const int grp = (4 * dg) / kQG, e0 = (4 * dg) % kQG;
#pragma unroll
                for (int i = 0; i < C::TPT; i++) {
                    const int t = ts + i * C::TS;
                    const uint32_t byte = vc[(t * C::NG + grp) * 8 + e0 / 4];
                    const uint32_t params = *reinterpret_cast<const uint32_t *>(vp + (t * C::NG + grp) * 4);
                    const float sc = __half2float(__ushort_as_half((unsigned short)(params & 0xffffu)));
                    const float zz = __half2float(__ushort_as_half((unsigned short)(params >> 16)));
                    float v4[4];
#pragma unroll
                    for (int j = 0; j < 4; j++) v4[j] = fmaf((float)((byte >> (2 * j)) & 3u), sc, zz);
                    float pg[C::GP];
#pragma unroll
                    for (int g = 0; g < C::GP; g += 4) {
                        const float4 pp = *reinterpret_cast<const float4 *>(P + t * C::GP + g);
                        pg[g] = pp.x;
                        pg[g + 1] = pp.y;
                        pg[g + 2] = pp.z;
                        pg[g + 3] = pp.w;
                    }
#pragma unroll
                    for (int g = 0; g < G; g++)
#pragma unroll
                        for (int j = 0; j < 4; j++) acc[g][j] = fmaf(pg[g], v4[j], acc[g][j]);
                }
            }
        }
        __syncthreads();  // buffer bi and P are reused next
        cur = nxt;
        bi ^= 1;
    }
    cp_async_wait<0>();
    __syncthreads();

    // ---- reduce the token subsets: red[ts][g][D] in the staging buffers
    float *red = reinterpret_cast<float *>(smem + C::oBuf);
#pragma unroll
    for (int g = 0; g < G; g++)
        *reinterpret_cast<float4 *>(red + ((size_t)ts * G + g) * D + 4 * dg) =
            make_float4(acc[g][0], acc[g][1], acc[g][2], acc[g][3]);
    __syncthreads();
    float *part = a.part + ((size_t)u * a.S + x) * (2 * G + G * D);
    for (int i = tid; i < G * D; i += kThreads) {
        float o = 0.0f;
        for (int r = 0; r < C::TS; r++) o += red[(size_t)r * G * D + i];
        part[2 * G + i] = o;
    }
    if (tid < G) {
        part[tid] = st_m[tid];
        part[G + tid] = st_l[tid];
    }
}

template <int D, int G>
__global__ void __launch_bounds__(kThreads) tiered_combine_kernel(TieredArgs a, float *out,
                                                                  float *mass)
{
    __shared__ float sM[16], sL[16];
    const int u = blockIdx.x, b = u / a.Hkv, h = u % a.Hkv, tid = threadIdx.x;
    int64_t N = a.seq_len[b];
    if (N < 0 || N > a.cap) N = 0;
    const int64_t nw = (N + kWin - 1) / kWin;
    const float *part = a.part + (size_t)u * a.S * (2 * G + G * D);
    constexpr int PS = 2 * G + G * D;
    if (tid < G) {
        float M = -CUDART_INF_F;
        for (int x = 0; x < a.S; x++) M = fmaxf(M, part[x * PS + tid]);
        float L = 0.0f;
        if (M != -CUDART_INF_F)
            for (int x = 0; x < a.S; x++) {
                const float m = part[x * PS + tid];
                if (m != -CUDART_INF_F) L += part[x * PS + G + tid] * exp2f(m - M);
            }
        sM[tid] = M;
        sL[tid] = L;
    }
    __syncthreads();
    for (int i = tid; i < G * D; i += kThreads) {
        const int g = i / D;
        const float M = sM[g], L = sL[g];
        float o = 0.0f;
        if (L > 0.0f) {
            for (int x = 0; x < a.S; x++) {
                const float m = part[x * PS + g];
                if (m != -CUDART_INF_F) o += part[x * PS + 2 * G + i] * exp2f(m - M);
            }
            o /= L;
        }
        out[((size_t)b * a.Hkv * G + (size_t)h * G) * D + i] = o;
    }
    const size_t uw = (size_t)u * a.n_win;
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
    // 1. scores; 2. collect the live closed windows
    for (int64_t w = tid; w < nw; w += kRankThreads) {
        const int8_t t = checked_tier(a.tier[uw + w], r.err);
        if (t == KVR_TIER_EVICTED) continue;
        const int64_t sc = a.score[uw + w] + __float2ll_rn(r.mass[uw + w] * 4294967296.0f);
        a.score[uw + w] = sc;
        if (w < closed) {
            const int i = atomicAdd(&s_live, 1);
            key[i] = sc;
            win[i] = (int32_t)w;
        }
    }
    __syncthreads();
    const int live = s_live;
    for (int i = live + tid; i < r.P; i += kRankThreads) {
        key[i] = INT64_MIN;
        win[i] = INT32_MAX;
    }
    __syncthreads();
    // bitonic sort of [0, P) into rank order
    for (int k = 2; k <= r.P; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = tid; i < r.P; i += kRankThreads) {
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
            __syncthreads();
        }
    }
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
    const int n = n_moves[u];
    for (int i = blockIdx.x; i < n; i += gridDim.x) {
        const int32_t e = moves[uw + i];
        const int64_t w = e & ((1 << 30) - 1);
        const size_t row = (size_t)u * a.cap + (size_t)w * kWin;
        uint8_t *lg = a.ledger + (uw + w) * (size_t)ledger_bytes_of(D);
        if (e >> 30) dequantize_window<D>(lg, K + row * D, V + row * D);
        else quantize_window<D>(K + row * D, V + row * D, lg, err);
    }
}

int tiered_splits(int64_t U, int64_t n_win)
{
    const int64_t target = (4 * kSms + U - 1) / U;
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
    tier_count_kernel<<<U, kThreads, 0, c.stream>>>(a, seq_len);
    return check_launch();
}

template <int D, int G>
static kvr_status tiered_launch(const LaunchCtx &c, TieredArgs a, float *out, float *mass)
{
    using C = TieredCfg<D, G>;
    const void *k = reinterpret_cast<const void *>(&tiered_attend_kernel<D, G>);
    kvr_status st = raise_smem_limit(k, C::bytes);
    if (st != KVR_OK) return st;
    const int U = c.shape.B * c.shape.Hkv;
    tiered_attend_kernel<D, G><<<dim3(a.S, U), kThreads, C::bytes, c.stream>>>(a);
    tiered_combine_kernel<D, G><<<U, kThreads, 0, c.stream>>>(a, out, mass);
    return check_launch();
}

kvr_status tiered_attend_dispatch(const LaunchCtx &c, const kvr_tier_state &s, const void *q,
                                  const void *K, const void *V, const int32_t *seq_len,
                                  float scale, float *out, float *mass, uint8_t *ws, int32_t *err)
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
    return s.dtype == KVR_BF16 && G <= 8 && n_win <= kMaxWin && n_win * kWin >= s.cap;
}

}  // namespace kvr
