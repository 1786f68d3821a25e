// kvr_select.cu -- coarse collision scoring, candidate set, exact rescoring
// and final top-k for one decode step (kvr_select).
//
// ParisKV, "Pipeline di Recupero Nativa su GPU in Due Stadi": the query votes,
// per sub-block, for the centroids near its own with tiered weights; a key's
// coarse score is the sum of the votes of the buckets it sits in; the best
// few percent become candidates. The candidates are then rescored exactly
// with q.k and the top-k kept.
//
// Kernel chain per call (grid = chunks x units unless noted):
//   score_kernel     stream every pool code with 16-byte loads, XOR with the
//                    query code, per-byte popcount -> vote LUT -> integer
//                    score (uint8), per-chunk 256-bin histogram.
//   threshold_kernel (one CTA per unit) total histogram -> the score
//                    threshold T of the C'-th candidate, how many of the
//                    tied T-scores each chunk contributes (lowest indices
//                    first) and each chunk's output offset.
//   rescore_kernel   order-preserving compaction of the chunk's candidates
//                    (so the candidate list is ascending by index), then a
//                    gather of their K rows (16 lanes per row, 16-byte loads)
//                    and the canonical fp32 dot with q_bar.
//   topk_kernel      (one CTA per unit) 4-pass 8-bit radix select of the
//                    k'-th largest exact score in shared memory, then a
//                    stable compaction that emits the winners ascending.
#include "kvr_device.cuh"
#include "kvr_launch.h"

namespace kvr {

struct SelArgs {
    int Hq, Hkv, G;
    int64_t cap;
    int C, k, W;
    uint32_t lut_lo, lut_hi;  // vote weights for Hamming distance 0..3 and 4..7 (bytes)
    int lut8_minus_lut0;      // correction for distance 8 (selector index 8 reads lut[0])
    const void *q;
    const void *K;
    const uint32_t *codes;
    const int32_t *seq_len;
    const int8_t *sgn;
    int32_t *out_idx;
    int32_t *out_count;
    uint8_t *coarse;
    int32_t *cand_idx;
    float *cand_score;
    int32_t *cand_count;
    float *qbar;
    int32_t *chunk_hist;
    int32_t *chunk_off;
    int32_t *chunk_take;
    int32_t *unit_T;
    int64_t cap_pad;
    int chunk, nchunk;
    int32_t *err;
};

// Valid length of batch entry b, or 0 (with an error bit) when out of range.
__device__ __forceinline__ int64_t unit_len(const SelArgs &a, int b, bool report)
{
    const int64_t n = a.seq_len[b];
    if (n < 0 || n > a.cap) {
        if (report) set_err(a.err, KVR_DEVERR_SEQ_LEN);
        return 0;
    }
    return n;
}

// q_bar of unit u and its sign code, computed by one warp: lane l holds dims
// [l*E, l*E+E). q_bar_j = (q_0j + q_1j + ... + q_{G-1}j) / G, left to right.
template <int D, typename T>
__device__ __forceinline__ void query_code(const SelArgs &a, int u, uint32_t *s_qcode,
                                           float *g_qbar)
{
    constexpr int E = D / 32;
    const int lane = threadIdx.x & 31;
    const int b = u / a.Hkv, h = u % a.Hkv;
    const T *qg = static_cast<const T *>(a.q) + ((int64_t)b * a.Hq + (int64_t)h * a.G) * D;
    float x[E];
#pragma unroll
    for (int r = 0; r < E; r++) {
        const int j = lane * E + r;
        float acc = to_f32(qg[j]);
        for (int g = 1; g < a.G; g++) acc = acc + to_f32(qg[(int64_t)g * D + j]);
        x[r] = acc / (float)a.G;
        if (g_qbar) g_qbar[(int64_t)u * D + j] = x[r];
        if (a.sgn[j] < 0) x[r] = -x[r];
    }
    fwht_lanes<E, 32>(x, lane);
    const uint32_t w = sign_word<E>(x, lane);
    if ((lane % (32 / E)) == 0) s_qcode[(lane * E) / 32] = w;
}

// Votes of the 4 sub-blocks in one 32-bit code word XOR-ed with the query:
// per byte popcount (SWAR), then a 4-byte table lookup with prmt selecting
// lut[popcount & 7]; bytes at distance 8 are fixed up by the caller.
__device__ __forceinline__ uint32_t vote_bytes(uint32_t x, uint32_t lo, uint32_t hi,
                                               uint32_t &c8)
{
    x = x - ((x >> 1) & 0x55555555u);
    x = (x & 0x33333333u) + ((x >> 2) & 0x33333333u);
    x = (x + (x >> 4)) & 0x0f0f0f0fu;  // popcount per byte, 0..8
    c8 += (x >> 3) & 0x01010101u;      // bytes at distance 8
    const uint32_t y = x | (x >> 4);
    const uint32_t sel = (y & 0x77u) | ((y >> 8) & 0x7700u);
    return __byte_perm(lo, hi, sel);
}

template <int NW>
__device__ __forceinline__ int score_words(const uint32_t (&w)[NW], const uint32_t (&qw)[NW],
                                           const SelArgs &a)
{
    uint32_t acc = 0, c8 = 0;
#pragma unroll
    for (int i = 0; i < NW; i++) acc += vote_bytes(w[i] ^ qw[i], a.lut_lo, a.lut_hi, c8);
    int s = (int)((acc * 0x01010101u) >> 24);
    if (a.lut8_minus_lut0 != 0) s += a.lut8_minus_lut0 * (int)((c8 * 0x01010101u) >> 24);
    return s;
}

template <int D, typename T>
__global__ void __launch_bounds__(256) score_kernel(SelArgs a)
{
    constexpr int NW = D / 32;  // 32-bit code words per key
    constexpr int UNR = 4;
    __shared__ uint32_t s_qcode[NW];
    __shared__ int s_hist[256];
    const int u = blockIdx.y, c = blockIdx.x;
    const int b = u / a.Hkv;
    const int64_t N = unit_len(a, b, c == 0 && threadIdx.x == 0 && (u % a.Hkv) == 0);
    const int64_t pool = N > a.W ? N - a.W : 0;
    for (int i = threadIdx.x; i < 256; i += blockDim.x) s_hist[i] = 0;
    if (threadIdx.x < 32) query_code<D, T>(a, u, s_qcode, c == 0 ? a.qbar : nullptr);
    __syncthreads();
    uint32_t qw[NW];
#pragma unroll
    for (int i = 0; i < NW; i++) qw[i] = s_qcode[i];

    const int64_t start = (int64_t)c * a.chunk;
    const int64_t end = min(start + (int64_t)a.chunk, pool);
    const uint32_t *__restrict__ cw = a.codes + (int64_t)u * a.cap * NW;
    uint8_t *__restrict__ out = a.coarse + (int64_t)u * a.cap_pad;
    for (int64_t i0 = start + threadIdx.x; i0 < end; i0 += (int64_t)UNR * blockDim.x) {
        uint32_t w[UNR][NW];
#pragma unroll
        for (int r = 0; r < UNR; r++) {
            const int64_t i = i0 + (int64_t)r * blockDim.x;
            if (i < end) {
                if constexpr (NW == 4) {
                    const uint4 v = __ldg(reinterpret_cast<const uint4 *>(cw + i * 4));
                    w[r][0] = v.x; w[r][1] = v.y; w[r][2] = v.z; w[r][3] = v.w;
                } else {
                    const uint2 v = __ldg(reinterpret_cast<const uint2 *>(cw + i * 2));
                    w[r][0] = v.x; w[r][1] = v.y;
                }
            }
        }
#pragma unroll
        for (int r = 0; r < UNR; r++) {
            const int64_t i = i0 + (int64_t)r * blockDim.x;
            if (i < end) {
                const int s = score_words<NW>(w[r], qw, a);
                out[i] = (uint8_t)s;
                atomicAdd(&s_hist[s], 1);
            }
        }
    }
    __syncthreads();
    int32_t *gh = a.chunk_hist + ((int64_t)u * a.nchunk + c) * 256;
    for (int i = threadIdx.x; i < 256; i += blockDim.x) gh[i] = s_hist[i];
}

__global__ void __launch_bounds__(1024) threshold_kernel(SelArgs a)
{
    __shared__ int s_part[4][256];
    __shared__ int s_ge[257];
    __shared__ int s_scan[33];
    __shared__ int s_vmax;
    const int u = blockIdx.x, tid = threadIdx.x;
    const int b = u / a.Hkv;
    const int64_t N = unit_len(a, b, false);
    const int64_t pool = N > a.W ? N - a.W : 0;
    const int Cp = (int)min((int64_t)a.C, pool);

    const int bin = tid & 255, part = tid >> 8;
    int sum = 0;
    const int32_t *hist = a.chunk_hist + (int64_t)u * a.nchunk * 256;
    for (int c = part; c < a.nchunk; c += 4) sum += hist[(int64_t)c * 256 + bin];
    s_part[part][bin] = sum;
    if (tid == 0) s_vmax = -1;
    __syncthreads();
    // s_ge[t] = number of pool keys with score >= t (scan over bins 255 .. 0)
    const int tot = (tid < 256) ? s_part[0][255 - tid] + s_part[1][255 - tid] +
                                      s_part[2][255 - tid] + s_part[3][255 - tid]
                                : 0;
    if (tid < 256 && tot > 0) atomicMax(&s_vmax, 255 - tid);
    int total;
    const int ex = block_exclusive_scan(tot, s_scan, &total);
    if (tid < 256) s_ge[255 - tid] = ex + tot;
    if (tid == 0) s_ge[256] = 0;
    __syncthreads();
    // T = largest t with ge[t] >= Cp (ge is non-increasing in t)
    const int n_ok = __syncthreads_count(tid < 256 && s_ge[tid] >= Cp);
    const int T = (Cp == 0) ? 256 : n_ok - 1;
    const int n_gt = (T < 256) ? s_ge[T + 1] : 0;
    const int quota = Cp - n_gt;
    const int vmax = s_vmax;

    // per chunk: keys above T, ties at T, ties taken (lowest indices first), offset
    int gt = 0, eq = 0;
    const int c = tid;
    if (c < a.nchunk && T < 256) {
        const int32_t *hc = hist + (int64_t)c * 256;
        for (int v = T + 1; v <= vmax; v++) gt += hc[v];
        eq = hc[T];
    }
    int eq_tot;
    const int eq_before = block_exclusive_scan(eq, s_scan, &eq_tot);
    const int take = max(0, min(quota - eq_before, eq));
    int sel_tot;
    const int off = block_exclusive_scan(gt + take, s_scan, &sel_tot);
    if (c < a.nchunk) {
        a.chunk_off[(int64_t)u * a.nchunk + c] = off;
        a.chunk_take[(int64_t)u * a.nchunk + c] = take;
    }
    if (tid == 0) {
        a.unit_T[u] = T;
        a.cand_count[u] = Cp;
    }
}

// Keep the lowest n set bits of m.
__device__ __forceinline__ uint32_t lowest_bits(uint32_t m, int n)
{
    uint32_t r = 0;
    for (int i = 0; i < n && m; i++) {
        const uint32_t low = m & (0u - m);
        r |= low;
        m ^= low;
    }
    return r;
}

// Canonical exact score of the candidates in list[0..n): half-warp per row,
// lane gl holds dims [gl*D/16, (gl+1)*D/16), fma chain, butterfly 8,4,2,1.
template <int D, typename T>
__device__ __forceinline__ void rescore_list(const SelArgs &a, int u, const int32_t *list, int n,
                                             int64_t out_base, const float (&qv)[D / 16])
{
    constexpr int P = D / 16;
    constexpr int R = 4;  // rows in flight per half-warp
    const int hw = threadIdx.x >> 4, gl = threadIdx.x & 15;
    const int nhw = blockDim.x >> 4;
    const T *Ku = static_cast<const T *>(a.K) + (int64_t)u * a.cap * D;
    for (int base = 0; base < n; base += R * nhw) {
        float kv[R][P];
        int row[R];
#pragma unroll
        for (int r = 0; r < R; r++) {
            const int j = base + r * nhw + hw;
            row[r] = (j < n) ? list[j] : -1;
            if (row[r] >= 0) {
                widen<P>(Ku + (int64_t)row[r] * D + gl * P, kv[r]);
            } else {
#pragma unroll
                for (int e = 0; e < P; e++) kv[r][e] = 0.0f;
            }
        }
#pragma unroll
        for (int r = 0; r < R; r++) {
            float acc = 0.0f;
#pragma unroll
            for (int e = 0; e < P; e++) acc = __fmaf_rn(qv[e], kv[r][e], acc);
#pragma unroll
            for (int span = 8; span >= 1; span >>= 1) acc = acc + __shfl_xor_sync(kFull, acc, span);
            const int j = base + r * nhw + hw;
            if (gl == 0 && j < n) {
                if (acc != acc) set_err(a.err, KVR_DEVERR_NONFINITE);
                a.cand_score[(int64_t)u * a.C + out_base + j] = acc;
            }
        }
    }
}

template <int D, typename T>
__global__ void __launch_bounds__(256) rescore_kernel(SelArgs a)
{
    constexpr int ITEMS = 8;
    constexpr int TILE = 256 * ITEMS;
    __shared__ int s_scan[33];
    __shared__ int32_t s_list[TILE];
    __shared__ float s_qbar[D];
    const int u = blockIdx.y, c = blockIdx.x, tid = threadIdx.x;
    const int thr = a.unit_T[u];
    if (thr > 255) return;
    const int b = u / a.Hkv;
    const int64_t N = unit_len(a, b, false);
    const int64_t pool = N > a.W ? N - a.W : 0;
    const int64_t start = (int64_t)c * a.chunk;
    const int64_t end = min(start + (int64_t)a.chunk, pool);
    if (start >= end) return;
    const int take = a.chunk_take[(int64_t)u * a.nchunk + c];
    const int off = a.chunk_off[(int64_t)u * a.nchunk + c];
    for (int j = tid; j < D; j += blockDim.x) s_qbar[j] = a.qbar[(int64_t)u * D + j];
    __syncthreads();
    float qv[D / 16];
#pragma unroll
    for (int e = 0; e < D / 16; e++) qv[e] = s_qbar[(tid & 15) * (D / 16) + e];

    const uint8_t *sc = a.coarse + (int64_t)u * a.cap_pad;
    int32_t *cidx = a.cand_idx + (int64_t)u * a.C;
    int tie_carry = 0, sel_carry = 0;
    for (int64_t t0 = start; t0 < end; t0 += TILE) {
        const int64_t i0 = t0 + (int64_t)tid * ITEMS;
        uint32_t gtm = 0, eqm = 0;
        if (i0 + ITEMS <= end) {
            const uint2 v = *reinterpret_cast<const uint2 *>(sc + i0);
#pragma unroll
            for (int r = 0; r < ITEMS; r++) {
                const int s = (int)(((r < 4 ? v.x : v.y) >> (8 * (r & 3))) & 0xffu);
                gtm |= (s > thr ? 1u : 0u) << r;
                eqm |= (s == thr ? 1u : 0u) << r;
            }
        } else {
            for (int r = 0; r < ITEMS; r++) {
                if (i0 + r >= end) break;
                const int s = sc[i0 + r];
                gtm |= (s > thr ? 1u : 0u) << r;
                eqm |= (s == thr ? 1u : 0u) << r;
            }
        }
        int eq_tot;
        const int eq_before = block_exclusive_scan(__popc(eqm), s_scan, &eq_tot);
        const int allow = max(0, min(take - tie_carry - eq_before, __popc(eqm)));
        const uint32_t selm = gtm | lowest_bits(eqm, allow);
        int sel_tot;
        const int sel_before = block_exclusive_scan(__popc(selm), s_scan, &sel_tot);
        int r = 0;
        for (uint32_t m = selm; m; m &= m - 1, r++) {
            const int32_t idx = (int32_t)(i0 + __ffs(m) - 1);
            s_list[sel_before + r] = idx;
            cidx[off + sel_carry + sel_before + r] = idx;
        }
        __syncthreads();
        rescore_list<D, T>(a, u, s_list, sel_tot, off + sel_carry, qv);
        __syncthreads();
        tie_carry += eq_tot;
        sel_carry += sel_tot;
    }
}

__global__ void __launch_bounds__(1024) topk_kernel(SelArgs a)
{
    extern __shared__ uint32_t s_key[];
    __shared__ int s_hist[256];
    __shared__ int s_scan[33];
    __shared__ uint32_t s_prefix;
    __shared__ int s_remaining;
    const int u = blockIdx.x, tid = threadIdx.x;
    const int Cp = a.cand_count[u];
    const int kp = min(a.k, Cp);
    int32_t *orow = a.out_idx + (int64_t)u * a.k;
    for (int j = kp + tid; j < a.k; j += blockDim.x) orow[j] = -1;
    if (tid == 0) a.out_count[u] = kp;
    if (kp == 0) return;
    const float *S = a.cand_score + (int64_t)u * a.C;
    const int32_t *I = a.cand_idx + (int64_t)u * a.C;
    for (int j = tid; j < Cp; j += blockDim.x) s_key[j] = order_key(S[j]);

    // radix select of the kp-th largest key, 8 bits at a time from the top
    uint32_t prefix = 0, mask = 0;
    int remaining = kp;
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int i = tid; i < 256; i += blockDim.x) s_hist[i] = 0;
        __syncthreads();
        for (int j = tid; j < Cp; j += blockDim.x) {
            const uint32_t key = s_key[j];
            if ((key & mask) == prefix) atomicAdd(&s_hist[(key >> shift) & 255u], 1);
        }
        __syncthreads();
        if (tid < 32) {
            int cnt[8], sum = 0;
#pragma unroll
            for (int r = 0; r < 8; r++) {
                cnt[r] = s_hist[255 - (tid * 8 + r)];
                sum += cnt[r];
            }
            int incl = sum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(kFull, incl, o);
                if (tid >= o) incl += y;
            }
            int run = incl - sum;
            if (run < remaining && remaining <= incl) {
                for (int r = 0; r < 8; r++) {
                    if (run + cnt[r] >= remaining) {
                        s_prefix = prefix | ((uint32_t)(255 - (tid * 8 + r)) << shift);
                        s_remaining = remaining - run;
                        break;
                    }
                    run += cnt[r];
                }
            }
        }
        __syncthreads();
        prefix = s_prefix;
        remaining = s_remaining;
        mask |= 255u << shift;
    }
    const uint32_t keyT = prefix;  // the kp-th largest key
    const int quota = remaining;   // how many keys equal to keyT are taken

    // stable compaction in candidate order (= ascending token index)
    const int seg = (Cp + blockDim.x - 1) / blockDim.x;
    const int j0 = min(tid * seg, Cp), j1 = min(j0 + seg, Cp);
    int n_eq = 0;
    for (int j = j0; j < j1; j++) n_eq += (s_key[j] == keyT);
    int eq_tot;
    const int eq_before = block_exclusive_scan(n_eq, s_scan, &eq_tot);
    int n_sel = 0, seen = 0;
    for (int j = j0; j < j1; j++) {
        const uint32_t key = s_key[j];
        if (key > keyT) n_sel++;
        else if (key == keyT) n_sel += (eq_before + seen++ < quota);
    }
    int sel_tot;
    int pos = block_exclusive_scan(n_sel, s_scan, &sel_tot);
    seen = 0;
    for (int j = j0; j < j1; j++) {
        const uint32_t key = s_key[j];
        bool take = key > keyT;
        if (key == keyT) take = (eq_before + seen++ < quota);
        if (take) orow[pos++] = I[j];
    }
}

template <int D, typename T>
static kvr_status launch_select(const LaunchCtx &c, SelArgs &a)
{
    const int U = c.shape.B * c.shape.Hkv;
    const dim3 g(a.nchunk, U);
    score_kernel<D, T><<<g, 256, 0, c.stream>>>(a);
    threshold_kernel<<<U, 1024, 0, c.stream>>>(a);
    rescore_kernel<D, T><<<g, 256, 0, c.stream>>>(a);
    const size_t smem = (size_t)a.C * sizeof(uint32_t);
    if (smem > 48 * 1024) {
        kvr_status st = raise_smem_limit(reinterpret_cast<const void *>(topk_kernel),
                                         32768 * (int)sizeof(uint32_t));
        if (st != KVR_OK) return st;
    }
    topk_kernel<<<U, 1024, smem, c.stream>>>(a);
    return check_launch();
}

kvr_status select_dispatch(const LaunchCtx &c, const kvr_select_params &p, const SelectPlan &plan,
                           const void *q, const void *K, const uint8_t *codes,
                           const int32_t *seq_len, const int8_t *sgn, int32_t *out_idx,
                           int32_t *out_count, uint8_t *ws, int32_t *err)
{
    SelArgs a;
    a.Hq = c.shape.Hq;
    a.Hkv = c.shape.Hkv;
    a.G = c.shape.Hq / c.shape.Hkv;
    a.cap = c.shape.cap;
    a.C = p.C;
    a.k = p.k;
    a.W = p.W;
    a.lut_lo = (uint32_t)p.lut[0] | ((uint32_t)p.lut[1] << 8) | ((uint32_t)p.lut[2] << 16) |
               ((uint32_t)p.lut[3] << 24);
    a.lut_hi = (uint32_t)p.lut[4] | ((uint32_t)p.lut[5] << 8) | ((uint32_t)p.lut[6] << 16) |
               ((uint32_t)p.lut[7] << 24);
    a.lut8_minus_lut0 = p.lut[8] - p.lut[0];
    a.q = q;
    a.K = K;
    a.codes = reinterpret_cast<const uint32_t *>(codes);
    a.seq_len = seq_len;
    a.sgn = sgn;
    a.out_idx = out_idx;
    a.out_count = out_count;
    a.coarse = ws + plan.off_coarse;
    a.cand_idx = reinterpret_cast<int32_t *>(ws + plan.off_cand_idx);
    a.cand_score = reinterpret_cast<float *>(ws + plan.off_cand_score);
    a.cand_count = reinterpret_cast<int32_t *>(ws + plan.off_cand_count);
    a.qbar = reinterpret_cast<float *>(ws + plan.off_qbar);
    a.chunk_hist = reinterpret_cast<int32_t *>(ws + plan.off_chunk_hist);
    a.chunk_off = reinterpret_cast<int32_t *>(ws + plan.off_chunk_off);
    a.chunk_take = reinterpret_cast<int32_t *>(ws + plan.off_chunk_take);
    a.unit_T = reinterpret_cast<int32_t *>(ws + plan.off_unit_T);
    a.cap_pad = plan.cap_pad;
    a.chunk = plan.chunk;
    a.nchunk = plan.nchunk;
    a.err = err;
    const bool bf = c.shape.dtype == KVR_BF16;
    if (c.shape.d == 128)
        return bf ? launch_select<128, __nv_bfloat16>(c, a) : launch_select<128, float>(c, a);
    return bf ? launch_select<64, __nv_bfloat16>(c, a) : launch_select<64, float>(c, a);
}

}  // namespace kvr
