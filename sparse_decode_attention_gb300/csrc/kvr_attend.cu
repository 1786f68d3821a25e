// kvr_attend.cu -- fused gather + online-softmax GQA attention over the
// selected tokens plus the local window (kvr_sparse_attend), one launch.
//
// ParisKV, "Problematica": decode attends only to a top-k subset of past
// tokens; "Meccanismo di Aggiornamento a Finestra Scorrevole": the most
// recent tokens stay in a local region that is always attended.
//
// One thread-block cluster per (batch, kv head) unit. The unit's token list
// (selected indices, then the Local window, then the Sink) is cut into equal
// slices, one per CTA; the slice's index reads go out with the length and
// count reads, on the assumption of k indices and a full window, and are
// redone when the token count says otherwise. A CTA copies the K and V rows
// of its slice, in batches of 48 KB (K and V), into double-buffered shared
// memory with 16-byte cp.async pieces. Each warp takes a strided share of a
// batch, its slots without branches (so their shuffle chains interleave): a
// token's K row is spread over the 32 lanes (d/32 dims each), the G per-head
// partial dots are reduced with a butterfly that hands head h to lanes
// [h*32/G, (h+1)*32/G), the softmax state is updated once per batch (log2
// domain), and p*v is accumulated in registers for all heads. Warps merge in
// shared memory, CTAs merge their (max, sum, output) partials through
// distributed shared memory, each CTA finishing an equal share of the output.
#include <cooperative_groups.h>

#include "kvr_device.cuh"
#include "kvr_launch.h"

namespace cg = cooperative_groups;

namespace kvr {

constexpr float kLog2e = 1.4426950408889634f;

struct AttArgs {
    int Hq, Hkv;
    int64_t cap;
    int W, kmax;
    int sink;                   // Sink tokens [0, sink), always attended
    const int32_t *region_end;  // Retrieval end per batch entry, or null: N - W
    float scale_log2;  // scale * log2(e)
    const void *q;
    const void *K;
    const void *V;
    const int32_t *idx;
    const int32_t *count;
    const int32_t *seq_len;
    float *out;
    int32_t *err;
};

template <int D, typename T, int G> struct AttCfg {
    // 8 warps: a CTA of this kernel and one of the selection that precedes it
    // fit on one SM together (registers and shared memory), so the attention
    // becomes resident while the selection drains (16 warps measured slower)
    static constexpr int kThreads = 256;
    static constexpr int kWarps = kThreads / 32;
    static constexpr int kRowBytes = D * (int)sizeof(T);
    static constexpr int kTok = 24576 / kRowBytes;  // tokens per batch (K + V = 48 KB)
    static constexpr int kBatchBytes = 2 * kTok * kRowBytes;
    static constexpr int kE = D / 32;  // dims per lane
    static constexpr int kWarpPart = kWarps * G * (D + 2) * 4;
    static constexpr int kBufBytes =
        (2 * kBatchBytes > kWarpPart) ? 2 * kBatchBytes : kWarpPart;
    static constexpr int kChunk = 8 * kTok;                // token ids loaded at once
    static constexpr int oTok = kBufBytes;                // [kChunk] int32
    static constexpr int oPm = oTok + kChunk * 4;         // [G]
    static constexpr int oPl = oPm + 16 * 4;              // [G]
    static constexpr int oPo = oPl + 16 * 4;              // [G][D]
    static constexpr int bytes = oPo + G * D * 4;
    static_assert(kTok % kWarps == 0, "batch split");
};

template <int D, typename T, int G>
__global__ void __launch_bounds__(AttCfg<D, T, G>::kThreads, (G >= 16) ? 1 : 2) attend_kernel(AttArgs a)
{
    using CF = AttCfg<D, T, G>;
    constexpr int kAttThreads = CF::kThreads;
    constexpr int kAttWarps = CF::kWarps;
    constexpr int E = CF::kE;
    constexpr int RB = CF::kRowBytes;
    constexpr int TOK = CF::kTok;
    constexpr int TPW = TOK / kAttWarps;  // tokens per warp per batch
    constexpr int LPH = 32 / G;           // lanes per head after the reduction

    extern __shared__ __align__(128) uint8_t smem[];
    int32_t *sTok = reinterpret_cast<int32_t *>(smem + CF::oTok);
    float *sPm = reinterpret_cast<float *>(smem + CF::oPm);
    float *sPl = reinterpret_cast<float *>(smem + CF::oPl);
    float *sPo = reinterpret_cast<float *>(smem + CF::oPo);

    cg::cluster_group cluster = cg::this_cluster();
    // programmatic dependent launch: this grid may start while the previous one
    // drains; nothing is read before the previous grid's writes are visible
    grid_dependency_wait();
    grid_launch_dependents();
    const int CS = (int)cluster.num_blocks();
    const int rank = (int)cluster.block_rank();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int u = blockIdx.y;
    const int b = u / a.Hkv, hk = u % a.Hkv;

    // The selection normally returns kmax indices and the window is full: the
    // slice's index reads are issued on that assumption together with the
    // length and count reads (one round trip instead of two), and used only
    // if the token count confirms it (Sink and region runs load after).
    const bool spec = !a.region_end && a.sink <= 0;
    const int64_t nT_s = (int64_t)a.kmax + a.W;
    const int64_t lo_s = (int64_t)rank * nT_s / CS, hi_s = (int64_t)(rank + 1) * nT_s / CS;
    constexpr int SPN = (CF::kChunk + kAttThreads - 1) / kAttThreads;
    int32_t sp[SPN];
#pragma unroll
    for (int i = 0; i < SPN; i++) {
        const int64_t p = lo_s + tid + (int64_t)i * kAttThreads;
        sp[i] = (spec && tid + i * kAttThreads < CF::kChunk && p < hi_s && p < a.kmax)
                    ? a.idx[(size_t)u * a.kmax + p]
                    : -1;
    }
    int64_t N = a.seq_len[b];
    if (N < 0 || N > a.cap) {
        if (rank == 0 && tid == 0 && hk == 0) set_err(a.err, KVR_DEVERR_SEQ_LEN);
        N = 0;
    }
    // T = selected tokens, then [w0, N) (Local and buffer), then the Sink [0, p0)
    const int64_t p0 = min((int64_t)max(a.sink, 0), N);
    int64_t w0 = a.region_end ? (int64_t)a.region_end[b] : N - a.W;
    w0 = w0 < p0 ? p0 : (w0 > N ? N : w0);
    const int cnt = max(0, min(a.count[u], a.kmax));
    const int64_t nT = cnt + (N - w0) + p0;
    const int64_t lo = (int64_t)rank * nT / CS, hi = (int64_t)(rank + 1) * nT / CS;
    const int n = (int)(hi - lo);
    const int nbatch = (n + TOK - 1) / TOK;

    const uint8_t *Ku = static_cast<const uint8_t *>(a.K) + (size_t)u * a.cap * RB;
    const uint8_t *Vu = static_cast<const uint8_t *>(a.V) + (size_t)u * a.cap * RB;
    constexpr int PPR = RB / 16;
    constexpr int CH = CF::kChunk;
    const bool spec_ok = spec && nT == nT_s;  // then lo, hi and cnt are as assumed
    // token ids of the slice positions [c0, c0 + CH), loaded at once (-1 = skip)
    auto load_ids = [&](int c0) {
        const int cn = min(CH, n - c0);
#pragma unroll
        for (int i = 0; i < SPN; i++) {
            const int j = tid + i * kAttThreads;
            if (j >= cn) break;
            const int64_t p = lo + c0 + j;
            int32_t t;
            if (p < cnt) {
                t = (spec_ok && c0 == 0) ? sp[i] : a.idx[(size_t)u * a.kmax + p];
                if (t < p0 || t >= w0) {
                    set_err(a.err, KVR_DEVERR_INDEX);
                    t = -1;
                }
            } else if (p < cnt + (N - w0)) {
                t = (int32_t)(w0 + (p - cnt));
            } else {
                t = (int32_t)(p - cnt - (N - w0));
            }
            sTok[j] = t;
        }
    };
    // 16-byte cp.async copies of the K and V rows of batch bi (one commit
    // group per batch; skipped slots are zero-filled)
    auto issue = [&](int bi, int c0) {
        uint8_t *buf = smem + (bi & 1) * CF::kBatchBytes;
        const int32_t *tok = sTok + (bi * TOK - c0);
        const int rows = min(TOK, n - bi * TOK);
        static_assert((PPR & (PPR - 1)) == 0, "pieces per row: a power of two");
#pragma unroll
        for (int kv = 0; kv < 2; kv++) {
            const uint8_t *base = kv ? Vu : Ku;
            uint8_t *dst = buf + kv * TOK * RB;
#pragma unroll 4
            for (int pc = tid; pc < rows * PPR; pc += kAttThreads) {
                const int j = pc / PPR, part = pc % PPR;  // shifts: PPR is a power of two
                const int32_t t = tok[j];
                cp_async16(dst + j * RB + part * 16, base + (t >= 0 ? (size_t)t * RB : 0) + part * 16,
                           t >= 0 ? 16 : 0);
            }
        }
        cp_async_commit();
    };

    // the group's query heads, pre-scaled into the log2 domain
    float qr[G][E];
    {
        const T *qg = static_cast<const T *>(a.q) + ((size_t)b * a.Hq + (size_t)hk * G) * D;
#pragma unroll
        for (int g = 0; g < G; g++)
#pragma unroll
            for (int e = 0; e < E; e++) qr[g][e] = to_f32(qg[g * D + lane * E + e]) * a.scale_log2;
    }
    float acc[G][E];
#pragma unroll
    for (int g = 0; g < G; g++)
#pragma unroll
        for (int e = 0; e < E; e++) acc[g][e] = 0.0f;
    float m = -INFINITY, l = 0.0f;  // softmax state of head lane / LPH

    for (int c0 = 0; c0 < n; c0 += CH) {
        load_ids(c0);
        __syncthreads();
        const int b0 = c0 / TOK, b1 = min(nbatch, (c0 + CH) / TOK);
        issue(b0, c0);
        if (b0 + 1 < b1) issue(b0 + 1, c0);
        for (int bi = b0; bi < b1; bi++) {
            if (bi + 1 < b1) cp_async_wait<1>();
            else cp_async_wait<0>();
            __syncthreads();
            const int32_t *tok = sTok + (bi * TOK - c0);
            const uint8_t *buf = smem + (bi & 1) * CF::kBatchBytes;
            const int rows = min(TOK, n - bi * TOK);
            // Branch-free over the warp's TPW slots (j < TOK: always inside the
            // buffer), so the slots' shuffle chains interleave; a slot past the
            // batch or of a skipped token scores -inf and adds nothing below.
            float s[TPW];
            bool live[TPW];
#pragma unroll
            for (int jj = 0; jj < TPW; jj++) {
                const int j = warp + jj * kAttWarps;
                live[jj] = j < rows && tok[j] >= 0;  // warp-uniform
                float kv[E];
                load_lane<E, T>(buf + j * RB, lane, kv);
                float part[G];
#pragma unroll
                for (int g = 0; g < G; g++) {
                    float d = 0.0f;
#pragma unroll
                    for (int e = 0; e < E; e++) d = fmaf(qr[g][e], kv[e], d);
                    part[g] = d;
                }
                const float sc = reduce_heads<G>(part, lane);
                s[jj] = live[jj] ? sc : -INFINITY;
            }
            float mb = -INFINITY;
#pragma unroll
            for (int jj = 0; jj < TPW; jj++) mb = fmaxf(mb, s[jj]);
            const float m_new = fmaxf(m, mb);
            const float alpha = (m == -INFINITY) ? 0.0f : exp2f(m - m_new);
            float p[TPW], ps = 0.0f;
#pragma unroll
            for (int jj = 0; jj < TPW; jj++) {
                p[jj] = (s[jj] == -INFINITY) ? 0.0f : exp2f(s[jj] - m_new);
                ps += p[jj];
            }
            l = l * alpha + ps;
            m = m_new;
#pragma unroll
            for (int g = 0; g < G; g++) {
                const float ag = __shfl_sync(kFull, alpha, g * LPH);
#pragma unroll
                for (int e = 0; e < E; e++) acc[g][e] *= ag;
            }
#pragma unroll
            for (int jj = 0; jj < TPW; jj++) {
                const int j = warp + jj * kAttWarps;
                float vv[E];
                load_lane<E, T>(buf + (TOK + j) * RB, lane, vv);
#pragma unroll
                for (int e = 0; e < E; e++) vv[e] = live[jj] ? vv[e] : 0.0f;  // stale rows may hold NaN
#pragma unroll
                for (int g = 0; g < G; g++) {
                    const float pg = __shfl_sync(kFull, p[jj], g * LPH);
#pragma unroll
                    for (int e = 0; e < E; e++) acc[g][e] = fmaf(pg, vv[e], acc[g][e]);
                }
            }
            __syncthreads();
            if (bi + 2 < b1) issue(bi + 2, c0);
        }
    }

    // merge the warps (their partials reuse the batch buffers)
    float *sWm = reinterpret_cast<float *>(smem);  // [warps][G]
    float *sWl = sWm + kAttWarps * G;              // [warps][G]
    float *sWo = sWl + kAttWarps * G;              // [warps][G][D]
    __syncthreads();
    if ((lane % LPH) == 0) {
        sWm[warp * G + lane / LPH] = m;
        sWl[warp * G + lane / LPH] = l;
    }
#pragma unroll
    for (int g = 0; g < G; g++)
#pragma unroll
        for (int e = 0; e < E; e++) sWo[(warp * G + g) * D + lane * E + e] = acc[g][e];
    __syncthreads();
    for (int t = tid; t < G * D; t += kAttThreads) {
        const int g = t / D, dim = t % D;
        float M = -INFINITY;
        for (int w = 0; w < kAttWarps; w++) M = fmaxf(M, sWm[w * G + g]);
        float L = 0.0f, O = 0.0f;
        if (M != -INFINITY) {
            for (int w = 0; w < kAttWarps; w++) {
                const float mw = sWm[w * G + g];
                if (mw == -INFINITY) continue;
                const float f = exp2f(mw - M);
                L = fmaf(sWl[w * G + g], f, L);
                O = fmaf(sWo[(w * G + g) * D + dim], f, O);
            }
        }
        sPo[t] = O;
        if (dim == 0) {
            sPm[g] = M;
            sPl[g] = L;
        }
    }
    __syncthreads();
    cluster.sync();  // CTA partials published

    // every CTA finishes an equal share of the unit's G*D outputs
    const int e0 = rank * (G * D) / CS, e1 = (rank + 1) * (G * D) / CS;
    for (int t = e0 + tid; t < e1; t += kAttThreads) {
        const int g = t / D, dim = t % D;
        // all remote loads first (independent), then the arithmetic
        float mr[16], lr[16], orr[16];
#pragma unroll
        for (int r = 0; r < 16; r++) {
            mr[r] = (r < CS) ? *cluster.map_shared_rank(&sPm[g], r) : -INFINITY;
            lr[r] = (r < CS) ? *cluster.map_shared_rank(&sPl[g], r) : 0.0f;
            orr[r] = (r < CS) ? *cluster.map_shared_rank(&sPo[t], r) : 0.0f;
        }
        float M = -INFINITY;
#pragma unroll
        for (int r = 0; r < 16; r++) M = fmaxf(M, mr[r]);
        float L = 0.0f, O = 0.0f;
        if (M != -INFINITY) {
#pragma unroll
            for (int r = 0; r < 16; r++) {
                if (mr[r] == -INFINITY) continue;
                const float f = exp2f(mr[r] - M);
                L = fmaf(lr[r], f, L);
                O = fmaf(orr[r], f, O);
            }
        }
        a.out[((size_t)b * a.Hq + (size_t)hk * G + g) * D + dim] = (L > 0.0f) ? O / L : 0.0f;
    }
    __syncthreads();
    cluster.sync();  // no CTA leaves while another may read its shared memory
}

int attend_cluster_size(int U, int64_t most_tokens)
{
    // On GB300 (152 SMs) 16-CTA clusters fit only 7 times at one CTA per SM
    // and 12-CTA ones 8 times (occupancy query): with 8 units, 16-CTA
    // clusters pack CTAs two to an SM and the packed ones set every cluster
    // barrier; 12-CTA clusters keep each CTA on its own SM (attention per
    // call 16.6 -> 14.4 us at 128K).
    int cs = (U == 8) ? 12 : 16;
    while (cs > 1 && (int64_t)U * cs > 2 * sm_count()) cs >>= 1;
    while (cs > 1 && most_tokens < (int64_t)cs * 32) cs >>= 1;  // >= 32 tokens per CTA
    return cs;
}

template <int D, typename T, int G>
static kvr_status launch_attend_g(const LaunchCtx &c, const AttArgs &a, int cs)
{
    auto kern = attend_kernel<D, T, G>;
    const int smem = AttCfg<D, T, G>::bytes;
    kvr_status st = prepare_cluster_kernel(reinterpret_cast<const void *>(kern), smem);
    if (st != KVR_OK) return st;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cs, c.shape.B * c.shape.Hkv, 1);
    cfg.blockDim = dim3(AttCfg<D, T, G>::kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = c.stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    if (cudaLaunchKernelEx(&cfg, kern, a) != cudaSuccess) return KVR_ERR_CUDA;
    return check_launch();
}

template <int D, typename T>
static kvr_status launch_attend(const LaunchCtx &c, const AttArgs &a, int cs, int G)
{
    switch (G) {
    case 1: return launch_attend_g<D, T, 1>(c, a, cs);
    case 2: return launch_attend_g<D, T, 2>(c, a, cs);
    case 4: return launch_attend_g<D, T, 4>(c, a, cs);
    case 8: return launch_attend_g<D, T, 8>(c, a, cs);
    case 16: return launch_attend_g<D, T, 16>(c, a, cs);
    }
    return KVR_ERR_UNSUPPORTED;
}

kvr_status attend_dispatch(const LaunchCtx &c, const AttendPlan &plan, const void *q,
                           const void *K, const void *V, const int32_t *idx, int kmax,
                           const int32_t *count, const int32_t *seq_len, int W, int sink,
                           const int32_t *region_end, float scale, float *out, uint8_t *ws,
                           int32_t *err)
{
    (void)plan;
    (void)ws;
    AttArgs a;
    a.Hq = c.shape.Hq;
    a.Hkv = c.shape.Hkv;
    a.cap = c.shape.cap;
    a.W = W;
    a.kmax = kmax;
    a.sink = sink;
    a.region_end = region_end;
    a.scale_log2 = scale * kLog2e;
    a.q = q;
    a.K = K;
    a.V = V;
    a.idx = idx;
    a.count = count;
    a.seq_len = seq_len;
    a.out = out;
    a.err = err;
    const int G = c.shape.Hq / c.shape.Hkv;
    // tokens per unit for the cluster size (load balance only): with regions
    // the Local + buffer length lives on the device, 256 stands in for it
    const int64_t most = (int64_t)kmax + (region_end ? (int64_t)sink + 256 : (int64_t)W);
    const int cs = attend_cluster_size(c.shape.B * c.shape.Hkv, most);
    const bool bf = c.shape.dtype == KVR_BF16;
    if (c.shape.d == 128)
        return bf ? launch_attend<128, __nv_bfloat16>(c, a, cs, G)
                  : launch_attend<128, float>(c, a, cs, G);
    return bf ? launch_attend<64, __nv_bfloat16>(c, a, cs, G)
              : launch_attend<64, float>(c, a, cs, G);
}

}  // namespace kvr
