// kvr_attend.cu -- fused gather + online-softmax GQA attention over the
// selected tokens plus the local window (kvr_sparse_attend).
//
// ParisKV, "Problematica": decode attends only to a top-k subset of past
// tokens; "Meccanismo di Aggiornamento a Finestra Scorrevole": the most
// recent tokens stay in a local region that is always attended.
//
// Split-K ("flash-decoding") layout: the token list of a unit (selected
// indices, then the window) is cut into segments of kTPC tokens; one CTA per
// (segment, unit) stages the K and V rows of its segment into shared memory
// with 16-byte cp.async copies (rows padded by 16 bytes so that 8 lanes
// reading 8 different rows hit 8 different bank groups), then walks the
// segment in tiles of 32 tokens: one warp computes the 32 logits of one
// query head, updates that head's running max / sum, and all threads
// accumulate p * v in registers (thread = one dim of a group of heads). The
// partial (m, l, o) of every CTA goes to the workspace and combine_kernel
// merges the partials of a unit.
#include "kvr_device.cuh"
#include "kvr_launch.h"

namespace kvr {

constexpr int kTPC = 128;   // tokens per CTA
constexpr int kTile = 32;   // tokens per softmax tile
constexpr int kAttThreads = 128;
constexpr float kLog2e = 1.4426950408889634f;

struct AttArgs {
    int Hq, Hkv, G;
    int64_t cap;
    int W, kmax, nsplit;
    float scale_log2;  // scale * log2(e): logits are kept in the log2 domain
    const void *q;
    const void *K;
    const void *V;
    const int32_t *idx;
    const int32_t *count;
    const int32_t *seq_len;
    float *out;
    float *part_m, *part_l, *part_o;  // [U][nsplit][G], [U][nsplit][G], [U][nsplit][G][D]
    int32_t *err;
};

__device__ __forceinline__ void cp_async16(void *dst, const void *src, int src_bytes)
{
    const uint32_t d = (uint32_t)__cvta_generic_to_shared(dst);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(d), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;\n" ::: "memory"); }

// Number of tokens a unit attends to and the start of its window.
__device__ __forceinline__ void unit_tokens(const AttArgs &a, int u, int64_t &w0, int &cnt,
                                            int64_t &nT, bool report)
{
    const int b = u / a.Hkv;
    int64_t N = a.seq_len[b];
    if (N < 0 || N > a.cap) {
        if (report) set_err(a.err, KVR_DEVERR_SEQ_LEN);
        N = 0;
    }
    w0 = N > a.W ? N - a.W : 0;
    cnt = max(0, min(a.count[u], a.kmax));
    nT = cnt + (N - w0);
}

template <int D, typename T> struct AttSmem {
    static constexpr int kRowBytes = D * (int)sizeof(T);
    static constexpr int kRowStride = kRowBytes + 16;
    static constexpr int kChunks = kRowBytes / 16;
    static constexpr size_t kKV = (size_t)kTPC * kRowStride;  // one of K, V
    static constexpr size_t bytes(int G)
    {
        return 2 * kKV + (size_t)G * D * 4 + 2 * (size_t)G * kTile * 4 + 3 * (size_t)G * 4 +
               kTPC * 4;
    }
};

template <int D, typename T>
__global__ void __launch_bounds__(kAttThreads) attend_partial_kernel(AttArgs a)
{
    using SM = AttSmem<D, T>;
    constexpr int E = Elem<T>::kVec;  // elements per 16-byte chunk
    constexpr int HG = kAttThreads / D;  // head groups in the V accumulation (1 or 2)
    constexpr int MAXH = 16 / HG;        // accumulators per thread (G <= 16)
    extern __shared__ __align__(16) uint8_t smem[];
    uint8_t *sK = smem;
    uint8_t *sV = smem + SM::kKV;
    float *sQ = reinterpret_cast<float *>(smem + 2 * SM::kKV);  // [G][D], pre-scaled
    float *sLogit = sQ + a.G * D;                                  // [G][kTile]
    float *sP = sLogit + a.G * kTile;                              // [G][kTile]
    float *sM = sP + a.G * kTile;                                  // [G]
    float *sL = sM + a.G;                                          // [G]
    float *sAlpha = sL + a.G;                                      // [G]
    int32_t *sTok = reinterpret_cast<int32_t *>(sAlpha + a.G);     // [kTPC]

    const int u = blockIdx.y, s = blockIdx.x, tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int b = u / a.Hkv, h = u % a.Hkv;
    const int G = a.G;
    int64_t w0, nT;
    int cnt;
    unit_tokens(a, u, w0, cnt, nT, s == 0 && tid == 0 && h == 0);
    const int64_t seg0 = (int64_t)s * kTPC;
    const int ntok = (int)max((int64_t)0, min(nT - seg0, (int64_t)kTPC));
    const size_t pbase = ((size_t)u * a.nsplit + s) * G;
    if (ntok == 0) {
        for (int i = tid; i < G; i += blockDim.x) {
            a.part_m[pbase + i] = -INFINITY;
            a.part_l[pbase + i] = 0.0f;
        }
        for (int i = tid; i < G * D; i += blockDim.x) a.part_o[pbase * D + i] = 0.0f;
        return;
    }

    // token ids of the segment (-1 = skipped)
    for (int j = tid; j < kTPC; j += blockDim.x) {
        int32_t t = -1;
        if (j < ntok) {
            const int64_t p = seg0 + j;
            if (p < cnt) {
                t = a.idx[(int64_t)u * a.kmax + p];
                if (t < 0 || t >= w0) {
                    set_err(a.err, KVR_DEVERR_INDEX);
                    t = -1;
                }
            } else {
                t = (int32_t)(w0 + (p - cnt));
            }
        }
        sTok[j] = t;
    }
    __syncthreads();

    // stage K and V rows (zero-filled for skipped slots)
    const uint8_t *Kb = static_cast<const uint8_t *>(a.K) + (size_t)u * a.cap * SM::kRowBytes;
    const uint8_t *Vb = static_cast<const uint8_t *>(a.V) + (size_t)u * a.cap * SM::kRowBytes;
    const int nrows = (ntok + kTile - 1) / kTile * kTile;
    for (int e = tid; e < nrows * SM::kChunks; e += blockDim.x) {
        const int j = e / SM::kChunks, ch = e % SM::kChunks;
        const int32_t t = sTok[j];
        const size_t go = (t >= 0 ? (size_t)t * SM::kRowBytes : 0) + (size_t)ch * 16;
        const int nb = t >= 0 ? 16 : 0;
        cp_async16(sK + (size_t)j * SM::kRowStride + ch * 16, Kb + go, nb);
        cp_async16(sV + (size_t)j * SM::kRowStride + ch * 16, Vb + go, nb);
    }
    cp_async_commit();

    // query heads of the group, pre-multiplied by scale * log2(e)
    const T *qg = static_cast<const T *>(a.q) + ((int64_t)b * a.Hq + (int64_t)h * G) * D;
    for (int i = tid; i < G * D; i += blockDim.x) sQ[i] = to_f32(qg[i]) * a.scale_log2;
    for (int i = tid; i < G; i += blockDim.x) {
        sM[i] = -INFINITY;
        sL[i] = 0.0f;
    }
    cp_async_wait_all();
    __syncthreads();

    const int dim = tid % D, hg = tid / D;
    float acc[MAXH];
#pragma unroll
    for (int i = 0; i < MAXH; i++) acc[i] = 0.0f;

    for (int t0 = 0; t0 < ntok; t0 += kTile) {
        // logits: thread -> (head, token) pairs; a warp shares one head
        for (int jd = tid; jd < G * kTile; jd += blockDim.x) {
            const int hh = jd / kTile, tt = jd % kTile;
            float lg = -INFINITY;
            if (t0 + tt < ntok && sTok[t0 + tt] >= 0) {
                const uint8_t *row = sK + (size_t)(t0 + tt) * SM::kRowStride;
                const float *qh = sQ + hh * D;
                float dot = 0.0f;
#pragma unroll
                for (int ch = 0; ch < SM::kChunks; ch++) {
                    float kv[E];
                    widen<E>(reinterpret_cast<const T *>(row + ch * 16), kv);
#pragma unroll
                    for (int e2 = 0; e2 < E; e2++) dot = fmaf(qh[ch * E + e2], kv[e2], dot);
                }
                lg = dot;
            }
            sLogit[jd] = lg;
        }
        __syncthreads();
        // online softmax update, one warp per head
        for (int hh = warp; hh < G; hh += blockDim.x / 32) {
            const float x = sLogit[hh * kTile + lane];
            float mt = x;
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, o));
            const float m_old = sM[hh];
            const float m_new = fmaxf(m_old, mt);
            const float p = (x == -INFINITY) ? 0.0f : exp2f(x - m_new);
            const float alpha = (m_old == -INFINITY) ? 0.0f : exp2f(m_old - m_new);
            float ps = p;
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) ps += __shfl_xor_sync(kFull, ps, o);
            sP[hh * kTile + lane] = p;
            __syncwarp();
            if (lane == 0) {
                sL[hh] = sL[hh] * alpha + ps;
                sM[hh] = m_new;
                sAlpha[hh] = alpha;
            }
        }
        __syncthreads();
        // o += p * v; this thread owns dim `dim` of heads hg, hg + HG, ...
        const int tmax = min(kTile, ntok - t0);
#pragma unroll
        for (int i = 0; i < MAXH; i++) {
            const int hh = hg + i * HG;
            if (hh < G) acc[i] *= sAlpha[hh];
        }
        for (int tt = 0; tt < tmax; tt++) {
            const T *vrow = reinterpret_cast<const T *>(sV + (size_t)(t0 + tt) * SM::kRowStride);
            const float v = to_f32(vrow[dim]);
#pragma unroll
            for (int i = 0; i < MAXH; i++) {
                const int hh = hg + i * HG;
                if (hh < G) acc[i] = fmaf(sP[hh * kTile + tt], v, acc[i]);
            }
        }
        __syncthreads();
    }
    for (int i = tid; i < G; i += blockDim.x) {
        a.part_m[pbase + i] = sM[i];
        a.part_l[pbase + i] = sL[i];
    }
#pragma unroll
    for (int i = 0; i < MAXH; i++) {
        const int hh = hg + i * HG;
        if (hh < G) a.part_o[(pbase + hh) * D + dim] = acc[i];
    }
}

// Merge the nsplit partials of each (unit, head): out = sum_s 2^(m_s - M) o_s /
// sum_s 2^(m_s - M) l_s, M = max_s m_s; an empty unit gives zeros.
template <int D>
__global__ void __launch_bounds__(D) combine_kernel(AttArgs a)
{
    const int u = blockIdx.y, hh = blockIdx.x, dim = threadIdx.x;
    const int G = a.G;
    const int b = u / a.Hkv, h = u % a.Hkv;
    float M = -INFINITY;
    for (int s = 0; s < a.nsplit; s++)
        M = fmaxf(M, a.part_m[((size_t)u * a.nsplit + s) * G + hh]);
    float L = 0.0f, o = 0.0f;
    if (M != -INFINITY) {
        for (int s = 0; s < a.nsplit; s++) {
            const size_t pi = ((size_t)u * a.nsplit + s) * G + hh;
            const float m = a.part_m[pi];
            if (m == -INFINITY) continue;
            const float f = exp2f(m - M);
            L = fmaf(a.part_l[pi], f, L);
            o = fmaf(a.part_o[pi * D + dim], f, o);
        }
    }
    a.out[((size_t)b * a.Hq + (size_t)h * G + hh) * D + dim] = (L > 0.0f) ? o / L : 0.0f;
}

template <int D, typename T>
static kvr_status launch_attend(const LaunchCtx &c, AttArgs &a)
{
    const int U = c.shape.B * c.shape.Hkv;
    const size_t smem = AttSmem<D, T>::bytes(a.G);
    if (smem > 48 * 1024) {
        kvr_status st = raise_smem_limit(reinterpret_cast<const void *>(attend_partial_kernel<D, T>),
                                         (int)AttSmem<D, T>::bytes(16));
        if (st != KVR_OK) return st;
    }
    attend_partial_kernel<D, T><<<dim3(a.nsplit, U), kAttThreads, smem, c.stream>>>(a);
    combine_kernel<D><<<dim3(a.G, U), D, 0, c.stream>>>(a);
    return check_launch();
}

kvr_status attend_dispatch(const LaunchCtx &c, const AttendPlan &plan, const void *q,
                           const void *K, const void *V, const int32_t *idx, int kmax,
                           const int32_t *count, const int32_t *seq_len, int W, float scale,
                           float *out, uint8_t *ws, int32_t *err)
{
    AttArgs a;
    a.Hq = c.shape.Hq;
    a.Hkv = c.shape.Hkv;
    a.G = c.shape.Hq / c.shape.Hkv;
    a.cap = c.shape.cap;
    a.W = W;
    a.kmax = kmax;
    a.nsplit = plan.nsplit;
    a.scale_log2 = scale * kLog2e;
    a.q = q;
    a.K = K;
    a.V = V;
    a.idx = idx;
    a.count = count;
    a.seq_len = seq_len;
    a.out = out;
    a.part_m = reinterpret_cast<float *>(ws + plan.off_m);
    a.part_l = reinterpret_cast<float *>(ws + plan.off_l);
    a.part_o = reinterpret_cast<float *>(ws + plan.off_o);
    a.err = err;
    const bool bf = c.shape.dtype == KVR_BF16;
    if (c.shape.d == 128)
        return bf ? launch_attend<128, __nv_bfloat16>(c, a) : launch_attend<128, float>(c, a);
    return bf ? launch_attend<64, __nv_bfloat16>(c, a) : launch_attend<64, float>(c, a);
}

}  // namespace kvr
