// kvr_rsq.cu -- per-key records of the calibrated inner-product reranker
// (RSQ-IP) and the tables of its 3-bit magnitude quantiser.
//
// Source: ParisKV, "Pipeline di Recupero Nativa su GPU in Due Stadi",
// candidate reranking: each sub-space direction of a rotated key coded with
// a sign bit and 3 magnitude bits from the Beta prior of the rotation, a
// calibration scale per key and sub-space, and the inner-product estimate
// ||q|| sum_b w_b <v_b, q~_b> that needs no full-precision key.
//
// The quantiser: for a uniformly random unit vector in R^8 a coordinate has
// u_j^2 ~ Beta(1/2, 7/2); |u_j| is cut into 8 bins of equal probability and
// each bin dequantises to its conditional mean. The tables are computed here
// once on the host: the bin edges by bisection on the regularised incomplete
// beta function (continued fraction), the levels from the closed form of the
// conditional mean, E[t; a < t < b] = ((1-a^2)^B - (1-b^2)^B) / (B Beta(1/2, B))
// with B = 7/2, both in double and rounded to fp32.
#include <cmath>
#include <mutex>

#include <cuda_bf16.h>

#include "kvr_device.cuh"
#include "kvr_launch.h"

namespace kvr {

namespace {

constexpr int kM = 8;        // coordinates per sub-block
constexpr int kLevels = 8;   // magnitude levels (3 bits)

// Regularised incomplete beta I_x(a, b), continued fraction (modified Lentz).
double beta_cf(double a, double b, double x)
{
    const double tiny = 1e-300;
    double c = 1.0, d = 1.0 - (a + b) * x / (a + 1.0);
    if (std::fabs(d) < tiny) d = tiny;
    d = 1.0 / d;
    double f = d;
    for (int m = 1; m < 400; m++) {
        const double m2 = 2.0 * m;
        double num = m * (b - m) * x / ((a + m2 - 1.0) * (a + m2));
        d = 1.0 + num * d;
        if (std::fabs(d) < tiny) d = tiny;
        c = 1.0 + num / c;
        if (std::fabs(c) < tiny) c = tiny;
        d = 1.0 / d;
        f *= d * c;
        num = -(a + m) * (a + b + m) * x / ((a + m2) * (a + m2 + 1.0));
        d = 1.0 + num * d;
        if (std::fabs(d) < tiny) d = tiny;
        c = 1.0 + num / c;
        if (std::fabs(c) < tiny) c = tiny;
        d = 1.0 / d;
        const double step = d * c;
        f *= step;
        if (std::fabs(step - 1.0) < 1e-16) break;
    }
    return f;
}

double inc_beta(double a, double b, double x)
{
    if (x <= 0.0) return 0.0;
    if (x >= 1.0) return 1.0;
    const double lbeta = std::lgamma(a) + std::lgamma(b) - std::lgamma(a + b);
    const double front = std::exp(a * std::log(x) + b * std::log1p(-x) - lbeta);
    if (x < (a + 1.0) / (a + b + 2.0)) return front * beta_cf(a, b, x) / a;
    return 1.0 - front * beta_cf(b, a, 1.0 - x) / b;
}

RsqTables make_tables()
{
    RsqTables t;
    const double a = 0.5, B = 0.5 * (kM - 1);
    const double lbeta = std::lgamma(a) + std::lgamma(B) - std::lgamma(a + B);
    double x[kLevels + 1];  // squared bin edges
    x[0] = 0.0;
    x[kLevels] = 1.0;
    for (int i = 1; i < kLevels; i++) {
        double lo = x[i - 1], hi = 1.0;
        const double target = (double)i / kLevels;
        for (int it = 0; it < 100; it++) {
            const double mid = 0.5 * (lo + hi);
            if (inc_beta(a, B, mid) < target) lo = mid;
            else hi = mid;
        }
        x[i] = 0.5 * (lo + hi);
    }
    for (int i = 0; i < kLevels; i++) {
        t.bsq[i] = (float)x[i];
        // E[t | x_i < t^2 < x_{i+1}] with probability 1/8 per bin
        const double mass = (std::pow(1.0 - x[i], B) - std::pow(1.0 - x[i + 1], B)) / B;
        t.lev[i] = (float)(kLevels * mass * std::exp(-lbeta));
    }
    return t;
}

// ---------------------------------------------------------------- records

// One warp per key: z = FWHT(D k) with the codes' canonical stage order
// (E coordinates per lane, coordinate i at lane i / E), then per sub-block of
// 8 coordinates (LPB = 8 / E lanes): s = fma chain of z_j^2 over j ascending
// from +0, mag_j = #{i : fl(z_j^2) >= fl(bsq_i s)}, c = fma chain of
// |z_j| lev[mag_j], w = bf16(s / c) (0 when c == 0). The chains run through
// the block's lanes in coordinate order. Word of the block: nibble j =
// mag_j | sign_j << 3.
template <int D, typename T>
__device__ __forceinline__ void rsq_encode_body(const T *__restrict__ K, int Hkv, int64_t cap,
                                                const int32_t *__restrict__ pos0, int n_new,
                                                int64_t units, const int8_t *__restrict__ sgn,
                                                const RsqTables &tab, uint8_t *__restrict__ rec,
                                                int32_t *err)
{
    constexpr int E = D / 32;       // coordinates per lane
    constexpr int LPB = kM / E;     // lanes per sub-block
    constexpr int NB = D / kM;      // sub-blocks
    constexpr int RB = 6 * NB;      // record bytes
    __shared__ float s_bsq[kLevels], s_lev[kLevels];
    if (threadIdx.x < kLevels) {
        s_bsq[threadIdx.x] = tab.bsq[threadIdx.x];
        s_lev[threadIdx.x] = tab.lev[threadIdx.x];
    }
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int64_t gw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t total = units * n_new;
    if (gw >= total) return;  // warp-uniform
    const int64_t u = gw / n_new;
    const int t = (int)(gw % n_new);
    const int b = (int)(u / Hkv);
    const int64_t row = (int64_t)pos0[b] + t;
    if (row < 0 || row >= cap) {
        if (lane == 0) set_err(err, KVR_DEVERR_POSITION);
        return;
    }
    const T *kr = K + ((size_t)u * cap + row) * D + lane * E;
    float z[E];
#pragma unroll
    for (int r = 0; r < E; r++) z[r] = to_f32(kr[r]) * (float)sgn[lane * E + r];
    fwht_lanes<E, 32>(z, lane);

    const int pos = lane % LPB;                 // position of this lane in its block
    const int first = lane - pos;               // first lane of the block
    float s = 0.0f;
#pragma unroll
    for (int k = 0; k < LPB; k++) {
        float sk = s;
        if (pos == k) {
#pragma unroll
            for (int r = 0; r < E; r++) sk = fmaf(z[r], z[r], sk);
        }
        __syncwarp();
        s = __shfl_sync(kFull, sk, first + k);
    }
    int mag[E];
    uint32_t word = 0;
#pragma unroll
    for (int r = 0; r < E; r++) {
        const float a2 = z[r] * z[r];
        int m = 0;
#pragma unroll
        for (int i = 1; i < kLevels; i++)
            if (a2 >= s_bsq[i] * s) m = i;
        mag[r] = m;
        const int j = pos * E + r;  // coordinate within the block
        word |= ((uint32_t)m | (uint32_t)(z[r] < 0.0f) << 3) << (4 * j);
    }
    float c = 0.0f;
#pragma unroll
    for (int k = 0; k < LPB; k++) {
        float ck = c;
        if (pos == k) {
#pragma unroll
            for (int r = 0; r < E; r++) ck = fmaf(fabsf(z[r]), s_lev[mag[r]], ck);
        }
        __syncwarp();
        c = __shfl_sync(kFull, ck, first + k);
    }
#pragma unroll
    for (int o = 1; o < LPB; o <<= 1) word |= __shfl_xor_sync(kFull, word, o);
    if (pos == 0) {
        const int blk = lane / LPB;
        uint8_t *out = rec + ((size_t)u * cap + row) * RB;
        *reinterpret_cast<uint32_t *>(out + 4 * blk) = word;
        const float w = (c > 0.0f) ? __fdiv_rn(s, c) : 0.0f;
        const __nv_bfloat16 wb = __float2bfloat16_rn(w);
        *reinterpret_cast<uint16_t *>(out + 4 * NB + 2 * blk) = *reinterpret_cast<const uint16_t *>(&wb);
    }
}

// LATE: the decode step's form, launched after the attention as its
// programmatic dependent; it waits for that grid before finishing, so what
// follows on the stream still follows the attention.
template <int D, typename T, bool LATE>
__global__ void __launch_bounds__(256)
rsq_encode_kernel(const T *__restrict__ K, int Hkv, int64_t cap, const int32_t *__restrict__ pos0,
                  int n_new, int64_t units, const int8_t *__restrict__ sgn, RsqTables tab,
                  uint8_t *__restrict__ rec, int32_t *err)
{
    rsq_encode_body<D, T>(K, Hkv, cap, pos0, n_new, units, sgn, tab, rec, err);
    if constexpr (LATE) grid_dependency_wait();
}

template <int D, typename T>
kvr_status launch_rsq_encode(const LaunchCtx &c, const void *K, const int32_t *pos0, int n_new,
                             int64_t units, int64_t blocks, const int8_t *sgn, uint8_t *rec,
                             int32_t *err, bool late)
{
    const kvr_shape &s = c.shape;
    const T *Kt = static_cast<const T *>(K);
    const RsqTables &tab = rsq_tables();
    if (!late) {
        rsq_encode_kernel<D, T, false><<<(unsigned)blocks, 256, 0, c.stream>>>(
            Kt, s.Hkv, s.cap, pos0, n_new, units, sgn, tab, rec, err);
        return check_launch();
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks, 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = c.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, rsq_encode_kernel<D, T, true>, Kt, s.Hkv, s.cap, pos0, n_new, units,
                           sgn, tab, rec, err) != cudaSuccess)
        return KVR_ERR_CUDA;
    return check_launch();
}

}  // namespace

const RsqTables &rsq_tables()
{
    static const RsqTables t = make_tables();
    return t;
}

kvr_status rsq_encode_dispatch(const LaunchCtx &c, const void *K, const int32_t *pos0, int n_new,
                               const int8_t *sgn, uint8_t *rec, int32_t *err, bool late)
{
    const kvr_shape &s = c.shape;
    const int64_t units = (int64_t)s.B * s.Hkv;
    const int64_t warps = units * n_new;
    const int64_t blocks = (warps * 32 + 255) / 256;
    if (blocks > 0x7fffffff) return KVR_ERR_UNSUPPORTED;
    if (s.dtype == KVR_BF16)
        return s.d == 128
                   ? launch_rsq_encode<128, __nv_bfloat16>(c, K, pos0, n_new, units, blocks, sgn, rec, err, late)
                   : launch_rsq_encode<64, __nv_bfloat16>(c, K, pos0, n_new, units, blocks, sgn, rec, err, late);
    return s.d == 128 ? launch_rsq_encode<128, float>(c, K, pos0, n_new, units, blocks, sgn, rec, err, late)
                      : launch_rsq_encode<64, float>(c, K, pos0, n_new, units, blocks, sgn, rec, err, late);
}

}  // namespace kvr
