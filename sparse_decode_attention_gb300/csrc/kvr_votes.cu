// kvr_votes.cu -- per-query vote lists of the magnitude-aware coarse votes.
//
// Source: ParisKV, "Pipeline di Recupero Nativa su GPU in Due Stadi": per
// sub-space the query picks its top-rho most similar centroids and the keys
// in those buckets receive tiered votes. Here the centroids of a sub-block
// are ranked by their similarity to the rotated query sub-vector: with
// a_j = |zq_j| (zq = FWHT(D q_bar)), the centroid that differs from the query
// code in the flip set x has similarity (sum_j a_j - 2 f(x)) / sqrt(8),
// f(x) = sum over the set bits j of x, ascending, of a_j (fp32 from +0).
// Patterns are ordered by (f(x), x); the ranks fall into the Hamming ring
// sizes 1, 8, 28, 56, 70, 56, 28, 8, 1 as tiers, and a pattern's vote is
// lut[tier]. Per (unit, sub-block) the kernel lists the patterns with a
// non-zero vote as (x | vote << 8); the selection matches every key's flip
// pattern against that list.
#include <cuda_bf16.h>

#include "kvr_device.cuh"
#include "kvr_launch.h"

namespace kvr {

namespace {

__device__ __constant__ int kRingEnd[9] = {1, 9, 37, 93, 163, 219, 247, 255, 256};

template <int D, typename T>
__global__ void __launch_bounds__(256) vote_list_kernel(VoteArgs a)
{
    constexpr int E = D / 32;
    __shared__ float s_a[8];
    __shared__ uint64_t s_key[256];
    __shared__ int s_cnt;
    grid_dependency_wait();  // q may come from the previous grid
    grid_launch_dependents();
    const int sb = blockIdx.x, u = blockIdx.y;
    const int b = u / a.Hkv, h = u % a.Hkv;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) s_cnt = 0;
    if (warp == 0) {
        // q_bar and zq in the canonical orders of the codes and the selection
        const T *qg = static_cast<const T *>(a.q) + ((int64_t)b * a.Hq + (int64_t)h * a.G) * D + lane * E;
        float x[E];
#pragma unroll
        for (int r = 0; r < E; r++) {
            float acc = to_f32(qg[r]);
            for (int g = 1; g < a.G; g++) acc = acc + to_f32(qg[(int64_t)g * D + r]);
            x[r] = acc / (float)a.G;
            if (a.sgn[lane * E + r] < 0) x[r] = -x[r];
        }
        fwht_lanes<E, 32>(x, lane);
#pragma unroll
        for (int r = 0; r < E; r++) {
            const int i = lane * E + r;
            if (i >= sb * 8 && i < sb * 8 + 8) s_a[i - sb * 8] = fabsf(x[r]);
        }
    }
    __syncthreads();
    const unsigned xp = (unsigned)tid;  // this thread's flip pattern
    float f = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; j++)
        if ((xp >> j) & 1u) f = f + s_a[j];
    const uint64_t key = ((uint64_t)__float_as_uint(f) << 8) | xp;  // f >= +0: bit order = value order
    s_key[tid] = key;
    __syncthreads();
    int rank = 0;
#pragma unroll 8
    for (int y = 0; y < 256; y++) rank += s_key[y] < key;
    int tier = 0;
    while (rank >= kRingEnd[tier]) tier++;
    const int v = a.lut[tier];
    uint16_t *out = a.lists + ((size_t)u * a.nb + sb) * kVoteStride;
    if (v > 0) out[atomicAdd(&s_cnt, 1)] = (uint16_t)(xp | (unsigned)v << 8);
    __syncthreads();
    if (tid == 0) out[256] = (uint16_t)s_cnt;
}

}  // namespace

kvr_status vote_list_dispatch(const LaunchCtx &c, const void *q, const int8_t *sgn,
                              const int32_t *lut, uint16_t *lists)
{
    VoteArgs a;
    a.q = q;
    a.sgn = sgn;
    a.Hq = c.shape.Hq;
    a.Hkv = c.shape.Hkv;
    a.G = c.shape.Hq / c.shape.Hkv;
    a.nb = c.shape.d / 8;
    for (int i = 0; i < 9; i++) a.lut[i] = lut[i];
    a.lists = lists;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)a.nb, (unsigned)(c.shape.B * c.shape.Hkv), 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = c.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e;
    const bool bf = c.shape.dtype == KVR_BF16;
    if (c.shape.d == 128)
        e = bf ? cudaLaunchKernelEx(&cfg, vote_list_kernel<128, __nv_bfloat16>, a)
               : cudaLaunchKernelEx(&cfg, vote_list_kernel<128, float>, a);
    else
        e = bf ? cudaLaunchKernelEx(&cfg, vote_list_kernel<64, __nv_bfloat16>, a)
               : cudaLaunchKernelEx(&cfg, vote_list_kernel<64, float>, a);
    if (e != cudaSuccess) return KVR_ERR_CUDA;
    return check_launch();
}

}  // namespace kvr
