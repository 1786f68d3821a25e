// kvr_encode.cu -- append-time rotation and sign code of keys.
//
// ParisKV, "Centroidi Analitici Robusti al Drift": keys are rotated by a
// shared SRHT and assigned to the nearest fixed sign-pattern centroid; with
// the sub-block split of "Pipeline di Recupero Nativa su GPU in Due Stadi"
// the code of a key is the sign bits of its rotated vector.
//
// Codes are stored as bit-planes so that the scorer works on 32 keys per
// 32-bit word: 32 consecutive tokens form a block whose d code bits are d
// words (word p holds bit p of the 32 codes, bit i for token i); 32 blocks
// form a 1024-token tile stored as [chunk c = 4 planes][block j] 16-byte
// units, so that a warp reading one chunk of 32 blocks reads 512 contiguous
// bytes.
//
// One warp handles one 32-token block: it rotates the block's new rows
// (a row spread over d*sizeof(T)/16 lanes, one 16-byte load each, FWHT in
// registers with shuffles), then transposes the codes into planes with
// ballots and merges them into the block, keeping the bits of tokens outside
// the encoded range.
#include "kvr_device.cuh"
#include "kvr_launch.h"

namespace kvr {

template <int D, typename T>
__device__ __forceinline__ void encode_body(const T *__restrict__ K, int Hkv, int64_t cap,
                                            int64_t tiles, const int32_t *__restrict__ pos0,
                                            int n_new, int64_t units, int blocks_per_unit,
                                            const int8_t *__restrict__ sgn,
                                            uint8_t *__restrict__ codes, int32_t *err)
{
    constexpr int E = Elem<T>::kVec;  // elements per lane
    constexpr int L = D / E;          // lanes per row
    constexpr int KPW = 32 / L;       // rows per warp pass
    constexpr int NW = D / 32;        // code words per token
    constexpr int NCH = D / 4;        // 16-byte chunks per block
    static_assert(L >= 32 / E && L <= 32, "lane split");
    __shared__ uint32_t s_code[8][32][NW];

    const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
    const int gl = lane % L;
    const int64_t gw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t unit = gw / blocks_per_unit;
    if (unit >= units) return;  // whole warp
    const int kb = (int)(gw - unit * blocks_per_unit);
    const int b = (int)(unit / Hkv);
    const int64_t p0 = pos0[b];
    if ((p0 < 0 || p0 + n_new > cap) && kb == 0 && lane == 0) set_err(err, KVR_DEVERR_POSITION);
    const int64_t lo = p0 > 0 ? p0 : 0;
    const int64_t hi = (p0 + n_new < cap) ? p0 + n_new : cap;
    if (lo >= hi) return;
    const int64_t blk = lo / 32 + kb;
    if (blk * 32 >= hi) return;  // whole warp
    const int64_t t_lane = blk * 32 + lane;
    __syncwarp();
    const uint32_t inmask = __ballot_sync(kFull, t_lane >= lo && t_lane < hi);
    uint4 *dst = reinterpret_cast<uint4 *>(codes + ((size_t)unit * tiles + (size_t)(blk >> 5)) *
                                                       (D * 128)) +
                 ((size_t)lane * 32 + (size_t)(blk & 31));
    // a partly covered block keeps its other tokens' bits: fetch them early
    uint4 old = make_uint4(0u, 0u, 0u, 0u);
    if (inmask != 0xffffffffu && lane < NCH) old = *dst;

    const T *Ku = K + (size_t)unit * cap * D;
    for (int s0 = 0; s0 < 32; s0 += KPW) {
        if (((inmask >> s0) & ((1u << KPW) - 1u)) == 0u && KPW < 32) continue;  // warp-uniform
        const int slot = s0 + lane / L;
        const bool v = (inmask >> slot) & 1u;
        float x[E];
        if (v) {
            widen<E>(Ku + (size_t)(blk * 32 + slot) * D + gl * E, x);
        } else {
#pragma unroll
            for (int r = 0; r < E; r++) x[r] = 0.0f;
        }
        // D x: exact sign flips, no multiply (nothing for the compiler to contract)
#pragma unroll
        for (int r = 0; r < E; r++)
            if (sgn[gl * E + r] < 0) x[r] = -x[r];
        fwht_lanes<E, L>(x, gl);
        const uint32_t w = sign_word<E>(x, gl);
        if (v && (gl % (32 / E)) == 0) s_code[wib][slot][(gl * E) / 32] = w;
    }
    __syncwarp();

    // transpose into planes; lane c builds chunk c (planes 4c..4c+3)
    uint32_t mine[4] = {0u, 0u, 0u, 0u};
    if (__popc(inmask) <= 4) {
        // few tokens (the decode-time append): insert their bits directly
        if (lane < NCH)
            for (uint32_t m = inmask; m; m &= m - 1) {
                const int i = __ffs(m) - 1;
#pragma unroll
                for (int w4 = 0; w4 < 4; w4++) {
                    const int p = 4 * lane + w4;
                    mine[w4] |= ((s_code[wib][i][p >> 5] >> (p & 31)) & 1u) << i;
                }
            }
    } else {
        // plane p = ballot over the tokens of code bit p
        const bool have = (inmask >> lane) & 1u;
        for (int c = 0; c < NCH; c++) {
#pragma unroll
            for (int w4 = 0; w4 < 4; w4++) {
                const int p = 4 * c + w4;
                const uint32_t bit = have ? (s_code[wib][lane][p >> 5] >> (p & 31)) & 1u : 0u;
                const uint32_t word = __ballot_sync(kFull, bit);
                if (lane == c) mine[w4] = word;
            }
        }
    }
    if (lane < NCH) {
        const uint32_t keep = ~inmask;
        *dst = make_uint4((old.x & keep) | (mine[0] & inmask), (old.y & keep) | (mine[1] & inmask),
                          (old.z & keep) | (mine[2] & inmask), (old.w & keep) | (mine[3] & inmask));
    }
}

// LATE: launched after a decode step's attention as its programmatic
// dependent, so it runs beside it; before finishing it waits for that grid,
// so whatever follows on the stream still follows the attention. The key
// must lie in the window [seq_len - W, seq_len), which the step's selection
// does not read; a key before it sets KVR_DEVERR_POSITION.
template <int D, typename T, bool LATE>
__global__ void __launch_bounds__(256)
encode_kernel(const T *__restrict__ K, int Hkv, int64_t cap, int64_t tiles,
              const int32_t *__restrict__ pos0, int n_new, int64_t units, int blocks_per_unit,
              const int8_t *__restrict__ sgn, uint8_t *__restrict__ codes, int32_t *err,
              const int32_t *__restrict__ seq_len, int W)
{
    encode_body<D, T>(K, Hkv, cap, tiles, pos0, n_new, units, blocks_per_unit, sgn, codes, err);
    if constexpr (LATE) {
        if (blockIdx.x == 0)
            for (int64_t b = threadIdx.x; b < units / Hkv; b += blockDim.x)
                if ((int64_t)pos0[b] < (int64_t)seq_len[b] - W) set_err(err, KVR_DEVERR_POSITION);
        grid_dependency_wait();
    }
}

template <int D, typename T>
static kvr_status launch_encode(const LaunchCtx &c, const void *K, const int32_t *pos0, int n_new,
                                const int8_t *sgn, uint8_t *codes, int32_t *err,
                                const int32_t *late_seq_len, int W)
{
    const int64_t units = (int64_t)c.shape.B * c.shape.Hkv;
    const int bpu = (int)((n_new + 31) / 32 + 1);  // blocks a range of n_new tokens can touch
    const int64_t warps = units * bpu;
    const int64_t blocks = (warps + 7) / 8;
    const int64_t tiles = (c.shape.cap + 1023) / 1024;
    const T *Kt = static_cast<const T *>(K);
    if (!late_seq_len) {
        encode_kernel<D, T, false><<<(unsigned)blocks, 256, 0, c.stream>>>(
            Kt, c.shape.Hkv, c.shape.cap, tiles, pos0, n_new, units, bpu, sgn, codes, err, nullptr, 0);
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
    if (cudaLaunchKernelEx(&cfg, encode_kernel<D, T, true>, Kt, c.shape.Hkv, c.shape.cap, tiles, pos0,
                           n_new, units, bpu, sgn, codes, err, late_seq_len, W) != cudaSuccess)
        return KVR_ERR_CUDA;
    return check_launch();
}

kvr_status encode_dispatch(const LaunchCtx &c, const void *K, const int32_t *pos0, int n_new,
                           const int8_t *sgn, uint8_t *codes, int32_t *err,
                           const int32_t *late_seq_len, int W)
{
    const bool bf = c.shape.dtype == KVR_BF16;
    if (c.shape.d == 128)
        return bf ? launch_encode<128, __nv_bfloat16>(c, K, pos0, n_new, sgn, codes, err, late_seq_len, W)
                  : launch_encode<128, float>(c, K, pos0, n_new, sgn, codes, err, late_seq_len, W);
    return bf ? launch_encode<64, __nv_bfloat16>(c, K, pos0, n_new, sgn, codes, err, late_seq_len, W)
              : launch_encode<64, float>(c, K, pos0, n_new, sgn, codes, err, late_seq_len, W);
}

}  // namespace kvr
