// kvr_encode.cu -- append-time rotation and sign code of keys.
//
// ParisKV, "Centroidi Analitici Robusti al Drift": keys are rotated by a
// shared SRHT and assigned to the nearest fixed sign-pattern centroid; with
// the sub-block split of "Pipeline di Recupero Nativa su GPU in Due Stadi"
// the code of a key is the sign bits of its rotated vector.
//
// One key is spread over L = d / E lanes (E = 16 bytes / element size), so
// each lane issues one 16-byte load of its row and a warp covers 32 / L keys
// whose rows are contiguous when the positions are (coalesced). The FWHT runs
// in registers with warp shuffles; the code words are gathered with shuffles
// and written as 32-bit stores.
#include "kvr_device.cuh"
#include "kvr_launch.h"

namespace kvr {

template <int D, typename T>
__global__ void __launch_bounds__(256)
encode_kernel(const T *__restrict__ K, int Hkv, int64_t cap, const int32_t *__restrict__ pos0,
              int n_new, int64_t total, const int8_t *__restrict__ sgn,
              uint32_t *__restrict__ codes, int32_t *err)
{
    constexpr int E = Elem<T>::kVec;  // elements per lane
    constexpr int L = D / E;          // lanes per key
    constexpr int KPW = 32 / L;       // keys per warp
    constexpr int NW = D / 32;        // code words per key
    static_assert(L >= 32 / E && L <= 32, "lane split");

    const int lane = threadIdx.x & 31;
    const int gl = lane % L;
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t key = warp * KPW + lane / L;

    bool valid = key < total;
    int64_t base = 0;
    if (valid) {
        const int64_t unit = key / n_new;
        const int t = (int)(key - unit * n_new);
        const int b = (int)(unit / Hkv);
        const int64_t row = (int64_t)pos0[b] + t;
        if (row < 0 || row >= cap) {
            if (gl == 0) set_err(err, KVR_DEVERR_POSITION);
            valid = false;
        } else {
            base = unit * cap + row;
        }
    }
    float x[E];
    if (valid) {
        widen<E>(K + base * D + gl * E, x);
    } else {
#pragma unroll
        for (int r = 0; r < E; r++) x[r] = 0.0f;
    }
    // D x: exact sign flips, no multiply (nothing for the compiler to contract).
#pragma unroll
    for (int r = 0; r < E; r++)
        if (sgn[gl * E + r] < 0) x[r] = -x[r];
    fwht_lanes<E, L>(x, gl);
    const uint32_t w = sign_word<E>(x, gl);
    if (valid && (gl % (32 / E)) == 0)
        codes[base * NW + (gl * E) / 32] = w;
}

template <int D, typename T>
static kvr_status launch_encode(const LaunchCtx &c, const void *K, const int32_t *pos0, int n_new,
                                const int8_t *sgn, uint8_t *codes, int32_t *err)
{
    constexpr int L = D / Elem<T>::kVec;
    constexpr int KPB = 8 * (32 / L);  // 8 warps per block
    const int64_t total = (int64_t)c.shape.B * c.shape.Hkv * n_new;
    const int64_t blocks = (total + KPB - 1) / KPB;
    encode_kernel<D, T><<<(unsigned)blocks, 256, 0, c.stream>>>(
        static_cast<const T *>(K), c.shape.Hkv, c.shape.cap, pos0, n_new, total, sgn,
        reinterpret_cast<uint32_t *>(codes), err);
    return check_launch();
}

kvr_status encode_dispatch(const LaunchCtx &c, const void *K, const int32_t *pos0, int n_new,
                           const int8_t *sgn, uint8_t *codes, int32_t *err)
{
    const bool bf = c.shape.dtype == KVR_BF16;
    if (c.shape.d == 128)
        return bf ? launch_encode<128, __nv_bfloat16>(c, K, pos0, n_new, sgn, codes, err)
                  : launch_encode<128, float>(c, K, pos0, n_new, sgn, codes, err);
    return bf ? launch_encode<64, __nv_bfloat16>(c, K, pos0, n_new, sgn, codes, err)
              : launch_encode<64, float>(c, K, pos0, n_new, sgn, codes, err);
}

}  // namespace kvr
