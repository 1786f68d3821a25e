// kvr_device.cuh -- device helpers shared by the libkvr kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kvr.h"

namespace kvr {

constexpr unsigned kFull = 0xffffffffu;

// ---------------------------------------------------------------- elements

// Element traits: a 16-byte vector holds kVec elements.
template <typename T> struct Elem;
template <> struct Elem<float> {
    static constexpr int kVec = 4;
};
template <> struct Elem<__nv_bfloat16> {
    static constexpr int kVec = 8;
};

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Widen n (4 or 8) consecutive elements at a 16-byte aligned address.
template <int N> __device__ __forceinline__ void widen(const float *p, float (&x)[N])
{
#pragma unroll
    for (int i = 0; i < N; i += 4) {
        float4 v = *reinterpret_cast<const float4 *>(p + i);
        x[i] = v.x; x[i + 1] = v.y; x[i + 2] = v.z; x[i + 3] = v.w;
    }
}
template <int N> __device__ __forceinline__ void widen(const __nv_bfloat16 *p, float (&x)[N])
{
    static_assert(N % 4 == 0, "bf16 widen works on 8-byte groups");
#pragma unroll
    for (int i = 0; i < N; i += 8) {
        if (N - i >= 8) {
            uint4 v = *reinterpret_cast<const uint4 *>(p + i);
            x[i] = bf16_lo(v.x); x[i + 1] = bf16_hi(v.x);
            x[i + 2] = bf16_lo(v.y); x[i + 3] = bf16_hi(v.y);
            x[i + 4] = bf16_lo(v.z); x[i + 5] = bf16_hi(v.z);
            x[i + 6] = bf16_lo(v.w); x[i + 7] = bf16_hi(v.w);
        } else {
            uint2 v = *reinterpret_cast<const uint2 *>(p + i);
            x[i] = bf16_lo(v.x); x[i + 1] = bf16_hi(v.x);
            x[i + 2] = bf16_lo(v.y); x[i + 3] = bf16_hi(v.y);
        }
    }
}

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

// ---------------------------------------------------------------- attention rows

// The E consecutive elements of a row that lane `lane` holds (d = 32 E).
template <int E, typename T>
__device__ __forceinline__ void load_lane(const uint8_t *row, int lane, float (&x)[E])
{
    const T *p = reinterpret_cast<const T *>(row) + lane * E;
    if constexpr (sizeof(T) == 2 && E == 2) {
        const uint32_t w = *reinterpret_cast<const uint32_t *>(p);
        x[0] = bf16_lo(w);
        x[1] = bf16_hi(w);
    } else if constexpr (sizeof(T) == 4 && E == 2) {
        const float2 v = *reinterpret_cast<const float2 *>(p);
        x[0] = v.x;
        x[1] = v.y;
    } else {
        widen<E>(p, x);
    }
}

// Sum G per-lane values over the warp; lane l returns the total of head
// l / (32 / G). Splitting halves of the value set between partner lanes costs
// G - 1 + 5 - log2(G) shuffles instead of 5G.
template <int G>
__device__ __forceinline__ float reduce_heads(float (&v)[G], int lane)
{
    __syncwarp();
    constexpr int LG = (G >= 16) ? 4 : (G >= 8) ? 3 : (G >= 4) ? 2 : (G >= 2) ? 1 : 0;
#pragma unroll
    for (int s = 0; s < LG; s++) {
        const int o = 16 >> s;
        const int half = G >> (s + 1);
        const bool upper = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < half; i++) {
            const float send = upper ? v[i] : v[i + half];
            const float keep = upper ? v[i + half] : v[i];
            v[i] = keep + __shfl_xor_sync(kFull, send, o);
        }
    }
    float x = v[0];
#pragma unroll
    for (int o = 16 >> LG; o >= 1; o >>= 1) x += __shfl_xor_sync(kFull, x, o);
    return x;
}

// ---------------------------------------------------------------- tensor cores

// Shared-memory address of a generic pointer into this CTA's shared memory.
__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

// ---- warp-level tensor-core helpers: mma.sync m16n8k16, bf16 in, fp32 accumulate.
// Fragment layouts (g = lane / 4, c = lane % 4): A (16x16, row-major) holds
// (g, 2c..2c+1), (g+8, 2c..), (g, 2c+8..), (g+8, 2c+8..); B (16x8, k-major
// columns) holds (k = 2c..2c+1, n = g), (k = 2c+8.., n = g); C (16x8) holds
// (g, 2c..2c+1), (g+8, 2c..2c+1).

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void *p)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_u32(p)));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const void *p)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_u32(p)));
}

__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// (x0, x1) ~ hi + lo, hi = bf16(x), lo = bf16(x - hi), as bf16x2 words (x0 in
// the low half): about 16 bits of each value kept; r0, r1 are the values the
// tensor core sees (hi + lo).
__device__ __forceinline__ void split_bf16x2(float x0, float x1, uint32_t &hi, uint32_t &lo,
                                             float &r0, float &r1)
{
    const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
    hi = *reinterpret_cast<const uint32_t *>(&h);
    const float h0 = __uint_as_float(hi << 16), h1 = __uint_as_float(hi & 0xffff0000u);
    const __nv_bfloat162 l = __floats2bfloat162_rn(x0 - h0, x1 - h1);
    lo = *reinterpret_cast<const uint32_t *>(&l);
    r0 = h0 + __uint_as_float(lo << 16);
    r1 = h1 + __uint_as_float(lo & 0xffff0000u);
}

// ---------------------------------------------------------------- rotation

// Natural-order fast Walsh-Hadamard transform of one vector spread over a
// group of L lanes (aligned, power of two) that hold E consecutive elements
// each: element index = gl * E + r. Butterfly spans run ascending: first the
// spans inside a lane (h < E), then across lanes (h = E, 2E, ...). The lower
// element of a pair receives a + b and the upper a - b, each one fp32
// round-to-nearest addition, so every output matches the canonical
// sequential transform bit for bit. All 32 lanes of the warp must call it.
template <int E, int L>
__device__ __forceinline__ void fwht_lanes(float (&x)[E], int gl)
{
    __syncwarp();  // reconverge first: a diverged warp runs each shuffle once per branch
#pragma unroll
    for (int h = 1; h < E; h <<= 1) {
#pragma unroll
        for (int r = 0; r < E; r++) {
            if (r & h) continue;
            float a = x[r], b = x[r + h];
            x[r] = a + b;
            x[r + h] = a - b;
        }
    }
#pragma unroll
    for (int m = 1; m < L; m <<= 1) {
        const bool upper = (gl & m) != 0;
#pragma unroll
        for (int r = 0; r < E; r++) {
            float p = __shfl_xor_sync(kFull, x[r], m);
            x[r] = upper ? (p - x[r]) : (x[r] + p);
        }
    }
}

// Sign bits of the E elements a lane holds, placed at their bit position in
// the 32-bit code word (element i -> word i/32, bit i%32), OR-ed across the
// 32/E lanes sharing the word. Every lane returns its word; lanes with
// gl % (32/E) == 0 own it. All 32 lanes must call it.
template <int E>
__device__ __forceinline__ uint32_t sign_word(const float (&x)[E], int gl)
{
    __syncwarp();
    uint32_t bits = 0;
#pragma unroll
    for (int r = 0; r < E; r++)
        bits |= (x[r] < 0.0f ? 1u : 0u) << r;
    uint32_t v = bits << ((gl * E) & 31);
#pragma unroll
    for (int off = 1; off < 32 / E; off <<= 1)
        v |= __shfl_xor_sync(kFull, v, off);
    return v;
}

// ---------------------------------------------------------------- warp scans

__device__ __forceinline__ int warp_sum(int x)
{
    __syncwarp();
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) x += __shfl_xor_sync(kFull, x, o);
    return x;
}

// Sum N per-lane values over the warp (N a power of two <= 32); lane l gets
// the total of value l / (32 / N). Partner lanes split the value set in half
// at each of the first log2(N) steps: N - 1 + 5 - log2(N) shuffles in all.
template <int N, typename V>
__device__ __forceinline__ V warp_reduce_split(V (&v)[N])
{
    __syncwarp();
    const int lane = threadIdx.x & 31;
    constexpr int LG = (N >= 32) ? 5 : (N >= 16) ? 4 : (N >= 8) ? 3 : (N >= 4) ? 2 : (N >= 2) ? 1 : 0;
#pragma unroll
    for (int s = 0; s < LG; s++) {
        const int o = 16 >> s;
        const int half = N >> (s + 1);
        const bool upper = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < half; i++) {
            const V send = upper ? v[i] : v[i + half];
            const V keep = upper ? v[i + half] : v[i];
            v[i] = keep + __shfl_xor_sync(kFull, send, o);
        }
    }
    V x = v[0];
#pragma unroll
    for (int o = 16 >> LG; o >= 1; o >>= 1) x += __shfl_xor_sync(kFull, x, o);
    return x;
}

// Exclusive prefix sum over the lanes of a warp.
__device__ __forceinline__ int warp_exclusive_scan(int x)
{
    const int lane = threadIdx.x & 31;
    int s = x;
    __syncwarp();
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(kFull, s, o);
        s += (lane >= o) ? y : 0;
    }
    return s - x;
}

// Inclusive suffix sum over the lanes: lane l gets x[l] + x[l+1] + ... + x[31].
__device__ __forceinline__ int warp_suffix_sum(int x)
{
    const int lane = threadIdx.x & 31;
    __syncwarp();
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_down_sync(kFull, x, o);
        x += (lane + o < 32) ? y : 0;
    }
    return x;
}

// ---------------------------------------------------------------- block scans

// Exclusive prefix sum over the block of one value per thread; *total gets
// the block sum. blockDim.x must be a multiple of 32, <= 1024. scratch holds
// 33 ints. Contains __syncthreads: call from uniform control flow.
__device__ __forceinline__ int block_exclusive_scan(int v, int *scratch, int *total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    int x = v;
    __syncwarp();
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        int y = __shfl_up_sync(kFull, x, off);
        x += (lane >= off) ? y : 0;
    }
    if (lane == 31) scratch[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = (lane < nwarps) ? scratch[lane] : 0;
        int s = w;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            int y = __shfl_up_sync(kFull, s, off);
            s += (lane >= off) ? y : 0;
        }
        scratch[lane] = s - w;  // exclusive warp offsets
        if (lane == 31) scratch[32] = s;
    }
    __syncthreads();
    int res = scratch[warp] + x - v;
    *total = scratch[32];
    __syncthreads();
    return res;
}

// Two block-wide exclusive prefix sums in one pass (one value pair per
// thread): *ba / *bb get the sums of a / b over the lower threads. scratch
// holds 66 ints. Contains __syncthreads: call from uniform control flow.
__device__ __forceinline__ void block_exclusive_scan2(int a, int b, int *scratch, int *ba, int *bb)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    int x = a, y = b;
    __syncwarp();
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int xa = __shfl_up_sync(kFull, x, off);
        const int yb = __shfl_up_sync(kFull, y, off);
        x += (lane >= off) ? xa : 0;
        y += (lane >= off) ? yb : 0;
    }
    if (lane == 31) {
        scratch[warp] = x;
        scratch[33 + warp] = y;
    }
    __syncthreads();
    if (warp == 0) {
        const int wa = (lane < nwarps) ? scratch[lane] : 0;
        const int wb = (lane < nwarps) ? scratch[33 + lane] : 0;
        int sa = wa, sb = wb;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int ta = __shfl_up_sync(kFull, sa, off);
            const int tb = __shfl_up_sync(kFull, sb, off);
            sa += (lane >= off) ? ta : 0;
            sb += (lane >= off) ? tb : 0;
        }
        scratch[lane] = sa - wa;
        scratch[33 + lane] = sb - wb;
    }
    __syncthreads();
    *ba = scratch[warp] + x - a;
    *bb = scratch[33 + warp] + y - b;
    __syncthreads();
}

__device__ __forceinline__ void set_err(int32_t *err, int bit)
{
    if (err) atomicOr(err, bit);
}

// ---------------------------------------------------------------- TMA / mbarrier

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

// Make initialised mbarriers visible to the async (TMA) proxy and the cluster.
__device__ __forceinline__ void mbar_fence_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Default limit of a wait for a bulk copy: a copy lands within microseconds,
// so a wait still open after a second means the copy was never issued.
constexpr uint64_t kWaitLimitNs = 1000000000ull;

// Wait for phase `parity` of an mbarrier for at most limit_ns nanoseconds
// (device global timer); on expiry the error bit is set, false is returned
// and the caller carries on (its outputs are invalid; it must stop issuing
// copies and wait, again with a limit, for those still in flight).
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, int32_t *err,
                                          uint64_t limit_ns = kWaitLimitNs)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (;;) {
        for (int i = 0; i < 32; i++)
            if (mbar_try_wait(bar, parity)) return true;
        if (global_ns() - t0 > limit_ns) break;
    }
    set_err(err, KVR_DEVERR_TIMEOUT);
    return false;
}

// Order this thread's earlier generic-proxy shared-memory accesses before
// later async-proxy (bulk copy) accesses to the same bytes.
__device__ __forceinline__ void fence_proxy_async()
{
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}

// 1-D bulk copy global -> this CTA's shared memory, completing on `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::
            "r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Prefetch of the 128-byte lines of [p, p + bytes) into L2 (p 128-byte
// aligned, bytes a multiple of 128); nothing waits for it, nothing is written.
// Per-thread line prefetches issue in parallel across the warp; bulk-copy
// prefetches were measured slower (one copy engine per SM serialises them).
__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes)
{
    for (uint32_t o = 0; o < bytes; o += 128)
        asm volatile("prefetch.global.L2 [%0];\n" ::"l"(static_cast<const char *>(p) + o) : "memory");
}

// Prefetch of the one 128-byte line that holds p into L2.
__device__ __forceinline__ void prefetch_l2_line(const void *p)
{
    asm volatile("prefetch.global.L2 [%0];\n" ::"l"(p) : "memory");
}

// 16-byte asynchronous global -> shared copy (L2 only); src_bytes < 16 zero-fills.
__device__ __forceinline__ void cp_async16(void *dst, const void *src, int src_bytes = 16)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(dst)), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit()
{
    asm volatile("cp.async.commit_group;\n" ::: "memory");
}
// Wait until at most `n` of this thread's committed groups are still in flight.
template <int n> __device__ __forceinline__ void cp_async_wait()
{
    asm volatile("cp.async.wait_group %0;\n" ::"n"(n) : "memory");
}

// Programmatic dependent launch: wait until the preceding grid's memory is
// visible (no-op when the launch was not programmatic).
__device__ __forceinline__ void grid_dependency_wait()
{
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
}
__device__ __forceinline__ void grid_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

// Split cluster barrier: every thread of every CTA of the cluster arrives
// (release: its earlier memory accesses, including reads of other CTAs'
// shared memory, are complete) and later waits (acquire). Work between the
// two must not arrive at another cluster barrier.
__device__ __forceinline__ void cluster_arrive_release()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire()
{
    asm volatile("barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}

// fp32 -> uint32 key whose unsigned order is the float order; -0 maps as +0.
__device__ __forceinline__ uint32_t order_key(float s)
{
    uint32_t u = __float_as_uint(s);
    if (u == 0x80000000u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Inverse of order_key (-0 comes back as +0).
__device__ __forceinline__ float key_float(uint32_t k)
{
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

}  // namespace kvr
