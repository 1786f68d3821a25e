// kvr_noalloc.cu -- kvr_select for callers that cannot allocate device memory.
//
// Some hosts never let a library allocate on the GPU: plugin interfaces that
// hand a kernel only its input and output buffers, runtimes that reserve all
// device memory at start-up and expose no allocator, and latency-critical
// loops where a cudaMalloc (which can synchronise the device) is not allowed.
// kvr_select_static_scratch serves them: its scratch lives in a fixed
// file-scope device array that the module reserves on every GPU that loads
// this library, for as long as the process lives.
//
// The array's host-side name is only a stand-in for the device address, so
// the address is fetched with cudaGetSymbolAddress, with the device current,
// the first time the entry point runs in a device's context. It is kept per
// device together with that context: after a device reset the context (and
// the module's copy of the array) is new, and the address is fetched again.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "kvr_launch.h"

namespace {

constexpr size_t kScratchBytes = KVR_STATIC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_select_scratch[kScratchBytes];

std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices];
CUcontext g_scratch_ctx[kMaxDevices];

// cuCtxGetCurrent from the driver, looked up once (null if unavailable).
PFN_cuCtxGetCurrent_v4000 ctx_getter()
{
    static PFN_cuCtxGetCurrent_v4000 fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return (PFN_cuCtxGetCurrent_v4000) nullptr;
        return reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    }();
    return fn;
}

// Device address of g_select_scratch in the current device's context
// (set-up on first use in that context).
kvr_status scratch_for_current_device(void **out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KVR_ERR_CUDA;
    const PFN_cuCtxGetCurrent_v4000 get = ctx_getter();
    if (!get) return KVR_ERR_CUDA;
    // null before this thread's first runtime call on the device
    CUcontext ctx = nullptr;
    if (get(&ctx) != CUDA_SUCCESS) return KVR_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!ctx || !g_scratch_ptr[dev] || g_scratch_ctx[dev] != ctx) {
        // the lookup binds the device's primary context to this thread
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_select_scratch) != cudaSuccess || !p) return KVR_ERR_CUDA;
        if (get(&ctx) != CUDA_SUCCESS || !ctx) return KVR_ERR_CUDA;
        g_scratch_ptr[dev] = p;
        g_scratch_ctx[dev] = ctx;
    }
    *out = g_scratch_ptr[dev];
    return KVR_OK;
}

}  // namespace

extern "C" kvr_status kvr_select_static_scratch(const kvr_shape *shape,
                                                const kvr_select_params *p, const void *q,
                                                const void *K, const uint8_t *codes,
                                                const int32_t *seq_len,
                                                const int8_t *srht_sign, int32_t *out_idx,
                                                int32_t *out_count, int32_t *err_word,
                                                void *stream)
{
    void *scratch = nullptr;
    const kvr_status st = scratch_for_current_device(&scratch);
    if (st != KVR_OK) return st;
    // kvr_select validates every argument and returns KVR_ERR_WORKSPACE when
    // this shape needs more scratch than the fixed array holds.
    return kvr_select(shape, p, q, K, codes, seq_len, srht_sign, out_idx, out_count, scratch,
                      kScratchBytes, err_word, stream);
}
