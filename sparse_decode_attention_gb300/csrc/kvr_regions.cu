// kvr_regions.cu -- the Retrieval end of every batch entry's cache regions.
//
// Source: ParisKV, "Meccanismo di Aggiornamento a Finestra Scorrevole": the
// cache is kept as Sink (the first tokens), Local (recent tokens), Retrieval
// (older tokens, searched) and an Update Buffer taking the new tokens; when
// the buffer is full, the oldest local tokens move to Retrieval and the
// buffer's tokens become Local. With positions Sink [0, S), Retrieval
// [S, R), Local + buffer [R, N), the state is R per batch entry:
//   set-up:  R = max(min(S, N), N - L)
//   appends: R = max(R, min(S, N)); while N - R >= L + U: R += U
// (the sink takes the positions below S first; each time the buffer reaches
// U tokens, U local tokens retire to Retrieval).
#include "kvr_device.cuh"
#include "kvr_launch.h"

namespace kvr {

namespace {

__global__ void __launch_bounds__(128) regions_kernel(int B, const int32_t *__restrict__ seq_len,
                                                      int S, int L, int U, int init,
                                                      int32_t *__restrict__ region_end,
                                                      int32_t *err)
{
    // ordered after the previous kernel on the stream, and lets the next start
    grid_dependency_wait();
    grid_launch_dependents();
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    const int64_t N = seq_len[b];
    if (N < 0) {
        set_err(err, KVR_DEVERR_SEQ_LEN);
        return;
    }
    const int64_t s_eff = N < S ? N : S;
    int64_t R;
    if (init) {
        R = N - L;
        if (R < s_eff) R = s_eff;
    } else {
        R = region_end[b];
        if (R < s_eff) R = s_eff;
        // one step moves U tokens: at most (N - R) / U steps, done in one division
        if (N - R >= (int64_t)L + U) R += (int64_t)U * ((N - R - L) / U);
    }
    region_end[b] = (int32_t)R;
}

}  // namespace

kvr_status regions_dispatch(cudaStream_t stream, int B, const int32_t *seq_len, int sink,
                            int local, int buffer, int init, int32_t *region_end, int32_t *err)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((B + 127) / 128), 1, 1);
    cfg.blockDim = dim3(128, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, regions_kernel, B, seq_len, sink, local, buffer, init, region_end,
                           err) != cudaSuccess)
        return KVR_ERR_CUDA;
    return check_launch();
}

}  // namespace kvr
