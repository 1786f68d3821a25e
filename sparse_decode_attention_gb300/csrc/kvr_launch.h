// kvr_launch.h -- host-side glue between the C ABI (kvr_api.cu) and the
// kernel files. Arguments reaching these functions are already validated.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "kvr.h"

namespace kvr {

struct LaunchCtx {
    kvr_shape shape;
    cudaStream_t stream;
};

inline kvr_status check_launch()
{
    return cudaGetLastError() == cudaSuccess ? KVR_OK : KVR_ERR_CUDA;
}

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Opt a kernel into `bytes` of dynamic shared memory on the current device
// (once per kernel and device; later calls are a table lookup).
kvr_status raise_smem_limit(const void *kernel, int bytes);

// raise_smem_limit plus permission for cluster sizes above 8.
kvr_status prepare_cluster_kernel(const void *kernel, int smem_bytes);

// Streaming multiprocessors of the current device (queried once per device;
// 152 on GB300 if the query fails), for grid sizing.
int sm_count();

// Clusters of `cluster` CTAs of `kernel` (`threads` threads, `smem_bytes` of
// dynamic shared memory, limits already raised) resident on the current
// device at once; 0 if the query fails. Cached per device.
int max_active_clusters(const void *kernel, int cluster, int threads, int smem_bytes);

// Bytes of the bit-plane code buffer of one unit: ceil(cap/1024) tiles of d*128 bytes.
inline size_t codes_bytes_per_unit(int64_t cap, int d) { return (size_t)((cap + 1023) / 1024) * d * 128; }

// Select workspace plan (byte offsets).
struct SelectPlan {
    int64_t cap_pad;  // row length of the coarse-score array (multiple of 16)
    int64_t nblk;     // 32-token blocks per unit row of the score planes
    int64_t tiles;    // 1024-token code tiles per unit
    bool has_coarse;
    bool has_votes;   // magnitude-aware vote lists
    size_t off_planes, off_cand_idx, off_cand_score, off_cand_count, off_qbar, off_coarse;
    size_t off_votes;
    size_t bytes;
};

// Magnitude-aware vote lists (kvr_votes.cu): per unit and sub-block,
// kVoteStride uint16 entries: up to 256 (pattern | vote << 8), the count at
// index 256 (16-byte aligned rows).
constexpr int kVoteStride = 264;
struct VoteArgs {
    const void *q;
    const int8_t *sgn;
    int Hq, Hkv, G, nb;
    int lut[9];
    uint16_t *lists;
};
kvr_status vote_list_dispatch(const LaunchCtx &c, const void *q, const int8_t *sgn,
                              const int32_t *lut, uint16_t *lists);
SelectPlan plan_select(const kvr_shape &s, const kvr_select_params &p);

struct AttendPlan {
    size_t bytes;  // workspace bytes (0: partials merge on chip)
};
AttendPlan plan_attend(const kvr_shape &s, int kmax, int W);

// late_seq_len != null: the decode step's late form (after the attention, as
// its programmatic dependent; the keys must lie in the window of width W).
kvr_status encode_dispatch(const LaunchCtx &c, const void *K, const int32_t *pos0, int n_new,
                           const int8_t *sgn, uint8_t *codes, int32_t *err,
                           const int32_t *late_seq_len = nullptr, int W = 0);

// The attention fused into the selection's launch: value cache, logit
// scale (1/sqrt(d) in the caller's units) and output [B, Hq, d] fp32.
struct FusedAttend {
    const void *V;
    float scale;
    float *out;
};

// Whether kvr_select_attend runs as one launch for these arguments: query
// groups of up to 4 heads, exact rescoring, Hamming-ring votes.
bool select_attend_fusable(const kvr_shape &s, const kvr_select_params &p);

// att != null: the selection kernel also runs the step's attention (only
// when select_attend_fusable; KVR_ERR_UNSUPPORTED otherwise).
kvr_status select_dispatch(const LaunchCtx &c, const kvr_select_params &p, const SelectPlan &plan,
                           const void *q, const void *K, const uint8_t *codes,
                           const int32_t *seq_len, const int8_t *sgn, int32_t *out_idx,
                           int32_t *out_count, uint8_t *ws, int32_t *err,
                           const FusedAttend *att = nullptr);

kvr_status attend_dispatch(const LaunchCtx &c, const AttendPlan &plan, const void *q,
                           const void *K, const void *V, const int32_t *idx, int kmax,
                           const int32_t *count, const int32_t *seq_len, int W, int sink,
                           const int32_t *region_end, float scale, float *out, uint8_t *ws,
                           int32_t *err);

// Cache regions (kvr_regions.cu).
kvr_status regions_dispatch(cudaStream_t stream, int B, const int32_t *seq_len, int sink,
                            int local, int buffer, int init, int32_t *region_end, int32_t *err);

// Calibrated inner-product reranker (kvr_rsq.cu): fp32 tables of the
// 3-bit magnitude quantiser (bsq[i] = squared bin edge, bsq[0] = 0; lev[i] =
// level of bin i).
struct RsqTables {
    float bsq[8];
    float lev[8];
};
const RsqTables &rsq_tables();
kvr_status rsq_encode_dispatch(const LaunchCtx &c, const void *K, const int32_t *pos0, int n_new,
                               const int8_t *sgn, uint8_t *rec, int32_t *err, bool late = false);

// Tiered window cache (kvr_tiers.cu).
bool tier_shape_ok(const kvr_shape &s, int64_t n_win);
size_t tiered_attend_ws_bytes(const kvr_shape &s, int64_t n_win);
size_t tier_update_ws_bytes(const kvr_shape &s, int64_t n_win);
kvr_status tier_init_dispatch(const LaunchCtx &c, const kvr_tier_state &s, const int8_t *init,
                              const void *K, const void *V, const int32_t *seq_len, int32_t *err);
// wait_ns: limit of each wait for a bulk copy; withhold_last: the test hook
// of kvr_testing_tiered_withheld_copy (each CTA never issues its last copy).
kvr_status tiered_attend_dispatch(const LaunchCtx &c, const kvr_tier_state &s, const void *q,
                                  const void *K, const void *V, const int32_t *seq_len,
                                  float scale, float *out, float *mass, uint8_t *ws, int32_t *err,
                                  uint64_t wait_ns = 1000000000ull, bool withhold_last = false);
kvr_status tier_update_dispatch(const LaunchCtx &c, const kvr_tier_state &s, const float *mass,
                                const int32_t *seq_len, void *K, void *V, int32_t *stats,
                                uint8_t *ws, int32_t *err);

}  // namespace kvr
