// kvr_api.cu -- the extern "C" entry points of libkvr: argument validation,
// workspace plans and dispatch to the kernel files. Nothing here allocates
// device memory or synchronises, except kvr_read_error, whose job it is.
#include <algorithm>
#include <cstring>
#include <mutex>

#include "kvr_launch.h"
#include "kvr_testing.h"

namespace kvr {

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxC = 16384;

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

kvr_status check_shape(const kvr_shape *s)
{
    if (!s) return KVR_ERR_INVALID_ARG;
    if (s->B < 1 || s->Hkv < 1 || s->Hq < 1 || s->cap < 1) return KVR_ERR_INVALID_ARG;
    if (s->Hq % s->Hkv != 0) return KVR_ERR_INVALID_ARG;
    if (s->d != 64 && s->d != 128) return KVR_ERR_UNSUPPORTED;
    if (s->dtype != KVR_BF16 && s->dtype != KVR_F32) return KVR_ERR_UNSUPPORTED;
    const int G = s->Hq / s->Hkv;
    if (G > 16 || (G & (G - 1)) != 0) return KVR_ERR_UNSUPPORTED;  // 1, 2, 4, 8, 16
    if ((int64_t)s->B * s->Hkv > 65535) return KVR_ERR_UNSUPPORTED;  // grid.y
    if (s->cap > ((int64_t)1 << 31) - 1) return KVR_ERR_UNSUPPORTED;  // int32 indices
    return KVR_OK;
}

kvr_status check_params(const kvr_select_params *p)
{
    if (!p) return KVR_ERR_INVALID_ARG;
    if (p->C < 0 || p->C > kMaxC || p->k < 0 || p->k > p->C || p->W < 0)
        return KVR_ERR_INVALID_ARG;
    for (int i = 0; i < 9; i++)
        if (p->lut[i] < 0 || p->lut[i] > 15) return KVR_ERR_INVALID_ARG;
    if (p->flags & ~(KVR_SELECT_STORE_COARSE | KVR_SELECT_EARLY_INPUTS | KVR_SELECT_MAGNITUDE_VOTES))
        return KVR_ERR_INVALID_ARG;
    if (!aligned16(p->V_prefetch) || !aligned16(p->rsq_records)) return KVR_ERR_INVALID_ARG;
    if (p->sink < 0 || (reinterpret_cast<uintptr_t>(p->region_end) & 3u) != 0)
        return KVR_ERR_INVALID_ARG;
    return KVR_OK;
}

}  // namespace

namespace {

// Per device: kernels opted into more dynamic shared memory, and how much.
struct SmemTable {
    std::mutex mu;
    const void *kernel[kMaxDevices][64];
    int bytes[kMaxDevices][64];
};

// Raise `kernel`'s dynamic shared-memory limit on the current device to at
// least `bytes` (a call asking for more than an earlier one raises it again).
kvr_status raise_in(SmemTable &t, const void *kernel, int bytes, bool cluster)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KVR_ERR_CUDA;
    std::lock_guard<std::mutex> lock(t.mu);
    int slot = -1;
    for (int i = 0; i < 64; i++) {
        if (t.kernel[dev][i] == kernel) {
            if (t.bytes[dev][i] >= bytes) return KVR_OK;
            slot = i;
            break;
        }
        if (!t.kernel[dev][i] && slot < 0) slot = i;
    }
    if (slot < 0) return KVR_ERR_CUDA;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) !=
        cudaSuccess)
        return KVR_ERR_CUDA;
    if (cluster &&
        cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
            cudaSuccess)
        return KVR_ERR_CUDA;
    t.kernel[dev][slot] = kernel;
    t.bytes[dev][slot] = bytes;
    return KVR_OK;
}

SmemTable g_plain, g_cluster;

}  // namespace

int sm_count()
{
    static std::mutex mu;
    static int count[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 152;
    std::lock_guard<std::mutex> lock(mu);
    if (count[dev] <= 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
            n = 152;
        count[dev] = n;
    }
    return count[dev];
}

int max_active_clusters(const void *kernel, int cluster, int threads, int smem_bytes)
{
    static std::mutex mu;
    struct Entry {
        const void *kernel;
        int cluster, threads, smem, count;
    };
    static Entry table[kMaxDevices][128];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    std::lock_guard<std::mutex> lock(mu);
    int slot = -1;
    for (int i = 0; i < 128; i++) {
        const Entry &e = table[dev][i];
        if (e.kernel == kernel && e.cluster == cluster && e.threads == threads && e.smem == smem_bytes)
            return e.count;
        if (!e.kernel && slot < 0) slot = i;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cluster, 1, 1);
    cfg.blockDim = dim3(threads, 1, 1);
    cfg.dynamicSmemBytes = smem_bytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();  // a refused query is an answer of none, not a sticky error
        n = 0;
    }
    if (slot >= 0) table[dev][slot] = Entry{kernel, cluster, threads, smem_bytes, n};
    return n;
}

kvr_status raise_smem_limit(const void *kernel, int bytes)
{
    return raise_in(g_plain, kernel, bytes, false);
}

kvr_status prepare_cluster_kernel(const void *kernel, int smem_bytes)
{
    return raise_in(g_cluster, kernel, smem_bytes, true);
}

SelectPlan plan_select(const kvr_shape &s, const kvr_select_params &p)
{
    SelectPlan pl;
    const int64_t U = (int64_t)s.B * s.Hkv;
    pl.cap_pad = (int64_t)align_up((size_t)s.cap, 16);
    pl.nblk = (s.cap + 31) / 32;
    pl.tiles = (s.cap + 1023) / 1024;
    pl.has_coarse = (p.flags & KVR_SELECT_STORE_COARSE) != 0;
    size_t o = 0;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o = align_up(o + bytes, 256);
        return at;
    };
    pl.off_planes = take((size_t)U * 8 * pl.nblk * 4);
    pl.off_cand_idx = take((size_t)U * p.C * 4);
    pl.off_cand_score = take((size_t)U * p.C * 4);
    pl.off_cand_count = take((size_t)U * 4);
    pl.off_qbar = take((size_t)U * s.d * 4);
    pl.off_coarse = pl.has_coarse ? take((size_t)U * pl.cap_pad) : 0;
    pl.has_votes = (p.flags & KVR_SELECT_MAGNITUDE_VOTES) != 0;
    pl.off_votes = pl.has_votes ? take((size_t)U * (s.d / 8) * kVoteStride * 2) : 0;
    pl.bytes = o;
    return pl;
}

AttendPlan plan_attend(const kvr_shape &s, int kmax, int W)
{
    // the cluster kernel merges its partials in distributed shared memory
    (void)s;
    (void)kmax;
    (void)W;
    AttendPlan pl;
    pl.bytes = 0;
    return pl;
}

}  // namespace kvr

using namespace kvr;

extern "C" {

const char *kvr_status_string(kvr_status s)
{
    switch (s) {
    case KVR_OK: return "ok";
    case KVR_ERR_INVALID_ARG: return "invalid argument";
    case KVR_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case KVR_ERR_WORKSPACE: return "workspace too small";
    case KVR_ERR_CUDA: return "CUDA runtime error";
    case KVR_ERR_DEVICE: return "device-side error bits set";
    }
    return "unknown status";
}

int kvr_version(void) { return 200; }

size_t kvr_codes_bytes(const kvr_shape *shape)
{
    if (check_shape(shape) != KVR_OK) return 0;
    return (size_t)shape->B * shape->Hkv * codes_bytes_per_unit(shape->cap, shape->d);
}

kvr_status kvr_encode_keys(const kvr_shape *shape, const void *K, const int32_t *pos0, int n_new,
                           const int8_t *srht_sign, uint8_t *codes, int32_t *err_word,
                           void *stream)
{
    kvr_status st = check_shape(shape);
    if (st != KVR_OK) return st;
    if (n_new < 0) return KVR_ERR_INVALID_ARG;
    if (!K || !pos0 || !srht_sign || !codes) return KVR_ERR_INVALID_ARG;
    if (!aligned16(K) || !aligned16(codes)) return KVR_ERR_INVALID_ARG;
    if (n_new == 0) return KVR_OK;
    if ((int64_t)shape->B * shape->Hkv * n_new > ((int64_t)1 << 40)) return KVR_ERR_INVALID_ARG;
    LaunchCtx c{*shape, static_cast<cudaStream_t>(stream)};
    return encode_dispatch(c, K, pos0, n_new, srht_sign, codes, err_word);
}

size_t kvr_rsq_record_bytes(int d)
{
    return (d == 64 || d == 128) ? (size_t)6 * (d / 8) : 0;
}

kvr_status kvr_rsq_tables(float *bsq, float *lev)
{
    if (!bsq || !lev) return KVR_ERR_INVALID_ARG;
    const RsqTables &t = rsq_tables();
    std::memcpy(bsq, t.bsq, sizeof(t.bsq));
    std::memcpy(lev, t.lev, sizeof(t.lev));
    return KVR_OK;
}

kvr_status kvr_encode_rsq(const kvr_shape *shape, const void *K, const int32_t *pos0, int n_new,
                          const int8_t *srht_sign, uint8_t *records, int32_t *err_word,
                          void *stream)
{
    kvr_status st = check_shape(shape);
    if (st != KVR_OK) return st;
    if (n_new < 0) return KVR_ERR_INVALID_ARG;
    if (!K || !pos0 || !srht_sign || !records) return KVR_ERR_INVALID_ARG;
    if (!aligned16(K) || !aligned16(records)) return KVR_ERR_INVALID_ARG;
    if (n_new == 0) return KVR_OK;
    if ((int64_t)shape->B * shape->Hkv * n_new > ((int64_t)1 << 40)) return KVR_ERR_INVALID_ARG;
    LaunchCtx c{*shape, static_cast<cudaStream_t>(stream)};
    return rsq_encode_dispatch(c, K, pos0, n_new, srht_sign, records, err_word);
}

size_t kvr_select_workspace_size(const kvr_shape *shape, const kvr_select_params *p)
{
    if (check_shape(shape) != KVR_OK || check_params(p) != KVR_OK) return 0;
    return plan_select(*shape, *p).bytes;
}

kvr_status kvr_select_workspace_views(const kvr_shape *shape, const kvr_select_params *p,
                                      kvr_select_views *views)
{
    kvr_status st = check_shape(shape);
    if (st != KVR_OK) return st;
    if ((st = check_params(p)) != KVR_OK) return st;
    if (!views) return KVR_ERR_INVALID_ARG;
    const SelectPlan pl = plan_select(*shape, *p);
    views->coarse = pl.has_coarse ? pl.off_coarse : (size_t)-1;
    views->cand_idx = pl.off_cand_idx;
    views->cand_score = pl.off_cand_score;
    views->cand_count = pl.off_cand_count;
    views->qbar = pl.off_qbar;
    return KVR_OK;
}

kvr_status kvr_select(const kvr_shape *shape, const kvr_select_params *p, const void *q,
                      const void *K, const uint8_t *codes, const int32_t *seq_len,
                      const int8_t *srht_sign, int32_t *out_idx, int32_t *out_count,
                      void *workspace, size_t workspace_bytes, int32_t *err_word, void *stream)
{
    kvr_status st = check_shape(shape);
    if (st != KVR_OK) return st;
    if ((st = check_params(p)) != KVR_OK) return st;
    if (!q || !K || !codes || !seq_len || !srht_sign || !out_count || !workspace)
        return KVR_ERR_INVALID_ARG;
    if (p->k > 0 && !out_idx) return KVR_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(K) || !aligned16(codes) || !aligned16(out_idx) ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return KVR_ERR_INVALID_ARG;
    const SelectPlan pl = plan_select(*shape, *p);
    if (workspace_bytes < pl.bytes) return KVR_ERR_WORKSPACE;
    LaunchCtx c{*shape, static_cast<cudaStream_t>(stream)};
    return select_dispatch(c, *p, pl, q, K, codes, seq_len, srht_sign, out_idx, out_count,
                           static_cast<uint8_t *>(workspace), err_word);
}

kvr_status kvr_select_attend(const kvr_shape *shape, const kvr_select_params *p, const void *q,
                             const void *K, const void *V, const uint8_t *codes,
                             const int32_t *seq_len, const int8_t *srht_sign, float scale,
                             int32_t *out_idx, int32_t *out_count, float *out, void *workspace,
                             size_t workspace_bytes, int32_t *err_word, void *stream)
{
    kvr_status st = check_shape(shape);
    if (st != KVR_OK) return st;
    if ((st = check_params(p)) != KVR_OK) return st;
    if (!q || !K || !V || !codes || !seq_len || !srht_sign || !out_count || !out || !workspace)
        return KVR_ERR_INVALID_ARG;
    if (p->k > 0 && !out_idx) return KVR_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(K) || !aligned16(V) || !aligned16(codes) ||
        !aligned16(out_idx) || !aligned16(out) ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return KVR_ERR_INVALID_ARG;
    if (!(scale == scale)) return KVR_ERR_INVALID_ARG;
    const SelectPlan pl = plan_select(*shape, *p);
    if (workspace_bytes < pl.bytes) return KVR_ERR_WORKSPACE;
    LaunchCtx c{*shape, static_cast<cudaStream_t>(stream)};
    if (select_attend_fusable(*shape, *p)) {
        const FusedAttend att{V, scale, out};
        return select_dispatch(c, *p, pl, q, K, codes, seq_len, srht_sign, out_idx, out_count,
                               static_cast<uint8_t *>(workspace), err_word, &att);
    }
    if ((st = select_dispatch(c, *p, pl, q, K, codes, seq_len, srht_sign, out_idx, out_count,
                              static_cast<uint8_t *>(workspace), err_word)) != KVR_OK)
        return st;
    if (p->region_end)
        return attend_dispatch(c, plan_attend(*shape, p->k, 0), q, K, V, out_idx, p->k, out_count,
                               seq_len, 0, p->sink, p->region_end, scale, out, nullptr, err_word);
    return attend_dispatch(c, plan_attend(*shape, p->k, p->W), q, K, V, out_idx, p->k, out_count,
                           seq_len, p->W, 0, nullptr, scale, out, nullptr, err_word);
}

kvr_status kvr_decode_step(const kvr_shape *shape, const kvr_select_params *p, const void *q,
                           const void *K, const void *V, uint8_t *codes, const int32_t *seq_len,
                           const int32_t *pos_new, const int8_t *srht_sign, int32_t *out_idx,
                           int32_t *out_count, float scale, float *out, void *workspace,
                           size_t workspace_bytes, int32_t *err_word, void *stream)
{
    kvr_status st = check_shape(shape);
    if (st != KVR_OK) return st;
    if ((st = check_params(p)) != KVR_OK) return st;
    if (!pos_new || !out || !(scale == scale)) return KVR_ERR_INVALID_ARG;
    // validated before anything is enqueued: the attention's arguments too
    if (!V || !aligned16(V) || !aligned16(out)) return KVR_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(pos_new) & 3u) != 0) return KVR_ERR_INVALID_ARG;
    if (workspace_bytes < plan_select(*shape, *p).bytes) return KVR_ERR_WORKSPACE;
    // the appended key's code and record, checked here with the rest
    if (!K || !srht_sign || !codes || !aligned16(K) || !aligned16(codes)) return KVR_ERR_INVALID_ARG;
    uint8_t *records = const_cast<uint8_t *>(p->rsq_records);
    LaunchCtx c{*shape, static_cast<cudaStream_t>(stream)};
    // With a window (W >= 1, no regions) the appended key lies in it, where
    // the step's selection reads no code or record: they are written after
    // the attention, beside it (the encodes wait for the attention before
    // they finish). Otherwise they come first and the selection must not
    // start on its inputs early.
    const bool late = !p->region_end && p->W >= 1;
    kvr_select_params ps = *p;
    if (!late) {
        ps.flags &= ~KVR_SELECT_EARLY_INPUTS;
        if ((st = encode_dispatch(c, K, pos_new, 1, srht_sign, codes, err_word)) != KVR_OK) return st;
        if (records &&
            (st = rsq_encode_dispatch(c, K, pos_new, 1, srht_sign, records, err_word)) != KVR_OK)
            return st;
    }
    if ((st = kvr_select_attend(shape, &ps, q, K, V, codes, seq_len, srht_sign, scale, out_idx,
                                out_count, out, workspace, workspace_bytes, err_word, stream)) !=
        KVR_OK)
        return st;
    if (!late) return KVR_OK;
    if ((st = encode_dispatch(c, K, pos_new, 1, srht_sign, codes, err_word, seq_len, p->W)) != KVR_OK)
        return st;
    if (records && (st = rsq_encode_dispatch(c, K, pos_new, 1, srht_sign, records, err_word, true)) !=
                       KVR_OK)
        return st;
    return KVR_OK;
}

size_t kvr_attend_workspace_size(const kvr_shape *shape, int kmax, int W)
{
    if (check_shape(shape) != KVR_OK || kmax < 0 || W < 0) return 0;
    return plan_attend(*shape, kmax, W).bytes;
}

kvr_status kvr_sparse_attend(const kvr_shape *shape, const void *q, const void *K,
                             const void *V, const int32_t *idx, int kmax,
                             const int32_t *count, const int32_t *seq_len, int W,
                             float scale, float *out, void *workspace, size_t workspace_bytes,
                             int32_t *err_word, void *stream)
{
    kvr_status st = check_shape(shape);
    if (st != KVR_OK) return st;
    if (kmax < 0 || W < 0) return KVR_ERR_INVALID_ARG;
    if (!q || !K || !V || !count || !seq_len || !out) return KVR_ERR_INVALID_ARG;
    if (kmax > 0 && !idx) return KVR_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(K) || !aligned16(V) || !aligned16(out) ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return KVR_ERR_INVALID_ARG;
    if (!(scale == scale)) return KVR_ERR_INVALID_ARG;
    const AttendPlan pl = plan_attend(*shape, kmax, W);
    if (workspace_bytes < pl.bytes) return KVR_ERR_WORKSPACE;
    LaunchCtx c{*shape, static_cast<cudaStream_t>(stream)};
    return attend_dispatch(c, pl, q, K, V, idx, kmax, count, seq_len, W, 0, nullptr, scale, out,
                           static_cast<uint8_t *>(workspace), err_word);
}

kvr_status kvr_sparse_attend_regions(const kvr_shape *shape, const void *q, const void *K,
                                     const void *V, const int32_t *idx, int kmax,
                                     const int32_t *count, const int32_t *seq_len, int sink,
                                     const int32_t *region_end, float scale, float *out,
                                     void *workspace, size_t workspace_bytes, int32_t *err_word,
                                     void *stream)
{
    kvr_status st = check_shape(shape);
    if (st != KVR_OK) return st;
    if (kmax < 0 || sink < 0) return KVR_ERR_INVALID_ARG;
    if (!q || !K || !V || !count || !seq_len || !out || !region_end) return KVR_ERR_INVALID_ARG;
    if (kmax > 0 && !idx) return KVR_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(K) || !aligned16(V) || !aligned16(out) ||
        (reinterpret_cast<uintptr_t>(region_end) & 3u) != 0 ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return KVR_ERR_INVALID_ARG;
    if (!(scale == scale)) return KVR_ERR_INVALID_ARG;
    const AttendPlan pl = plan_attend(*shape, kmax, 0);
    if (workspace_bytes < pl.bytes) return KVR_ERR_WORKSPACE;
    LaunchCtx c{*shape, static_cast<cudaStream_t>(stream)};
    return attend_dispatch(c, pl, q, K, V, idx, kmax, count, seq_len, 0, sink, region_end, scale,
                           out, static_cast<uint8_t *>(workspace), err_word);
}

kvr_status kvr_regions_update(int B, const int32_t *seq_len, int sink, int local, int buffer,
                              int init, int32_t *region_end, int32_t *err_word, void *stream)
{
    if (B < 0 || sink < 0 || local < 0 || buffer < 1) return KVR_ERR_INVALID_ARG;
    if (B == 0) return KVR_OK;
    if (!seq_len || !region_end) return KVR_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(seq_len) & 3u) || (reinterpret_cast<uintptr_t>(region_end) & 3u))
        return KVR_ERR_INVALID_ARG;
    return regions_dispatch(static_cast<cudaStream_t>(stream), B, seq_len, sink, local, buffer,
                            init, region_end, err_word);
}

size_t kvr_ledger_bytes(int d)
{
    return (d == 64 || d == 128) ? (size_t)48 * d : 0;
}

}  // extern "C"

namespace {

kvr_status check_tiers(const kvr_shape *shape, const kvr_tier_state *s, bool need_ledger)
{
    kvr_status st = check_shape(shape);
    if (st != KVR_OK) return st;
    if (!s) return KVR_ERR_INVALID_ARG;
    if (s->n_win < 1 || s->n_win * KVR_WINDOW < shape->cap) return KVR_ERR_INVALID_ARG;
    if (!tier_shape_ok(*shape, s->n_win)) return KVR_ERR_UNSUPPORTED;
    if (!s->tier || !s->score || !s->has_ledger || !s->quota || !s->budget)
        return KVR_ERR_INVALID_ARG;
    if (need_ledger && (!s->ledger || !aligned16(s->ledger))) return KVR_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(s->score) & 7u) || (reinterpret_cast<uintptr_t>(s->budget) & 7u) ||
        (reinterpret_cast<uintptr_t>(s->quota) & 3u))
        return KVR_ERR_INVALID_ARG;
    return KVR_OK;
}

}  // namespace

extern "C" {

kvr_status kvr_tier_init(const kvr_shape *shape, const kvr_tier_state *state,
                         const int8_t *initial_tier, const void *K, const void *V,
                         const int32_t *seq_len, int32_t *err_word, void *stream)
{
    kvr_status st = check_tiers(shape, state, true);
    if (st != KVR_OK) return st;
    if (!initial_tier || !K || !V || !seq_len) return KVR_ERR_INVALID_ARG;
    if (!aligned16(K) || !aligned16(V)) return KVR_ERR_INVALID_ARG;
    LaunchCtx c{*shape, static_cast<cudaStream_t>(stream)};
    return tier_init_dispatch(c, *state, initial_tier, K, V, seq_len, err_word);
}

size_t kvr_tiered_attend_workspace_size(const kvr_shape *shape, int64_t n_win)
{
    if (check_shape(shape) != KVR_OK || n_win < 1 || n_win * KVR_WINDOW < shape->cap ||
        !tier_shape_ok(*shape, n_win))
        return 0;
    return tiered_attend_ws_bytes(*shape, n_win);
}

kvr_status kvr_sparse_attend_tiered(const kvr_shape *shape, const kvr_tier_state *state,
                                    const void *q, const void *K, const void *V,
                                    const int32_t *seq_len, float scale, float *out,
                                    float *window_mass, void *workspace,
                                    size_t workspace_bytes, int32_t *err_word, void *stream)
{
    kvr_status st = check_tiers(shape, state, true);
    if (st != KVR_OK) return st;
    if (!q || !K || !V || !seq_len || !out || !window_mass || !workspace)
        return KVR_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(K) || !aligned16(V) || !aligned16(out) ||
        (reinterpret_cast<uintptr_t>(window_mass) & 3u) ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return KVR_ERR_INVALID_ARG;
    if (!(scale == scale)) return KVR_ERR_INVALID_ARG;
    if (workspace_bytes < tiered_attend_ws_bytes(*shape, state->n_win)) return KVR_ERR_WORKSPACE;
    LaunchCtx c{*shape, static_cast<cudaStream_t>(stream)};
    return tiered_attend_dispatch(c, *state, q, K, V, seq_len, scale, out, window_mass,
                                  static_cast<uint8_t *>(workspace), err_word);
}

kvr_status kvr_testing_tiered_withheld_copy(const kvr_shape *shape, const kvr_tier_state *state,
                                            const void *q, const void *K, const void *V,
                                            const int32_t *seq_len, float scale, float *out,
                                            float *window_mass, void *workspace,
                                            size_t workspace_bytes, int32_t *err_word,
                                            void *stream, int64_t wait_ns)
{
    kvr_status st = check_tiers(shape, state, true);
    if (st != KVR_OK) return st;
    if (!q || !K || !V || !seq_len || !out || !window_mass || !workspace)
        return KVR_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(K) || !aligned16(V) || !aligned16(out) ||
        (reinterpret_cast<uintptr_t>(window_mass) & 3u) ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return KVR_ERR_INVALID_ARG;
    if (!(scale == scale) || wait_ns < 1 || wait_ns > 10000000000ll) return KVR_ERR_INVALID_ARG;
    if (workspace_bytes < tiered_attend_ws_bytes(*shape, state->n_win)) return KVR_ERR_WORKSPACE;
    LaunchCtx c{*shape, static_cast<cudaStream_t>(stream)};
    return tiered_attend_dispatch(c, *state, q, K, V, seq_len, scale, out, window_mass,
                                  static_cast<uint8_t *>(workspace), err_word, (uint64_t)wait_ns,
                                  true);
}

size_t kvr_tier_update_workspace_size(const kvr_shape *shape, int64_t n_win)
{
    if (check_shape(shape) != KVR_OK || n_win < 1 || n_win * KVR_WINDOW < shape->cap ||
        !tier_shape_ok(*shape, n_win))
        return 0;
    return tier_update_ws_bytes(*shape, n_win);
}

kvr_status kvr_tier_update(const kvr_shape *shape, const kvr_tier_state *state,
                           const float *window_mass, const int32_t *seq_len, void *K, void *V,
                           int32_t *stats, void *workspace, size_t workspace_bytes,
                           int32_t *err_word, void *stream)
{
    kvr_status st = check_tiers(shape, state, true);
    if (st != KVR_OK) return st;
    if (!window_mass || !seq_len || !K || !V || !workspace) return KVR_ERR_INVALID_ARG;
    if (!aligned16(K) || !aligned16(V) || (reinterpret_cast<uintptr_t>(window_mass) & 3u) ||
        (reinterpret_cast<uintptr_t>(stats) & 3u) ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return KVR_ERR_INVALID_ARG;
    if (workspace_bytes < tier_update_ws_bytes(*shape, state->n_win)) return KVR_ERR_WORKSPACE;
    LaunchCtx c{*shape, static_cast<cudaStream_t>(stream)};
    return tier_update_dispatch(c, *state, window_mass, seq_len, K, V, stats,
                                static_cast<uint8_t *>(workspace), err_word);
}

kvr_status kvr_read_error(int32_t *err_word, int32_t *bits_out, void *stream)
{
    if (!err_word) return KVR_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int32_t host = 0;
    if (cudaMemcpyAsync(&host, err_word, sizeof(host), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return KVR_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return KVR_ERR_CUDA;
    if (cudaMemsetAsync(err_word, 0, sizeof(int32_t), s) != cudaSuccess) return KVR_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return KVR_ERR_CUDA;
    if (bits_out) *bits_out = host;
    return host ? KVR_ERR_DEVICE : KVR_OK;
}

}  // extern "C"
