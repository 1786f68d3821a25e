/*
 * kvr.h -- C ABI of libkvr: retrieval-based sparse decode attention over a
 * long KV cache on one NVIDIA GB300 (sm_103a).
 *
 * Per decode step and KV head the library
 *   1. rotates keys and the query with a shared SRHT after l2 normalisation
 *      (ParisKV, "Centroidi Analitici Robusti al Drift"),
 *   2. codes each key by its nearest analytic sign-pattern centroid
 *      +-1/sqrt(8) per 8-dim sub-block, i.e. by its sign bits (same section),
 *   3. scores the codes against the query code with tiered collision votes
 *      and keeps a candidate set (ParisKV, "Pipeline di Recupero Nativa su GPU
 *      in Due Stadi"),
 *   4. rescores the candidates exactly with q.k and keeps the top-k,
 *   5. attends over the top-k tokens plus a local window of the newest tokens
 *      (ParisKV, "Problematica"; the local region of "Meccanismo di
 *      Aggiornamento a Finestra Scorrevole").
 *
 * Conventions shared by every call
 *   - Every pointer argument named as "device" is a device pointer into memory
 *     the caller allocated and owns; the library never allocates, frees or
 *     retains a pointer after the call returns.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and runs asynchronously: no call synchronises the host, so a
 *     sequence of calls can be captured into a CUDA graph.
 *   - Arguments are validated on the host before anything is enqueued; an
 *     invalid call returns an error status and enqueues nothing.
 *   - Conditions only the device can see (a sequence length beyond the
 *     capacity, a selected index outside the pool, a non-finite score) set
 *     bits of the optional device word `err_word` (int32, may be NULL) with
 *     atomicOr and are otherwise handled as documented per call; the caller
 *     clears the word and reads it when convenient (kvr_read_error).
 *
 * Layouts (row-major, element strides 1; "unit" = one (batch b, kv head h)):
 *   K, V      [B, Hkv, cap, d]  dtype KVR_BF16 or KVR_F32; token stride d.
 *   codes     bit-planes, kvr_codes_bytes(shape) bytes. A token's code has d
 *             bits; bit p is set iff coordinate p of its rotated vector is
 *             negative (sub-block j = bits 8j..8j+7). Per unit, tokens are
 *             grouped in tiles of 1024 = 32 blocks of 32; a tile is
 *             d*128 bytes laid out as [chunk c < d/4][block j < 32] 16-byte
 *             units of four uint32 words; word w of unit (c, j) holds code bit
 *             p = 4c + w of the 32 tokens of block j, bit i for token
 *             tile*1024 + 32j + i. Unit (b, h) starts at byte
 *             (b*Hkv + h) * ceil(cap/1024) * d*128.
 *   q         [B, Hq, d]        same dtype as K; query head g belongs to kv
 *             head g / (Hq/Hkv) (contiguous GQA groups).
 *   seq_len   [B] int32 device: tokens 0..seq_len[b]-1 of batch b are valid.
 *   srht_sign [d] int8 device: the +-1 diagonal of the rotation.
 * All base pointers must be 16-byte aligned.
 *
 * Host-resident caches (ParisKV, "Offloading tramite Indirizzamento Virtuale
 * Unificato": the full-precision KV stays in host memory and the GPU gathers
 * only the rows it needs, with no copy call): the K and V arguments of
 * kvr_encode_keys, kvr_encode_rsq, kvr_select and kvr_sparse_attend may point
 * to page-locked host memory mapped into the device's address space
 * (cudaHostAlloc, or cudaHostRegister with mapping; under unified addressing
 * the host pointer itself). The kernels then read those rows over the
 * host-GPU link. Pageable host memory is not allowed (the library does not
 * query pointer kinds). With kvr_select_params.rsq_records set, kvr_select
 * reads no K rows, so only the attention's gathers cross the link. The tier
 * calls need device memory.
 */
#ifndef KVR_H_
#define KVR_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum kvr_status {
    KVR_OK = 0,
    KVR_ERR_INVALID_ARG = 1, /* null / misaligned pointer, bad size or range */
    KVR_ERR_UNSUPPORTED = 2, /* head_dim not in {64, 128}, group size, dtype */
    KVR_ERR_WORKSPACE = 3,   /* workspace smaller than the *_workspace_size value */
    KVR_ERR_CUDA = 4,        /* a CUDA runtime call failed (launch, attribute) */
    KVR_ERR_DEVICE = 5       /* kvr_read_error found device-side error bits */
} kvr_status;

typedef enum kvr_dtype { KVR_F32 = 0, KVR_BF16 = 1 } kvr_dtype;

/* Device error bits written to err_word. */
#define KVR_DEVERR_SEQ_LEN 0x1    /* seq_len[b] > cap or < 0: unit treated as empty */
#define KVR_DEVERR_POSITION 0x2   /* encode row outside [0, cap): row skipped */
#define KVR_DEVERR_INDEX 0x4      /* attend index outside the pool: token skipped */
#define KVR_DEVERR_NONFINITE 0x8  /* NaN exact score: its order is unspecified */
#define KVR_DEVERR_TIMEOUT 0x10   /* a bounded wait for a bulk copy ran out: outputs invalid */

/* kvr_select_params.flags */
#define KVR_SELECT_STORE_COARSE 0x1 /* also write every pool key's coarse score to the
                                       workspace (diagnostics; costs time) */
#define KVR_SELECT_MAGNITUDE_VOTES 0x4 /* coarse votes from the centroids ranked by their
                                       similarity to the rotated query (ParisKV, "Pipeline di
                                       Recupero Nativa su GPU in Due Stadi", top-rho centroids
                                       per sub-space): with a_j = |zq_j|, zq = FWHT(D q_bar),
                                       the flip pattern x of a key's sub-block code against the
                                       query code costs f(x) = sum over the set bits j of x,
                                       ascending, of a_j (fp32 from +0); patterns ordered by
                                       (f, x) fill the tiers of sizes 1, 8, 28, 56, 70, 56, 28,
                                       8, 1 and vote lut[tier] (instead of lut[popcount(x)]).
                                       One more kernel launch; the scoring does more work */
#define KVR_SELECT_EARLY_INPUTS 0x2 /* the caller asserts that codes, K, V_prefetch,
                                       rsq_records, region_end, seq_len and srht_sign were
                                       complete before the previous kernel
                                       on the stream was launched (only q may come from that
                                       kernel): the call then starts reading them while that
                                       kernel still runs (programmatic dependent launch) */

/* Shape of one layer's cache and query. */
typedef struct kvr_shape {
    int B;         /* batch */
    int Hq;        /* query heads; a multiple of Hkv, Hq/Hkv <= 16 */
    int Hkv;       /* kv heads */
    int d;         /* head dim: 64 or 128 */
    int64_t cap;   /* token capacity per unit of K, V and codes */
    kvr_dtype dtype;
} kvr_shape;

/* Selection parameters. */
typedef struct kvr_select_params {
    int C;       /* candidate budget of the coarse stage, 0 <= C <= 16384 */
    int k;       /* final top-k, 0 <= k <= C */
    int W;       /* local window: tokens [N-W, N) are always attended and never
                    selected; the pool is [0, max(0, N-W)) */
    int lut[9];  /* vote weight by Hamming distance 0..8 between a key's and
                    the query's sub-block codes; each in [0, 15] */
    int flags;   /* KVR_SELECT_* bits, 0 for none */
    const void *V_prefetch; /* optional hint, or NULL: the device V cache [B, Hkv, cap, d]
                               (shape->dtype, 16-byte aligned) of a kvr_sparse_attend
                               that follows; the selected tokens' V rows and the local
                               window's K and V rows are then prefetched into L2 as soon
                               as they are known. Results are unchanged. */
    const uint8_t *rsq_records; /* optional, or NULL: the device records [B, Hkv, cap,
                               kvr_rsq_record_bytes(d)] of the pool keys (kvr_encode_rsq);
                               when set, the candidates are ranked by the calibrated
                               estimate from the records instead of exact q_bar . k, and
                               K is not read (cand_score then holds the estimates) */
    int sink;               /* cache regions (ParisKV, "Meccanismo di Aggiornamento a
                               Finestra Scorrevole"): the first `sink` tokens are the Sink,
                               always attended, never candidates; 0 = none */
    const int32_t *region_end; /* optional, or NULL: device int32 [B], the end R_b of the
                               Retrieval region (kvr_regions_update); [R_b, N) is Local
                               plus the Update Buffer. NULL: R_b = N - W. The pool is
                               [S', R') with S' = min(sink, N), R' = min(max(R_b, S'), N) */
} kvr_select_params;

/* Byte offsets of the inspectable parts of the select workspace after a
   kvr_select call (see kvr_select_workspace_views). */
typedef struct kvr_select_views {
    size_t coarse;     /* uint8 [B*Hkv, roundup(cap, 16)]: coarse score of every pool
                          key; SIZE_MAX unless flags has KVR_SELECT_STORE_COARSE */
    size_t cand_idx;   /* int32 [B*Hkv, C]: candidate indices, ascending */
    size_t cand_score; /* float [B*Hkv, C]: exact q_bar.k of cand_idx entries */
    size_t cand_count; /* int32 [B*Hkv]: C' = min(C, pool) */
    size_t qbar;       /* float [B*Hkv, d]: group-mean query */
} kvr_select_views;

/* Human-readable name of a status. Never NULL. */
const char *kvr_status_string(kvr_status s);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int kvr_version(void);

/* Bytes of the code buffer of a cache of this shape (layout above), 0 when
   the shape is invalid. */
size_t kvr_codes_bytes(const kvr_shape *shape);

/*
 * kvr_encode_keys -- append-time rotation and sign code (steps 1-2).
 * Source: ParisKV, "Centroidi Analitici Robusti al Drift" (rotation and
 * analytic centroids) and "Pipeline di Recupero Nativa su GPU in Due Stadi"
 * (sub-blocks, nearest centroid per sub-block).
 *
 * For every unit (b, h) and t in [0, n_new): row r = pos0[b] + t of K is
 * transformed as z = FWHT(D * k) in fp32 (natural Hadamard order, butterfly
 * spans ascending; D = diag(srht_sign)) and the code bits of token r in
 * `codes` receive the sign bits of z; the bits of every other token are kept.
 * The l2 normalisation and the 1/sqrt(d) factor are positive scales and leave
 * the code unchanged, so they are not computed.
 *   K         device, [B, Hkv, cap, d] of shape->dtype (read).
 *   pos0      device int32 [B]: first row to encode per batch entry.
 *   n_new     rows per unit, >= 0 (0 enqueues nothing).
 *   srht_sign device int8 [d], entries +1 or -1.
 *   codes     device, kvr_codes_bytes(shape) bytes (bits of the rows only).
 *   err_word  device int32 or NULL: KVR_DEVERR_POSITION for rows outside
 *             [0, cap) (those rows are skipped).
 */
kvr_status kvr_encode_keys(const kvr_shape *shape, const void *K, const int32_t *pos0,
                           int n_new, const int8_t *srht_sign, uint8_t *codes,
                           int32_t *err_word, void *stream);

/*
 * Calibrated inner-product reranking (an alternative to exact rescoring).
 * Source: ParisKV, "Pipeline di Recupero Nativa su GPU in Due Stadi",
 * candidate reranking: each sub-space direction of a rotated key is coded
 * with a sign bit and 3 magnitude bits from the Beta prior the rotation
 * induces, a per-key, per-sub-space scale corrects the quantisation, and the
 * score is estimated without the full-precision key.
 *
 * Record of a key (kvr_rsq_record_bytes(d) = 6 d/8 bytes): with z = FWHT(D k)
 * and per sub-block b of 8 coordinates z_b:
 *   d/8 little-endian 32-bit words, nibble j (bits 4j .. 4j+3) of word b
 *   = mag_j | sign_j << 3 for coordinate 8b + j (sign_j = z_j < 0, the
 *   code bit); the magnitude mag_j = #{i in 1..7 :
 *   fl(z_j^2) >= fl(bsq[i] s)} with s = fma chain of z_j^2 over j ascending;
 *   then d/8 bf16 scales w_b = bf16(s / c), c = fma chain of |z_j| lev[mag_j]
 *   (0 when c = 0).
 * bsq / lev (kvr_rsq_tables): fl of the squared edges of the 8 equal-
 * probability bins of |u_j| for a uniformly random unit vector in R^8 (u_j^2 ~
 * Beta(1/2, 7/2)) and fl of each bin's conditional mean of |u_j|.
 * Estimate of a record against zq = FWHT(D q_bar): per block e_b = fma chain
 * over j ascending of (+-lev[mag_j]) zq_j from +0, t_b = w_b e_b, then
 * butterfly sums over 16 block slots (empty slots +0) with spans 8, 4, 2, 1.
 * ======================================================================== */

/* Bytes of one key's record, 0 for an unsupported d. */
size_t kvr_rsq_record_bytes(int d);

/* The quantiser tables (host): bsq[8] (bsq[0] = 0) and lev[8]. */
kvr_status kvr_rsq_tables(float *bsq, float *lev);

/*
 * kvr_encode_rsq -- records of rows [pos0[b], pos0[b] + n_new) of every unit
 * (append time, next to kvr_encode_keys).
 *   K        device [B, Hkv, cap, d] of shape->dtype.
 *   records  device [B, Hkv, cap, kvr_rsq_record_bytes(d)] bytes, 16-byte aligned.
 *   err_word KVR_DEVERR_POSITION for rows outside [0, cap) (skipped).
 */
kvr_status kvr_encode_rsq(const kvr_shape *shape, const void *K, const int32_t *pos0, int n_new,
                          const int8_t *srht_sign, uint8_t *records, int32_t *err_word,
                          void *stream);

/* Bytes of device workspace kvr_select needs for this shape and params. */
size_t kvr_select_workspace_size(const kvr_shape *shape, const kvr_select_params *p);

/* Fills *views with byte offsets into the select workspace. */
kvr_status kvr_select_workspace_views(const kvr_shape *shape, const kvr_select_params *p,
                                      kvr_select_views *views);

/*
 * kvr_select -- coarse scoring, candidate set, exact rescoring, top-k
 * (steps 1-4 for the query).
 * Source: ParisKV, "Pipeline di Recupero Nativa su GPU in Due Stadi" (coarse
 * collision votes prune to a candidate set); exact q.k rescoring of the
 * candidates replaces the page's code-only reranker.
 *
 * Per unit (b, h), with N = seq_len[b], pool = max(0, N - W),
 * C' = min(C, pool), k' = min(k, C'):
 *   q_bar  = mean of the G = Hq/Hkv query heads of the group, summed left to
 *            right in fp32 and divided by G;
 *   qcode  = sign code of q_bar (as kvr_encode_keys);
 *   s_i    = sum over sub-blocks j of lut[popcount(code_i[j] ^ qcode[j])];
 *   cand   = the first C' pool tokens by (s desc, index asc);
 *   S_i    = q_bar . k_i in fp32: 16 contiguous chunks of d/16 dims, each an
 *            fma chain from +0 over its dims ascending, then butterfly sums
 *            over chunk spans 8, 4, 2, 1; the result of chunk 0;
 *   top    = the first k' candidates by (S desc, index asc), -0 == +0.
 * out_idx[b, h, 0..k'-1] receives `top` ascending, the rest of the row -1;
 * out_count[b, h] = k'.
 *   q         device [B, Hq, d] of shape->dtype.
 *   K, codes  device, as in the layouts above; codes of rows [0, pool) must
 *             be current (kvr_encode_keys).
 *   seq_len   device int32 [B]; a value outside [0, cap] sets
 *             KVR_DEVERR_SEQ_LEN and the unit selects nothing.
 *   out_idx   device int32 [B, Hkv, p->k];  out_count device int32 [B, Hkv].
 *   workspace device, >= kvr_select_workspace_size bytes, 256-byte aligned;
 *             contents on entry are ignored; see kvr_select_workspace_views.
 */
kvr_status kvr_select(const kvr_shape *shape, const kvr_select_params *p, const void *q,
                      const void *K, const uint8_t *codes, const int32_t *seq_len,
                      const int8_t *srht_sign, int32_t *out_idx, int32_t *out_count,
                      void *workspace, size_t workspace_bytes, int32_t *err_word,
                      void *stream);

/*
 * kvr_select_attend -- kvr_select followed by the attention over its output,
 * as one call: steps 3-5 of a decode step (ParisKV, "Pipeline di Recupero
 * Nativa su GPU in Due Stadi" for the selection; "Problematica" and
 * "Meccanismo di Aggiornamento a Finestra Scorrevole" for the attention).
 *
 * out_idx / out_count are exactly kvr_select's. out [B, Hq, d] fp32 is the
 * attention of kvr_sparse_attend over {out_idx[b,h,0..k'-1]} U [N - W, N)
 * (kvr_sparse_attend_regions over the Sink, the top-k and [region_end[b], N)
 * when p->region_end is set), within the same floating-point tolerance of
 * the exact value; the summation order differs from the separate calls, so
 * the bits may too.
 * With Hq/Hkv <= 4, exact rescoring (p->rsq_records NULL) and Hamming-ring
 * votes, both run in one kernel launch: each thread-block cluster that
 * selects a unit's tokens attends over them, each CTA over the winners it
 * rescored plus a share of the window (and Sink), so the selected indices
 * never leave the chip before the attention; otherwise the two calls run one
 * after the other. p->V_prefetch is ignored (V is read anyway).
 *   q, K, codes, seq_len, srht_sign, p, out_idx, out_count, workspace: as
 *             in kvr_select (the workspace as kvr_select_workspace_size).
 *   V         device [B, Hkv, cap, d] (shape->dtype), or page-locked host
 *             memory as for kvr_sparse_attend.
 *   scale     logit scale (normally 1/sqrt(d)); NaN is KVR_ERR_INVALID_ARG.
 *   out       device float [B, Hq, d] (written).
 */
kvr_status kvr_select_attend(const kvr_shape *shape, const kvr_select_params *p, const void *q,
                             const void *K, const void *V, const uint8_t *codes,
                             const int32_t *seq_len, const int8_t *srht_sign, float scale,
                             int32_t *out_idx, int32_t *out_count, float *out, void *workspace,
                             size_t workspace_bytes, int32_t *err_word, void *stream);

/*
 * kvr_decode_step -- one decode step of every unit in one call: the code
 * (and, with p->rsq_records, the reranker record) of the appended key at row
 * pos_new[b], kvr_select, and the attention over its output (over the cache
 * regions when p->region_end is set, else over the top-k and the window W),
 * all enqueued on `stream` (the selection and attention as kvr_select_attend,
 * one launch where it fuses them). Order: with p->region_end set or W == 0, the
 * encodes first, then the selection (KVR_SELECT_EARLY_INPUTS is ignored: it
 * follows the encode that writes its codes), then the attention. With W >= 1
 * and no regions the appended key must lie in the window,
 * pos_new[b] >= seq_len[b] - W (the decode case: pos_new[b] = seq_len[b] - 1),
 * where the selection reads no code or record; the selection and attention
 * come first (KVR_SELECT_EARLY_INPUTS as in kvr_select) and the encodes run
 * beside the attention, finishing after it, so work enqueued after this call
 * follows all of it; a key before the window sets KVR_DEVERR_POSITION.
 * Arguments as in those calls; out_idx must hold p->k entries per unit; the
 * attention needs no workspace. Validation errors of any part are returned
 * before that part is enqueued; the parts before it stay enqueued.
 */
kvr_status kvr_decode_step(const kvr_shape *shape, const kvr_select_params *p, const void *q,
                           const void *K, const void *V, uint8_t *codes, const int32_t *seq_len,
                           const int32_t *pos_new, const int8_t *srht_sign, int32_t *out_idx,
                           int32_t *out_count, float scale, float *out, void *workspace,
                           size_t workspace_bytes, int32_t *err_word, void *stream);

/* Size of the fixed device scratch array behind kvr_select_static_scratch. */
#define KVR_STATIC_SCRATCH_BYTES ((size_t)16 << 20)

/*
 * kvr_select_static_scratch -- kvr_select without a caller-provided
 * workspace. No counterpart in the paper: this is a deployment variant.
 *
 * For callers that may not allocate device memory at all: plugin interfaces
 * that hand a kernel only its inputs and outputs, runtimes that reserve every
 * byte of device memory up front and expose no allocator, and hot loops where
 * a cudaMalloc (which can synchronise the device) is not acceptable. The
 * scratch kvr_select needs lives instead in a fixed file-scope device array of
 * KVR_STATIC_SCRATCH_BYTES (16 MiB) that every GPU loading this library holds
 * until the process exits; this call allocates and frees nothing.
 *
 * Arguments, results and errors are those of kvr_select minus the workspace.
 * A shape / params pair whose kvr_select_workspace_size exceeds
 * KVR_STATIC_SCRATCH_BYTES returns KVR_ERR_WORKSPACE and enqueues nothing
 * (for scale: 8 units of 1M tokens at C = 16384 need about 11 MiB, 8 units of
 * 128K tokens at C = 8192 about 2.1 MiB).
 *   - Set-up: the first call on a device looks up the array's device address
 *     with that device current (cudaGetSymbolAddress); make that first call
 *     before any stream capture on the device. The address is kept with the
 *     device's context: after a device reset (a new context) the next call
 *     looks it up again, so it too must come before any stream capture.
 *   - Every call on a device shares the one array and leaves its contents
 *     behind; kvr_select reads nothing from scratch that the same call did not
 *     write first, so no clearing is needed. Calls whose GPU work overlaps
 *     (different streams, or different host threads) race on the array: order
 *     them on one stream or serialise them.
 */
kvr_status kvr_select_static_scratch(const kvr_shape *shape, const kvr_select_params *p,
                                     const void *q, const void *K, const uint8_t *codes,
                                     const int32_t *seq_len, const int8_t *srht_sign,
                                     int32_t *out_idx, int32_t *out_count, int32_t *err_word,
                                     void *stream);

/*
 * Cache regions (ParisKV, "Meccanismo di Aggiornamento a Finestra
 * Scorrevole"): for unbounded generation a unit's tokens are Sink [0, S),
 * Retrieval [S, R) (searched by kvr_select), and Local followed by the Update
 * Buffer [R, N) (always attended, like the Sink). New tokens enter the
 * buffer; when it holds U tokens the U oldest local tokens move to Retrieval.
 *
 * kvr_regions_update -- the Retrieval end of every batch entry after appends:
 *   init != 0: region_end[b] = max(min(S, N), N - L)   (set-up, buffer empty)
 *   then:      R = max(region_end[b], min(S, N));
 *              while (N - R >= L + U) R += U;  region_end[b] = R
 * with N = seq_len[b]. One launch of one small kernel.
 *   seq_len     device int32 [B]; a negative value sets KVR_DEVERR_SEQ_LEN and
 *               leaves the entry unchanged.
 *   region_end  device int32 [B] (read unless init, written).
 *   sink, local >= 0; buffer >= 1; else KVR_ERR_INVALID_ARG.
 */
kvr_status kvr_regions_update(int B, const int32_t *seq_len, int sink, int local, int buffer,
                              int init, int32_t *region_end, int32_t *err_word, void *stream);

/* Bytes of device workspace kvr_sparse_attend needs (kmax = row length of idx). */
size_t kvr_attend_workspace_size(const kvr_shape *shape, int kmax, int W);

/*
 * kvr_sparse_attend -- fused gather + online-softmax GQA attention over the
 * selected tokens plus the local window (step 5).
 * Source: ParisKV, "Problematica" (attention restricted to a top-k subset of
 * past tokens) and "Meccanismo di Aggiornamento a Finestra Scorrevole"
 * (recent tokens kept in a local region).
 *
 * Per unit (b, h) with N = seq_len[b] and T = {idx[b,h,0..count[b,h]-1]} U
 * [max(0, N-W), N), for every query head g of the group:
 *   out[b, g, :] = sum_{t in T} softmax_t(scale * q_g . k_t) v_t,
 * accumulated in fp32 with an online softmax; an empty T gives zeros.
 *   q            device [B, Hq, d]; K, V device [B, Hkv, cap, d] (shape->dtype).
 *   idx          device int32 [B, Hkv, kmax] (e.g. kvr_select's out_idx);
 *                entries must lie in [0, N-W): others set KVR_DEVERR_INDEX and
 *                are skipped.
 *   count        device int32 [B, Hkv], each clamped to [0, kmax].
 *   out          device float [B, Hq, d] (written).
 *   workspace    device, >= kvr_attend_workspace_size bytes, 256-byte aligned.
 */
kvr_status kvr_sparse_attend(const kvr_shape *shape, const void *q, const void *K,
                             const void *V, const int32_t *idx, int kmax,
                             const int32_t *count, const int32_t *seq_len, int W,
                             float scale, float *out, void *workspace, size_t workspace_bytes,
                             int32_t *err_word, void *stream);

/*
 * kvr_sparse_attend_regions -- kvr_sparse_attend over the cache regions:
 * T = [0, S') U {idx[b,h,0..count-1]} U [R', N) with S' = min(sink, N) and
 * R' = min(max(region_end[b], S'), N); idx entries must lie in [S', R')
 * (others set KVR_DEVERR_INDEX and are skipped). Other arguments as in
 * kvr_sparse_attend; region_end is required (device int32 [B]).
 */
kvr_status kvr_sparse_attend_regions(const kvr_shape *shape, const void *q, const void *K,
                                     const void *V, const int32_t *idx, int kmax,
                                     const int32_t *count, const int32_t *seq_len, int sink,
                                     const int32_t *region_end, float scale, float *out,
                                     void *workspace, size_t workspace_bytes, int32_t *err_word,
                                     void *stream);

/* ======================================================================== *
 * Tiered window cache.
 * Source: QEvict, "Metodologia: QEvict" (contiguous windows routed between a
 * full-precision tier, a recoverable INT2 tier and an evicted tier under a
 * fixed memory budget) and "Meccanismi Chiave" (per-window routing,
 * cumulative attention scores, demotion / promotion, write-once quantisation
 * ledger, GQA).
 *
 * Windows are KVR_WINDOW = 64 tokens: window w of a unit holds tokens
 * [64w, 64w + 64). With N = seq_len[b], windows w < N/64 are closed and carry
 * a tier; the newest partial window (if N % 64 != 0) is open, bf16 and always
 * attended. K and V must be bf16.
 *
 * INT2 form, per token and per group of 32 contiguous channels, for K and V:
 *   z    = the fp16 value rounded toward -inf from the group minimum,
 *   s    = the smallest fp16 >= fl((max - z) / 3) with fmaf(3, s, z) >= max,
 *   code = clamp(rint((x - z) / s), 0, 3), 0 when s == 0,
 *   value = fmaf(code, s, z) (fp32); a promoted window stores the bf16
 *   nearest to each value in K, V.
 * Ledger of one window: kvr_ledger_bytes(d) = 48 d bytes laid out as
 *   [K codes: token t < 64, group g < d/32, 8 bytes, element j of the group at
 *   byte j/4, bits 2 (j%4)][K params: t, g, (fp16 scale, fp16 zero), little
 *   endian][V codes][V params].
 * ======================================================================== */

#define KVR_WINDOW 64
#define KVR_TIER_BF16 0
#define KVR_TIER_INT2 1
#define KVR_TIER_EVICTED 2

#define KVR_DEVERR_TIER 0x20   /* tier value outside {0, 1, 2}: window treated as evicted */
#define KVR_DEVERR_RANGE 0x40  /* an INT2 group's range does not fit fp16: its ledger
                                  entry is unspecified */

/* Device state of the tiered cache. Every array is caller-allocated device
   memory; "unit" u = b * Hkv + h. */
typedef struct kvr_tier_state {
    int64_t n_win;       /* windows per unit, >= ceil(cap / 64), <= 16384 */
    int8_t *tier;        /* [U, n_win] KVR_TIER_*; entries of non-closed windows are 0 */
    int64_t *score;      /* [U, n_win] cumulative score, sum of llrint(mass * 2^32) */
    uint8_t *has_ledger; /* [U, n_win] 1 once the window's ledger holds its INT2 form */
    uint8_t *ledger;     /* [U, n_win, kvr_ledger_bytes(d)], 16-byte aligned */
    int32_t *quota;      /* [U] bf16 windows kept (set by kvr_tier_init) */
    int64_t *budget;     /* [U] byte budget of the closed windows (set by kvr_tier_init) */
} kvr_tier_state;

/* Bytes of one window's ledger (48 d), 0 for an unsupported d. */
size_t kvr_ledger_bytes(int d);

/*
 * kvr_tier_init -- set up the tiers of every unit.
 * For each unit with N = seq_len[b]: windows w < N/64 take initial_tier[u, w]
 * (KVR_TIER_*), later windows bf16; scores 0; every closed INT2 window gets its
 * ledger quantised from its current K, V rows (has_ledger 1), the others
 * has_ledger 0; quota[u] = the number of closed bf16 windows and budget[u] =
 * quota * 64 * 2 * 2d + (closed INT2 windows) * kvr_ledger_bytes(d).
 *   initial_tier device int8 [U, n_win]; K, V device bf16 [B, Hkv, cap, d].
 *   err_word     KVR_DEVERR_TIER, KVR_DEVERR_RANGE, KVR_DEVERR_SEQ_LEN (unit
 *                left with every window bf16 and budget 0).
 */
kvr_status kvr_tier_init(const kvr_shape *shape, const kvr_tier_state *state,
                         const int8_t *initial_tier, const void *K, const void *V,
                         const int32_t *seq_len, int32_t *err_word, void *stream);

/* Bytes of device workspace kvr_sparse_attend_tiered needs. */
size_t kvr_tiered_attend_workspace_size(const kvr_shape *shape, int64_t n_win);

/*
 * kvr_sparse_attend_tiered -- attention over the bf16 and INT2 windows, with
 * the attention mass of every window (the tiered form of kvr_sparse_attend).
 *
 * Per unit and query head g of the group, over T = tokens of closed bf16
 * windows (from K, V) U tokens of closed INT2 windows (their ledger values,
 * dequantised in registers) U the open window's tokens:
 *   out[b, g, :] = sum_{t in T} softmax_t(scale * q_g . k_t) v_t   (fp32);
 *   window_mass[u, w] = sum over the group's heads g and tokens t of window w
 *   of that softmax probability (0 for evicted windows and w >= ceil(N/64)).
 *   q  device [B, Hq, d] bf16;  K, V device bf16 [B, Hkv, cap, d];
 *   out device float [B, Hq, d];  window_mass device float [U, n_win].
 *   workspace >= kvr_tiered_attend_workspace_size bytes, 256-byte aligned.
 */
kvr_status kvr_sparse_attend_tiered(const kvr_shape *shape, const kvr_tier_state *state,
                                    const void *q, const void *K, const void *V,
                                    const int32_t *seq_len, float scale, float *out,
                                    float *window_mass, void *workspace,
                                    size_t workspace_bytes, int32_t *err_word, void *stream);

/* Bytes of device workspace kvr_tier_update needs. */
size_t kvr_tier_update_workspace_size(const kvr_shape *shape, int64_t n_win);

/*
 * kvr_tier_update -- one routing step of every unit after the attention.
 *   1. score[u, w] += llrint(window_mass[u, w] * 2^32) for every non-evicted
 *      window w < ceil(N/64) (evicted windows keep their score);
 *   2. the live (not evicted) closed windows are ranked by (score desc,
 *      window asc); the first quota[u] become bf16, the others INT2;
 *   3. while the tier bytes (bf16: 64 * 2 * 2d, INT2: kvr_ledger_bytes(d))
 *      exceed budget[u], the lowest-ranked INT2 window is evicted, for good;
 *   4. data moves: bf16 -> INT2 quantises the window's K, V rows into its
 *      ledger unless has_ledger (write-once); INT2 -> bf16 writes the bf16
 *      values of the ledger into the window's K, V rows; evictions move nothing.
 *   K, V        device bf16 [B, Hkv, cap, d] (read and written).
 *   stats       device int32 [U, 3] or NULL: {promotions, demotions, evictions}.
 *   workspace   >= kvr_tier_update_workspace_size bytes, 256-byte aligned.
 */
kvr_status kvr_tier_update(const kvr_shape *shape, const kvr_tier_state *state,
                           const float *window_mass, const int32_t *seq_len, void *K, void *V,
                           int32_t *stats, void *workspace, size_t workspace_bytes,
                           int32_t *err_word, void *stream);

/*
 * kvr_read_error -- synchronise `stream`, read the device error word into
 * *bits_out (may be NULL) and clear it. Returns KVR_ERR_DEVICE when a bit was
 * set, KVR_ERR_CUDA when the synchronisation or copy failed, else KVR_OK.
 */
kvr_status kvr_read_error(int32_t *err_word, int32_t *bits_out, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* KVR_H_ */
