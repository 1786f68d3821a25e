// kvr_select.cu -- coarse collision scoring, candidate set, exact rescoring
// and final top-k of one decode step, as ONE kernel launch (kvr_select).
//
// ParisKV, "Pipeline di Recupero Nativa su GPU in Due Stadi": the query votes,
// per sub-block, for the centroids near its own with tiered weights; a key's
// coarse score is the sum of the votes of the buckets it sits in; the best few
// percent become candidates. The candidates are rescored exactly with q.k and
// the top-k kept.
//
// One thread-block cluster of CS CTAs serves one (batch, kv head) unit; the
// CTAs exchange histograms through distributed shared memory, so the whole
// step needs no second launch and no global synchronisation:
//   P1 each CTA streams its share of the unit's code tiles into shared memory
//      with 16-byte cp.async copies (one 512-token slot per warp; per-copy
//      overhead of 256-byte bulk copies was measured to dominate) and scores 32
//      keys at a time on bit-planes: XOR with the query planes, a carry-save
//      popcount of each 8-bit sub-block, the vote table as a mux tree, a
//      ripple adder into the score planes; a histogram of the top score bits
//      is kept in registers.
//   P2 two cluster exchanges of 16-bin histograms fix the threshold score T,
//      the tie quota and every CTA's candidate count and list offset (ties by
//      lowest index).
//   P3 candidates are compacted in index order into the workspace and, when
//      their spread over the CTAs is near even, kept by the CTA that found
//      them; otherwise they move through distributed shared memory to the CTA
//      whose equal slice of the list holds them (one more cluster barrier).
//   P4 every CTA rescores its slice: it loads the K rows (prefetched into L2
//      in P3) straight into registers, 16 lanes per row and 8 rows in flight
//      per half-warp, and computes the canonical fp32 dot q_bar . k
//      (half-warp per row).
//   P5 the k'-th largest exact score (order-preserving uint32 keys) in three
//      small cluster exchanges: the score range, a 256-bin linear histogram
//      of every CTA's slice over that range (16 bits per bin), then the keys
//      of the one boundary bin, located in one of 256 sub-bins of that bin
//      and ranked there by counting (a few keys: directly); a boundary bin
//      too large to gather (massive ties) falls back to every CTA gathering
//      all C' keys. Each CTA also gets its output offset.
//   P6 winners are written ascending by index.
//   P7 (the kvr_select_attend instantiations) the attention over the step's
//      tokens in the same cluster: each CTA over its winners and a share of
//      the window, partials merged through distributed shared memory.
// Every cluster barrier is reached by every CTA on every path (control flow
// around them depends only on per-unit values).
// The selection's loops stay rolled (`#pragma unroll 1`) unless they say
// otherwise: each phase runs once per launch and the kernel's largest stall
// is instruction fetch (about 180 KB of code); rolled, the million-token
// step measured 100.3 against 109.8 us and a 128K call 47.0 against 48.3 us.
#include <cooperative_groups.h>

#include "kvr_device.cuh"
#include "kvr_launch.h"

namespace cg = cooperative_groups;

namespace kvr {

constexpr int kSelThreads = 256;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kMaxSlice = 2048;  // candidates per CTA in P4-P6
constexpr int kPlaneCap = 512;   // 32-token blocks per CTA whose score planes stay on chip

struct SelArgs {
    int Hq, Hkv, G;
    int64_t cap;
    int C, k, W;
    uint32_t leaf[4];  // bit m of leaf[j] = bit j of lut[m], m = 0..8
    const void *q;
    const void *K;
    const void *V;  // optional: prefetch the winners' V rows and the window's rows
    bool early;     // KVR_SELECT_EARLY_INPUTS
    const uint8_t *rsq;  // reranker records, or null: exact rescoring
    int sink;                   // Sink tokens [0, sink)
    const int32_t *region_end;  // Retrieval end per batch entry, or null: N - W
    const uint16_t *votes;      // magnitude-aware vote lists of the units, or null
    float lev[8];        // reranker magnitude levels
    const uint8_t *codes;
    const int32_t *seq_len;
    const int8_t *sgn;
    int32_t *out_idx;
    int32_t *out_count;
    uint32_t *planes;  // [U][8][nblk] score bit-planes
    int32_t *cand_idx;
    float *cand_score;
    int32_t *cand_count;
    float *qbar;
    uint8_t *coarse;  // [U][cap_pad] or null
    int64_t nblk, cap_pad, tiles;
    int32_t *err;
    // fused attention (instantiations with GA > 0): output [B, Hq, d] fp32
    // and the logit scale in the log2 domain; V above is the value cache
    float *att_out;
    float att_scale_log2;
};

__host__ __device__ constexpr int bit_width(int v)
{
    int b = 0;
    while (v > 0) {
        b++;
        v >>= 1;
    }
    return b;
}
// score bits for nb sub-blocks of votes below 2^vb
__host__ __device__ constexpr int acc_bits(int nb, int vb) { return bit_width(nb * ((1 << vb) - 1)); }

__device__ __forceinline__ uint32_t maj3(uint32_t a, uint32_t b, uint32_t c)
{
    return (a & b) | (c & (a | b));
}
__device__ __forceinline__ uint32_t mux(uint32_t s, uint32_t one, uint32_t zero)
{
    return (s & one) | (~s & zero);
}

// Bit-sliced popcount of 8 planes (32 keys at once): c = x0 + ... + x7, 4 bits.
__device__ __forceinline__ void count8(const uint32_t (&x)[8], uint32_t &c0, uint32_t &c1,
                                       uint32_t &c2, uint32_t &c3)
{
    const uint32_t sa = x[0] ^ x[1] ^ x[2], ka = maj3(x[0], x[1], x[2]);
    const uint32_t sb = x[3] ^ x[4] ^ x[5], kb = maj3(x[3], x[4], x[5]);
    const uint32_t sc = sa ^ sb ^ x[6], kc = maj3(sa, sb, x[6]);
    c0 = sc ^ x[7];
    const uint32_t kd = sc & x[7];
    const uint32_t se = ka ^ kb ^ kc, ke = maj3(ka, kb, kc);
    c1 = se ^ kd;
    const uint32_t kf = se & kd;
    c2 = ke ^ kf;
    c3 = ke & kf;
}

// Bit-sliced table lookup v = lut[c] (c = 0..8) for one output bit; L[m] are
// all-ones / all-zero words holding that bit of lut[m].
__device__ __forceinline__ uint32_t lut_bit(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                            const uint32_t (&L)[9])
{
    const uint32_t m01 = mux(c0, L[1], L[0]), m23 = mux(c0, L[3], L[2]);
    const uint32_t m45 = mux(c0, L[5], L[4]), m67 = mux(c0, L[7], L[6]);
    const uint32_t m03 = mux(c1, m23, m01), m47 = mux(c1, m67, m45);
    return mux(c3, L[8], mux(c2, m47, m03));
}

// acc += v, bit-sliced, acc has A bits, v has V <= A bits (no overflow by design).
template <int A, int V>
__device__ __forceinline__ void add_planes(uint32_t (&acc)[A], const uint32_t (&v)[V])
{
    uint32_t carry = 0;
#pragma unroll
    for (int j = 0; j < A; j++) {
        const uint32_t x = (j < V) ? v[j] : 0u;
        const uint32_t t = acc[j] ^ x;
        const uint32_t nc = (acc[j] & x) | (carry & t);
        acc[j] = t ^ carry;
        carry = nc;
    }
}

// Masks of the keys whose A-bit score is > T and == T.
template <int A>
__device__ __forceinline__ void compare_planes(const uint32_t (&p)[A], int T, uint32_t &gt,
                                               uint32_t &eq)
{
    gt = 0u;
    eq = 0xffffffffu;
#pragma unroll
    for (int j = A - 1; j >= 0; j--) {
        if ((T >> j) & 1) {
            eq &= p[j];
        } else {
            gt |= eq & p[j];
            eq &= ~p[j];
        }
    }
}

// Keys of a 32-token block that lie in the pool [p0, pool).
__device__ __forceinline__ uint32_t pool_mask(int64_t blk, int64_t p0, int64_t pool)
{
    const int64_t lo = blk * 32;
    uint32_t m;
    if (lo + 32 <= pool) m = 0xffffffffu;
    else if (lo >= pool) m = 0u;
    else m = (1u << (uint32_t)(pool - lo)) - 1u;
    if (p0 > lo) m = (p0 >= lo + 32) ? 0u : m & (0xffffffffu << (uint32_t)(p0 - lo));
    return m;
}

template <int D, typename T> struct SelSmem {
    static constexpr int kChunks = D / 4;             // 16-byte chunks (4 planes) per block
    static constexpr int kHalfBytes = kChunks * 256;  // 16 blocks = 512 tokens
    // P1 code slots; in P5 the published boundary keys and the keys of one
    // sub-bin, or (massive ties) the order keys of up to 16384 candidates
    static constexpr int kRingBytes =
        (kSelWarps * kHalfBytes > 16384 * 4) ? kSelWarps * kHalfBytes : 16384 * 4;
    static constexpr int kRowBytes = D * (int)sizeof(T);
    static constexpr int kRowsPerBuf = kRingBytes / 2 / kRowBytes;
    static constexpr int oS = kRingBytes;
    static constexpr int oI = oS + kMaxSlice * 4;
    static constexpr int oQm = oI + kMaxSlice * 4;
    static constexpr int oQbar = oQm + kChunks * 16;
    static constexpr int oQsgn = oQbar + D * 4;
    static constexpr int oH1 = oQsgn + D * 4;
    static constexpr int oH2 = oH1 + 16 * 4;
    static constexpr int oRad = oH2 + 16 * 4;    // [2][256]
    static constexpr int oAll = oRad + 512 * 4;  // [16][16] level 1, [16][16] level 2
    static constexpr int oScan = oAll + 512 * 4;
    static constexpr int oMisc = oScan + 72 * 4;
    static constexpr int oWH = oMisc + 64 * 4;  // [kSelWarps][256] per-warp histograms
    static constexpr int oPl = oWH + kSelWarps * 256 * 4;  // [8][kPlaneCap] score planes
    static constexpr int oLev = oPl + 8 * kPlaneCap * 4;  // float [16] signed reranker levels
    static constexpr int oAtt = oLev + 16 * 4;  // fused attention: m[4], l[4], o[4][D] of the CTA
    static constexpr int bytes = oAtt + (8 + 4 * D) * 4;
    // fused attention: K and V rows of a chunk of tokens are staged over the
    // code ring and the candidate arrays (free once the winners are known)
    static constexpr int kStage = oQm;
    static_assert(16 * 256 * 4 <= kRingBytes, "radix exchange scratch must fit the ring");
    static_assert(oWH % 16 == 0, "boundary keys are read 16 bytes at a time");
    static_assert((D / 8) * kVoteStride * 2 <= 2 * kMaxSlice * 4, "vote lists must fit sS + sI");
};

enum {
    M_U1 = 0, M_REM1, M_T, M_TAKE, M_OFF, M_KTAKE, M_KOFF, M_NSUB, M_KEYT, M_QUOTA,
    M_CNT, M_ABOVEB, M_LOCAL, M_NW,
    M_BOUND = 16,  // [17] first candidate position of each CTA's P4 slice, then C'
    M_KMIN = 33, M_KMAX, M_AOWN,
    M_SEG = 40,    // [17] first boundary-key position of each CTA, then the total
};

// ---------------------------------------------------------------- P7
// Fused attention of one unit's step, run by each CTA of the selection's
// cluster after P6 (ParisKV, "Problematica": decode attends to the top-k
// subset; "Meccanismo di Aggiornamento a Finestra Scorrevole": the Local
// region is always attended). CTA `rank` takes its own winners (sWin, nw of
// them), every CS-th token of the Local (+ buffer) region [pool, N) and every
// CS-th Sink token [0, p0). The K and V rows of up to CH tokens at a time are
// staged in shared memory with 16-byte cp.async copies (over the code ring
// and the candidate arrays, dead by now). bf16 caches: warp w takes the
// 16-token tiles w, w + 8, ...; scores = K q^T and O^T += V^T P^T on the
// tensor cores (mma.sync m16n8k16, fp32 accumulate; the staged rows
// XOR-swizzled by 16-byte chunk so ldmatrix is conflict-free; P split into
// bf16 hi + lo), online softmax per warp in the log2 domain. fp32 caches: a
// token's row is spread over a warp (d/32 dims per lane) and the dots run on
// the CUDA cores. Heads past the group size G score against a zero query and
// are never written. Warps merge in shared memory, CTAs through distributed
// shared memory; each CTA writes an equal share of the unit's G*d outputs.
// Contains cluster barriers: every CTA calls it, after arriving at the split
// barrier that this function's first wait completes.
template <int D, typename T, int GA>
__device__ __forceinline__ void attend_tail(const SelArgs &a, uint8_t *smem, const int32_t *sWin,
                                            int nw, int b, int h, int64_t N, int64_t p0,
                                            int64_t pool, int rank, int CS)
{
    using SM = SelSmem<D, T>;
    constexpr bool TC = sizeof(T) == 2;        // tensor-core path (bf16)
    constexpr int E = D / 32, RB = SM::kRowBytes, PPR = RB / 16, LPH = 32 / GA;
    constexpr int CH = SM::kStage / (2 * RB);  // tokens staged at once
    constexpr int TPW = 4;                     // CUDA-core path: tokens per warp per round
    static_assert(CH >= kSelWarps * TPW && CH % 16 == 0, "a round fits the stage");
    static_assert(kSelWarps * GA * (D + 3) * 4 <= SM::kStage, "warp partials fit the stage");
    static_assert(kMaxSlice * 4 + kSelWarps * 512 <= 8 * kPlaneCap * 4, "P tiles fit the plane area");
    cg::cluster_group cluster = cg::this_cluster();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int gq = lane >> 2, cq = lane & 3;  // fragment row group, column pair
    const int lm = lane >> 3, lr = lane & 7;  // ldmatrix: matrix, row
    const int G = a.G;
    const int u = blockIdx.y;
    float *sPm = reinterpret_cast<float *>(smem + SM::oAtt);
    float *sPl = sPm + 4;
    float *sPo = sPm + 8;

    const int64_t nloc = N - pool;
    const int nlm = nloc > rank ? (int)((nloc - rank + CS - 1) / CS) : 0;
    const int nsm = p0 > rank ? (int)((p0 - rank + CS - 1) / CS) : 0;
    const int total = nw + nlm + nsm;
    auto token = [&](int i) -> int64_t {
        if (i < nw) return sWin[i];
        if (i < nw + nlm) return pool + rank + (int64_t)CS * (i - nw);
        return rank + (int64_t)CS * (i - nw - nlm);
    };
    const T *qg = static_cast<const T *>(a.q) + ((int64_t)b * a.Hq + (int64_t)h * G) * D;

    // CUDA-core state: the group's heads (log2 domain) per lane, softmax
    // state of head lane / LPH
    float qr[GA][E];
    float acc[GA][E];
    float m = -INFINITY, l = 0.0f;
    // tensor-core state: q as B fragments (column n = head gq; zero past G),
    // O^T tiles (16 dims x 8 heads), softmax state of heads 2cq, 2cq + 1
    constexpr int KS = TC ? D / 16 : 1, MD = TC ? D / 16 : 1;
    uint32_t qf[KS][2];
    float oacc[MD][4];
    float m2[2] = {-INFINITY, -INFINITY}, l2[2] = {0.0f, 0.0f};
    if constexpr (TC) {
#pragma unroll
        for (int ks = 0; ks < KS; ks++) {
            qf[ks][0] = qf[ks][1] = 0u;
            if (gq < G) {
                const uint32_t *row = reinterpret_cast<const uint32_t *>(qg + (size_t)gq * D);
                qf[ks][0] = row[(16 * ks + 2 * cq) / 2];
                qf[ks][1] = row[(16 * ks + 8 + 2 * cq) / 2];
            }
        }
#pragma unroll
        for (int md = 0; md < MD; md++)
#pragma unroll
            for (int i = 0; i < 4; i++) oacc[md][i] = 0.0f;
    } else {
#pragma unroll
        for (int g = 0; g < GA; g++)
#pragma unroll
            for (int e = 0; e < E; e++) {
                qr[g][e] = (g < G) ? to_f32(qg[g * D + lane * E + e]) * a.att_scale_log2 : 0.0f;
                acc[g][e] = 0.0f;
            }
    }

    const uint8_t *Ku = static_cast<const uint8_t *>(a.K) + (size_t)u * a.cap * RB;
    const uint8_t *Vu = static_cast<const uint8_t *>(a.V) + (size_t)u * a.cap * RB;
    uint8_t *stK = smem, *stV = smem + CH * RB;
    // this warp's P tile: [16 tokens][8 heads] bf16, hi then lo (after the winner list)
    uint8_t *sPt = smem + SM::oPl + kMaxSlice * 4 + warp * 512;
    __syncwarp();
    cluster_wait_acquire();  // no CTA reads this one's ring or scores any more (arrived after P5)
    for (int c0 = 0; c0 < total; c0 += CH) {
        const int ch = min(CH, total - c0);
        for (int pc = tid; pc < ch * PPR; pc += kSelThreads) {
            const int j = pc / PPR, part = pc % PPR;
            const size_t t = (size_t)token(c0 + j);
            // bf16: chunk `part` of row j at chunk position part ^ (j % 8)
            const int dpart = TC ? (part ^ (j & 7)) : part;
            cp_async16(stK + j * RB + dpart * 16, Ku + t * RB + part * 16);
            cp_async16(stV + j * RB + dpart * 16, Vu + t * RB + part * 16);
        }
        cp_async_commit();
        if constexpr (TC) {
            // V rows of the last tile past the chunk: zero (P is 0 there, 0 * NaN is not)
            const int pad = ((ch + 15) & ~15) - ch;
            for (int i = tid; i < pad * PPR; i += kSelThreads)
                *reinterpret_cast<uint4 *>(stV + (ch + i / PPR) * RB + (i % PPR) * 16) =
                    make_uint4(0u, 0u, 0u, 0u);
        }
        cp_async_wait<0>();
        __syncthreads();
        if constexpr (TC) {
            for (int mt = warp; 16 * mt < ch; mt += kSelWarps) {
                // scores of tokens 16 mt + gq, + 8 against heads 2cq, 2cq + 1
                float c4[4] = {0.0f, 0.0f, 0.0f, 0.0f}, c4b[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                const uint8_t *rowp = stK + (16 * mt + lr + ((lm & 1) ? 8 : 0)) * RB;
#pragma unroll
                for (int ks = 0; ks < KS; ks++) {
                    const int chk = 2 * ks + ((lm & 2) ? 1 : 0);
                    uint32_t af[4];
                    ldsm_x4(af, rowp + ((chk ^ lr) << 4));
                    mma16816((ks & 1) ? c4b : c4, af, qf[ks][0], qf[ks][1]);
                }
                const int t0 = 16 * mt + gq;
                float sc[4];
#pragma unroll
                for (int i = 0; i < 4; i++) {
                    const bool ok = ((i < 2) ? t0 : t0 + 8) < ch;
                    sc[i] = ok ? (c4[i] + c4b[i]) * a.att_scale_log2 : -INFINITY;
                }
                float ma = fmaxf(sc[0], sc[2]), mb = fmaxf(sc[1], sc[3]);
                __syncwarp();
#pragma unroll
                for (int o = 4; o < 32; o <<= 1) {
                    ma = fmaxf(ma, __shfl_xor_sync(kFull, ma, o));
                    mb = fmaxf(mb, __shfl_xor_sync(kFull, mb, o));
                }
                const float na = fmaxf(m2[0], ma), nb = fmaxf(m2[1], mb);
                const float ala = (m2[0] == -INFINITY) ? 0.0f : exp2f(m2[0] - na);
                const float alb = (m2[1] == -INFINITY) ? 0.0f : exp2f(m2[1] - nb);
                float p[4];
                p[0] = (sc[0] == -INFINITY) ? 0.0f : exp2f(sc[0] - na);
                p[1] = (sc[1] == -INFINITY) ? 0.0f : exp2f(sc[1] - nb);
                p[2] = (sc[2] == -INFINITY) ? 0.0f : exp2f(sc[2] - na);
                p[3] = (sc[3] == -INFINITY) ? 0.0f : exp2f(sc[3] - nb);
                float la = p[0] + p[2], lb = p[1] + p[3];
#pragma unroll
                for (int o = 4; o < 32; o <<= 1) {
                    la += __shfl_xor_sync(kFull, la, o);
                    lb += __shfl_xor_sync(kFull, lb, o);
                }
                l2[0] = l2[0] * ala + la;
                l2[1] = l2[1] * alb + lb;
                m2[0] = na;
                m2[1] = nb;
#pragma unroll
                for (int md = 0; md < MD; md++) {
                    oacc[md][0] *= ala;
                    oacc[md][1] *= alb;
                    oacc[md][2] *= ala;
                    oacc[md][3] *= alb;
                }
                // P (hi, lo) as [token][head] rows: the B operand of O^T += V^T P^T
                uint32_t hi, lo;
                float r0, r1;
                split_bf16x2(p[0], p[1], hi, lo, r0, r1);
                *reinterpret_cast<uint32_t *>(sPt + gq * 16 + 4 * cq) = hi;
                *reinterpret_cast<uint32_t *>(sPt + 256 + gq * 16 + 4 * cq) = lo;
                split_bf16x2(p[2], p[3], hi, lo, r0, r1);
                *reinterpret_cast<uint32_t *>(sPt + (gq + 8) * 16 + 4 * cq) = hi;
                *reinterpret_cast<uint32_t *>(sPt + 256 + (gq + 8) * 16 + 4 * cq) = lo;
                __syncwarp();
                uint32_t bq[4];
                ldsm_x4_t(bq, sPt + ((lm & 2) ? 256 : 0) + ((lm & 1) * 8 + lr) * 16);
                // A = V^T tile (16 dims x 16 tokens) from the token rows
                const uint8_t *vrow = stV + (16 * mt + lr + ((lm & 2) ? 8 : 0)) * RB;
#pragma unroll
                for (int md = 0; md < MD; md++) {
                    const int chk = 2 * md + (lm & 1);
                    uint32_t af[4];
                    ldsm_x4_t(af, vrow + ((chk ^ lr) << 4));
                    mma16816(oacc[md], af, bq[0], bq[1]);
                    mma16816(oacc[md], af, bq[2], bq[3]);
                }
                __syncwarp();  // the P tile is rewritten by the warp's next tile
            }
        } else {
            for (int jb = 0; jb < ch; jb += kSelWarps * TPW) {
                // branch-free over the warp's slots (the shuffle chains interleave);
                // a slot past the chunk scores -inf and adds nothing
                float s[TPW];
#pragma unroll
                for (int jj = 0; jj < TPW; jj++) {
                    const int j = jb + jj * kSelWarps + warp;
                    const bool live = j < ch;
                    float kv[E];
                    load_lane<E, T>(stK + (live ? j : 0) * RB, lane, kv);
                    float part[GA];
#pragma unroll
                    for (int g = 0; g < GA; g++) {
                        float d = 0.0f;
#pragma unroll
                        for (int e = 0; e < E; e++) d = fmaf(qr[g][e], kv[e], d);
                        part[g] = d;
                    }
                    const float sc = reduce_heads<GA>(part, lane);
                    s[jj] = live ? sc : -INFINITY;
                }
                float mb = -INFINITY;
#pragma unroll
                for (int jj = 0; jj < TPW; jj++) mb = fmaxf(mb, s[jj]);
                const float m_new = fmaxf(m, mb);
                const float alpha = (m == -INFINITY) ? 0.0f : exp2f(m - m_new);
                float p[TPW], ps = 0.0f;
#pragma unroll
                for (int jj = 0; jj < TPW; jj++) {
                    p[jj] = (s[jj] == -INFINITY) ? 0.0f : exp2f(s[jj] - m_new);
                    ps += p[jj];
                }
                l = l * alpha + ps;
                m = m_new;
#pragma unroll
                for (int g = 0; g < GA; g++) {
                    const float ag = __shfl_sync(kFull, alpha, g * LPH);
#pragma unroll
                    for (int e = 0; e < E; e++) acc[g][e] *= ag;
                }
#pragma unroll
                for (int jj = 0; jj < TPW; jj++) {
                    const int j = jb + jj * kSelWarps + warp;
                    const bool live = j < ch;
                    float vv[E];
                    load_lane<E, T>(stV + (live ? j : 0) * RB, lane, vv);
#pragma unroll
                    for (int e = 0; e < E; e++) vv[e] = live ? vv[e] : 0.0f;
#pragma unroll
                    for (int g = 0; g < GA; g++) {
                        const float pg = __shfl_sync(kFull, p[jj], g * LPH);
#pragma unroll
                        for (int e = 0; e < E; e++) acc[g][e] = fmaf(pg, vv[e], acc[g][e]);
                    }
                }
            }
        }
        __syncthreads();  // the stage is refilled (or reused for the warp partials)
    }

    // merge the warps (their partials over the stage)
    float *sWm = reinterpret_cast<float *>(smem);  // [warps][GA]
    float *sWl = sWm + kSelWarps * GA;             // [warps][GA]
    float *sWo = sWl + kSelWarps * GA;             // [warps][GA][D]
    if constexpr (TC) {
#pragma unroll
        for (int e = 0; e < 2; e++) {
            const int hh = 2 * cq + e;
            if (hh < GA) {
                if (gq == 0) {
                    sWm[warp * GA + hh] = m2[e];
                    sWl[warp * GA + hh] = l2[e];
                }
#pragma unroll
                for (int md = 0; md < MD; md++) {
                    sWo[(warp * GA + hh) * D + 16 * md + gq] = oacc[md][e];
                    sWo[(warp * GA + hh) * D + 16 * md + gq + 8] = oacc[md][2 + e];
                }
            }
        }
    } else {
        if ((lane % LPH) == 0) {
            sWm[warp * GA + lane / LPH] = m;
            sWl[warp * GA + lane / LPH] = l;
        }
#pragma unroll
        for (int g = 0; g < GA; g++)
#pragma unroll
            for (int e = 0; e < E; e++) sWo[(warp * GA + g) * D + lane * E + e] = acc[g][e];
    }
    __syncthreads();
    // every warp's weight per head, 2^(m_w - M) against the heads' maximum
    // (0 for a warp without tokens: its partial is zero), once per (warp,
    // head); then every output an fma chain over the warps in order
    float *sWf = sWo + kSelWarps * GA * D;  // [warps][GA]
    if (tid < kSelWarps * GA) {
        const int g = tid % GA;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kSelWarps; w++) M = fmaxf(M, sWm[w * GA + g]);
        const float mw = sWm[tid];
        sWf[tid] = (mw == -INFINITY) ? 0.0f : exp2f(mw - M);
        if (tid < GA) sPm[g] = M;
    }
    __syncthreads();
    for (int t = tid; t < G * D; t += kSelThreads) {
        const int g = t / D, dim = t % D;
        float O = 0.0f;
#pragma unroll
        for (int w = 0; w < kSelWarps; w++) O = fmaf(sWo[(w * GA + g) * D + dim], sWf[w * GA + g], O);
        sPo[t] = O;
        if (dim == 0) {
            float L = 0.0f;
#pragma unroll
            for (int w = 0; w < kSelWarps; w++) L = fmaf(sWl[w * GA + g], sWf[w * GA + g], L);
            sPl[g] = L;
        }
    }
    __syncthreads();
    cluster.sync();  // CTA partials published

    // every CTA finishes an equal share of the unit's G*D outputs; the
    // remote loads of an output are all issued before its arithmetic
    const int e0 = rank * (G * D) / CS, e1 = (rank + 1) * (G * D) / CS;
    for (int t = e0 + tid; t < e1; t += kSelThreads) {
        const int g = t / D, dim = t % D;
        float mr[16], lr2[16], orr[16];
#pragma unroll
        for (int r = 0; r < 16; r++) {
            mr[r] = (r < CS) ? *cluster.map_shared_rank(&sPm[g], r) : -INFINITY;
            lr2[r] = (r < CS) ? *cluster.map_shared_rank(&sPl[g], r) : 0.0f;
            orr[r] = (r < CS) ? *cluster.map_shared_rank(&sPo[t], r) : 0.0f;
        }
        float M = -INFINITY;
#pragma unroll
        for (int r = 0; r < 16; r++) M = fmaxf(M, mr[r]);
        float L = 0.0f, O = 0.0f;
        if (M != -INFINITY) {
#pragma unroll
            for (int r = 0; r < 16; r++) {
                if (mr[r] == -INFINITY) continue;
                const float f = exp2f(mr[r] - M);
                L = fmaf(lr2[r], f, L);
                O = fmaf(orr[r], f, O);
            }
        }
        a.att_out[((size_t)b * a.Hq + (size_t)h * G + g) * D + dim] = (L > 0.0f) ? O / L : 0.0f;
    }
}

// EXT: the instantiation carries the optional modes (reranker records,
// magnitude-aware votes); without it their code is compiled out, which keeps
// the common kernel smaller (instruction fetch is its top stall).
// GA > 0: the attention over the step's tokens runs in the same cluster
// after the selection (P7), for query groups of up to GA heads.
template <int D, typename T, int VB, bool EXT, int GA>
__global__ void __launch_bounds__(kSelThreads, 2) select_kernel(SelArgs a)
{
    using SM = SelSmem<D, T>;
    constexpr int NB = D / 8;
    constexpr int NCH = SM::kChunks;
    constexpr int ACC = acc_bits(NB, VB);
    constexpr int LOWB = ACC < 4 ? ACC : 4;
    constexpr int H1 = ACC - LOWB;
    constexpr int NL1 = 1 << H1, NL2 = 1 << LOWB;
    constexpr int RB = SM::kRowBytes;
    constexpr int P = D / 16;  // dims per lane in the exact dot

    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t *ring = smem;
    float *sS = reinterpret_cast<float *>(smem + SM::oS);
    int32_t *sI = reinterpret_cast<int32_t *>(smem + SM::oI);
    uint4 *sQm = reinterpret_cast<uint4 *>(smem + SM::oQm);
    float *sQbar = reinterpret_cast<float *>(smem + SM::oQbar);
    int *sQsgn = reinterpret_cast<int *>(smem + SM::oQsgn);
    int *sH1 = reinterpret_cast<int *>(smem + SM::oH1);
    int *sH2 = reinterpret_cast<int *>(smem + SM::oH2);
    int *sRad = reinterpret_cast<int *>(smem + SM::oRad);
    int *sAll = reinterpret_cast<int *>(smem + SM::oAll);
    int *sScan = reinterpret_cast<int *>(smem + SM::oScan);
    int *sMisc = reinterpret_cast<int *>(smem + SM::oMisc);

    cg::cluster_group cluster = cg::this_cluster();
    // Warm the L2 lines (and address translations) of the query group's rows
    // before anything waits: the loads themselves come after the dependency
    // wait, and a prefetch into L2 cannot return data older than L2 holds.
    {
        const int ub = blockIdx.y / a.Hkv, uh = blockIdx.y % a.Hkv;
        const uint8_t *qrows = static_cast<const uint8_t *>(a.q) +
                               ((int64_t)ub * a.Hq + (int64_t)uh * a.G) * D * (int64_t)sizeof(T);
        const int qbytes = a.G * D * (int)sizeof(T);
#pragma unroll 1
        for (int o = threadIdx.x * 128; o < qbytes; o += kSelThreads * 128) prefetch_l2_line(qrows + o);
    }
    // programmatic dependent launch: this grid may start while the previous one
    // drains; nothing is read before the previous grid's writes are visible
    // with KVR_SELECT_EARLY_INPUTS only q is waited for: the length, the code
    // copies and the row prefetches below start while the previous grid runs
    if (!a.early) grid_dependency_wait();
    grid_launch_dependents();
    const int CS = (int)cluster.num_blocks();
    const int rank = (int)cluster.block_rank();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int u = blockIdx.y;
    const int b = u / a.Hkv, h = u % a.Hkv;

    int64_t N = a.seq_len[b];
    if (N < 0 || N > a.cap) {
        if (rank == 0 && tid == 0 && h == 0) set_err(a.err, KVR_DEVERR_SEQ_LEN);
        N = 0;
    }
    // pool = the Retrieval region [p0, pool): after the Sink, before Local
    const int64_t p0 = min((int64_t)max(a.sink, 0), N);
    int64_t pend = a.region_end ? (int64_t)a.region_end[b] : N - a.W;
    pend = pend < p0 ? p0 : (pend > N ? N : pend);
    const int64_t pool = pend;
    const int Cp = (int)min((int64_t)a.C, pool - p0);
    const int kp = min(a.k, Cp);
    const int64_t nhalf = (pool + 511) / 512;
    const int64_t h0 = (int64_t)rank * nhalf / CS, h1 = (int64_t)(rank + 1) * nhalf / CS;
    const int64_t nb_pool = (pool + 31) / 32;
    const int64_t blk0 = min(h0 * 16, nb_pool), blk1 = min(h1 * 16, nb_pool);
    const uint8_t *codes_u = a.codes + (size_t)u * a.tiles * (D * 128);
    if (a.V) {
        // the local window's K and V rows, read by the attention that follows
        const uint8_t *Kb = static_cast<const uint8_t *>(a.K) + (size_t)u * a.cap * RB;
        const uint8_t *Vb = static_cast<const uint8_t *>(a.V) + (size_t)u * a.cap * RB;
#pragma unroll 1
        for (int64_t t = pool + rank + (int64_t)CS * tid; t < N; t += (int64_t)CS * kSelThreads) {
            prefetch_l2(Kb + (size_t)t * RB, RB);
            prefetch_l2(Vb + (size_t)t * RB, RB);
        }
#pragma unroll 1
        for (int64_t t = rank + (int64_t)CS * tid; t < p0; t += (int64_t)CS * kSelThreads) {  // the Sink
            prefetch_l2(Kb + (size_t)t * RB, RB);
            prefetch_l2(Vb + (size_t)t * RB, RB);
        }
    }

#pragma unroll 1
    for (int i = tid; i < 16; i += kSelThreads) {
        sH1[i] = 0;
        sH2[i] = 0;
    }
    // P4 slices: CTA r rescores candidate positions [bound[r], bound[r+1])
    if (tid <= CS) sMisc[M_BOUND + tid] = (int)((int64_t)tid * Cp / CS);
    __syncthreads();
    // the CTA whose P4 slice holds candidate position pos (bounds are monotone)
    auto slice_owner = [&](int pos) {
        int r = 0;
#pragma unroll
        for (int s = 8; s >= 1; s >>= 1)
            if (r + s < CS && sMisc[M_BOUND + r + s] <= pos) r += s;
        return r;
    };

    // Issue the first code half-tile of every warp before anything else: the
    // warp's 32 lanes copy its NCH chunks of 256 bytes (16 blocks x 16 B) as
    // 16-byte pieces, consecutive lanes on consecutive pieces.
    int64_t hh = (Cp > 0 || a.coarse != nullptr) ? h0 + warp : h1;
    uint8_t *slot = ring + warp * SM::kHalfBytes;
    auto issue_half = [&](int64_t half) {
        const uint8_t *tile = codes_u + (size_t)(half >> 1) * (D * 128) + (size_t)(half & 1) * 256;
#pragma unroll
        for (int i = 0; i < NCH / 2; i++) {
            const int piece = i * 32 + lane;  // chunk piece / 16, 16-byte part piece % 16
            const int c = piece >> 4, part = piece & 15;
            cp_async16(slot + c * 256 + part * 16, tile + (size_t)c * 512 + part * 16);
        }
        cp_async_commit();
    };
    if (hh < h1) issue_half(hh);
    if (a.early) grid_dependency_wait();  // q may come from the previous grid
    if (EXT && a.votes) {
        // this unit's vote lists (written by the previous grid) into the
        // candidate-score area, which P1 and P2 do not use
        const uint4 *src = reinterpret_cast<const uint4 *>(a.votes + (size_t)u * NB * kVoteStride);
        uint4 *dst = reinterpret_cast<uint4 *>(smem + SM::oS);
#pragma unroll 1
        for (int i = tid; i < NB * kVoteStride * 2 / 16; i += kSelThreads) dst[i] = src[i];
    }

    // q_bar and its code (every CTA of the cluster computes them)
    if (warp == 0) {
        // reconverge the warp (the branches above split it): its shuffles
        // below would otherwise run once per branch
        __syncwarp();
        constexpr int E = D / 32;
        const T *qg = static_cast<const T *>(a.q) + ((int64_t)b * a.Hq + (int64_t)h * a.G) * D + lane * E;
        // every load is issued before the first use (up to 4 heads' rows at
        // a time), then the heads are summed left to right
        int sg[E];
#pragma unroll
        for (int r = 0; r < E; r++) sg[r] = a.sgn[lane * E + r];
        float acc[E];
#pragma unroll 1
        for (int g0 = 0; g0 < a.G; g0 += 4) {
            float v[4][E];
#pragma unroll
            for (int i = 0; i < 4; i++)
#pragma unroll
                for (int r = 0; r < E; r++)
                    v[i][r] = (g0 + i < a.G) ? to_f32(__ldg(qg + (int64_t)(g0 + i) * D + r)) : 0.0f;
#pragma unroll
            for (int i = 0; i < 4; i++)
#pragma unroll
                for (int r = 0; r < E; r++)
                    if (g0 + i < a.G) acc[r] = (g0 + i == 0) ? v[i][r] : acc[r] + v[i][r];
        }
        float x[E];
#pragma unroll
        for (int r = 0; r < E; r++) {
            const int j = lane * E + r;
            x[r] = acc[r] / (float)a.G;
            sQbar[j] = x[r];
            if (rank == 0) a.qbar[(int64_t)u * D + j] = x[r];
            if (sg[r] < 0) x[r] = -x[r];
        }
        fwht_lanes<E, 32>(x, lane);
#pragma unroll
        for (int r = 0; r < E; r++) sQsgn[lane * E + r] = x[r] < 0.0f ? -1 : 0;
        // the reranker scores against zq = FWHT(D q_bar) itself, q_bar is not needed
        if (EXT && a.rsq)
#pragma unroll
            for (int r = 0; r < E; r++) sQbar[lane * E + r] = x[r];
    }
    // nibble code -> signed level: magnitude in bits 0..2, sign in bit 3
    if (tid < 16) reinterpret_cast<float *>(smem + SM::oLev)[tid] = (tid & 8) ? -a.lev[tid & 7] : a.lev[tid & 7];
    __syncthreads();
#pragma unroll 1
    for (int c = tid; c < NCH; c += kSelThreads)
        sQm[c] = make_uint4((uint32_t)sQsgn[4 * c], (uint32_t)sQsgn[4 * c + 1],
                            (uint32_t)sQsgn[4 * c + 2], (uint32_t)sQsgn[4 * c + 3]);
    uint32_t L[VB][9];  // vote-table leaves
#pragma unroll
    for (int j = 0; j < VB; j++)
#pragma unroll
        for (int m = 0; m < 9; m++) L[j][m] = ((a.leaf[j] >> m) & 1u) ? 0xffffffffu : 0u;
    __syncthreads();
    // The half-tiles copied in later rounds: start them into L2 now (up to 32
    // ahead), so each later copy waits on L2 rather than on DRAM. Whole tiles,
    // one 128-byte line per prefetch. Issued after the query load, which
    // they would otherwise queue ahead of.
    if (Cp > 0 || a.coarse != nullptr) {
        const int64_t pf0 = h0 + kSelWarps, pf1 = min(h1, h0 + kSelWarps + 32);
        if (pf0 < pf1) {
            const uint8_t *pbase = codes_u + (size_t)(pf0 >> 1) * (D * 128);
            const int64_t pbytes = (((pf1 + 1) >> 1) - (pf0 >> 1)) * (int64_t)(D * 128);
#pragma unroll 1
            for (int64_t o = (int64_t)tid * 128; o < pbytes; o += (int64_t)kSelThreads * 128)
                prefetch_l2_line(pbase + o);
        }
    }

    // ---------------------------------------------------------------- P1
    int cnt1[NL1];
#pragma unroll
    for (int i = 0; i < NL1; i++) cnt1[i] = 0;
    const int jb = lane & 15, sh = lane >> 4;  // block within the half-tile, sub-block half
    uint32_t *planes_u = a.planes + (size_t)u * 8 * a.nblk;
    // score plane j of block blk: on chip for this CTA's first kPlaneCap blocks
    uint32_t *sPl = reinterpret_cast<uint32_t *>(smem + SM::oPl);
    auto plane = [&](int j, int64_t blk) -> uint32_t & {
        const int64_t lb = blk - blk0;
        return (lb < kPlaneCap) ? sPl[j * kPlaneCap + lb] : planes_u[(size_t)j * a.nblk + blk];
    };
#pragma unroll 1
    for (; hh < h1; hh += kSelWarps) {
        cp_async_wait<0>();
        __syncwarp();  // every lane's pieces of the half-tile have landed
        uint32_t acc[ACC];
#pragma unroll
        for (int j = 0; j < ACC; j++) acc[j] = 0u;
#pragma unroll 2
        for (int sb = sh * (NB / 2); sb < (sh + 1) * (NB / 2); sb++) {
            const uint4 v0 = *reinterpret_cast<const uint4 *>(slot + (2 * sb) * 256 + jb * 16);
            const uint4 v1 = *reinterpret_cast<const uint4 *>(slot + (2 * sb + 1) * 256 + jb * 16);
            const uint4 q0 = sQm[2 * sb], q1 = sQm[2 * sb + 1];
            const uint32_t x[8] = {v0.x ^ q0.x, v0.y ^ q0.y, v0.z ^ q0.z, v0.w ^ q0.w,
                                   v1.x ^ q1.x, v1.y ^ q1.y, v1.z ^ q1.z, v1.w ^ q1.w};
            uint32_t vote[VB];
            if (EXT && a.votes) {
                // match the 32 keys' flip patterns against the voted patterns
                const uint16_t *lst = reinterpret_cast<const uint16_t *>(smem + SM::oS) + sb * kVoteStride;
                const int np = lst[256];
#pragma unroll
                for (int j = 0; j < VB; j++) vote[j] = 0u;
#pragma unroll 2
                for (int i = 0; i < np; i++) {
                    const uint32_t e = lst[i];
                    uint32_t miss = 0u;
#pragma unroll
                    for (int j = 0; j < 8; j++) miss |= x[j] ^ (0u - ((e >> j) & 1u));
#pragma unroll
                    for (int j = 0; j < VB; j++) vote[j] |= ((e >> (8 + j)) & 1u) ? ~miss : 0u;
                }
            } else {
                uint32_t c0, c1, c2, c3;
                count8(x, c0, c1, c2, c3);
#pragma unroll
                for (int j = 0; j < VB; j++) vote[j] = lut_bit(c0, c1, c2, c3, L[j]);
            }
            add_planes<ACC, VB>(acc, vote);
        }
        uint32_t other[ACC];  // the other half of the sub-blocks sits in lane ^ 16
        __syncwarp();
#pragma unroll
        for (int j = 0; j < ACC; j++) other[j] = __shfl_xor_sync(kFull, acc[j], 16);
        add_planes<ACC, ACC>(acc, other);
        // every lane has read the slot: refill it
        __syncwarp();
        const int64_t blk = hh * 16 + jb;
        if (hh + kSelWarps < h1) issue_half(hh + kSelWarps);
        // long ranges (past the 32 half-tiles prefetched at the start): keep
        // the half-tile 32 ahead streaming into L2, so every later copy
        // waits on L2 rather than on DRAM
        {
            const int64_t pfh = hh + 32;
            if (pfh >= h0 + kSelWarps + 32 && pfh < h1) {
                const uint8_t *pt = codes_u + (size_t)(pfh >> 1) * (D * 128) + (size_t)(pfh & 1) * 256;
#pragma unroll 1
                for (int i = lane; i < 2 * NCH; i += 32) prefetch_l2_line(pt + (i >> 1) * 512 + (i & 1) * 128);
            }
        }
        if (sh == 0 && blk < nb_pool) {
            const uint32_t vm = pool_mask(blk, p0, pool);
#pragma unroll
            for (int j = 0; j < ACC; j++) plane(j, blk) = acc[j];
#pragma unroll
            for (int v = 0; v < NL1; v++) {
                uint32_t m = vm;
#pragma unroll
                for (int j = 0; j < H1; j++) m &= ((v >> j) & 1) ? acc[LOWB + j] : ~acc[LOWB + j];
                cnt1[v] += __popc(m);
            }
        }
    }
    {
        const int s = warp_reduce_split<NL1>(cnt1);  // lane l: bucket l / (32 / NL1)
        if ((lane % (32 / NL1)) == 0 && s) atomicAdd(&sH1[lane / (32 / NL1)], s);
    }
    __syncthreads();
    cluster.sync();  // #1: level-1 histograms published

    // ---------------------------------------------------------------- P2
    // The threshold score T (the C'-th largest), the ties at T taken, and
    // every CTA's count of candidates and its offset in the index-ordered
    // list. When the candidates spread near evenly over the CTAs, each CTA
    // rescores its own (its P4 slice is its list segment: no redistribution,
    // no cluster barrier before P4); otherwise the list is cut into equal
    // slices and the candidates move to the CTA whose slice holds them.
    // Warp 0, lane r = CTA r: gt / eq = keys above / at T; the ties go to the
    // lowest indices, so to the CTAs in rank order.
    auto finish_threshold = [&](int Tthr, int quota, int gt, int eq) {
        const int eq_before = warp_exclusive_scan(eq);
        const int tk = (lane < CS) ? max(0, min(quota - eq_before, eq)) : 0;
        const int cnt = gt + tk;
        const int sel_before = warp_exclusive_scan(cnt);
        // local only when the spread is near even: ties go to the lowest
        // indices, so the first CTAs can hold many more than C'/CS, and the
        // slowest rescoring CTA sets every later barrier
        const int nmax = __reduce_max_sync(kFull, (unsigned)cnt);
        const int even = (Cp + CS - 1) / CS;
        const bool local = nmax <= kMaxSlice && nmax <= even + even / 16 + 16;
        if (local && lane <= CS) sMisc[M_BOUND + lane] = sel_before;  // lane CS: C'
        if (lane == 0) {
            sMisc[M_T] = Tthr;
            sMisc[M_LOCAL] = local ? 1 : 0;
        }
        if (lane == rank) {
            sMisc[M_TAKE] = tk;
            sMisc[M_OFF] = sel_before;
        }
    };
    {
#pragma unroll 1
        for (int t = tid; t < CS * NL1; t += kSelThreads) {
            const int r = t / NL1, v = t % NL1;
            sAll[r * 16 + v] = *cluster.map_shared_rank(&sH1[v], r);
        }
        __syncthreads();
        if (warp == 0) {
            // lane v: cluster-wide count of bucket v; the C'-th key sits in the
            // highest bucket whose suffix count reaches C'
            int tot = 0;
            if (lane < NL1)
#pragma unroll
                for (int r = 0; r < 16; r++) tot += (r < CS) ? sAll[r * 16 + lane] : 0;
            const int suf = warp_suffix_sum(tot);
            int u1 = -1, rem = Cp;
            if (Cp > 0) {
                const unsigned ok = __ballot_sync(kFull, lane < NL1 && suf >= Cp);
                u1 = __popc(ok) - 1;
                rem = Cp - __shfl_sync(kFull, suf - tot, u1);
            }
            if (lane == 0) {
                sMisc[M_U1] = u1;
                sMisc[M_REM1] = rem;
            }
        }
        __syncthreads();
        const int u1 = sMisc[M_U1];
        if (u1 >= 0) {
            int cnt2[NL2];
#pragma unroll
            for (int i = 0; i < NL2; i++) cnt2[i] = 0;
#pragma unroll 1
            for (int64_t blk = blk0 + tid; blk < blk1; blk += kSelThreads) {
                uint32_t p[ACC];
#pragma unroll
                for (int j = 0; j < ACC; j++) p[j] = plane(j, blk);
                uint32_t inb = pool_mask(blk, p0, pool);
#pragma unroll
                for (int j = 0; j < H1; j++) inb &= ((u1 >> j) & 1) ? p[LOWB + j] : ~p[LOWB + j];
#pragma unroll
                for (int v = 0; v < NL2; v++) {
                    uint32_t m = inb;
#pragma unroll
                    for (int j = 0; j < LOWB; j++) m &= ((v >> j) & 1) ? p[j] : ~p[j];
                    cnt2[v] += __popc(m);
                }
            }
            const int s = warp_reduce_split<NL2>(cnt2);  // lane l: value l / (32 / NL2)
            if ((lane % (32 / NL2)) == 0 && s) atomicAdd(&sH2[lane / (32 / NL2)], s);
        }
        __syncthreads();
        // pushed into row `rank` of every CTA's table: a remote store ahead of
        // the barrier costs no round trip after it
#pragma unroll 1
        for (int t = tid; t < CS * NL2; t += kSelThreads) {
            const int r = t / NL2, v = t % NL2;
            *cluster.map_shared_rank(&sAll[256 + rank * 16 + v], r) = sH2[v];
        }
        cluster.sync();  // #2: level-2 histograms published
        if (warp == 0) {
            int Tthr = 1 << 30, quota = 0, gt = 0, eq = 0;
            if (u1 >= 0) {
                const int rem = sMisc[M_REM1];
                int tot = 0;
                if (lane < NL2)
#pragma unroll
                    for (int r = 0; r < 16; r++) tot += (r < CS) ? sAll[256 + r * 16 + lane] : 0;
                const int suf = warp_suffix_sum(tot);
                const unsigned ok = __ballot_sync(kFull, lane < NL2 && suf >= rem);
                const int v2 = __popc(ok) - 1;
                quota = rem - __shfl_sync(kFull, suf - tot, v2);  // ties at T taken
                Tthr = (u1 << LOWB) | v2;
                if (lane < CS) {
#pragma unroll 1
                    for (int v = u1 + 1; v < NL1; v++) gt += sAll[lane * 16 + v];
#pragma unroll 1
                    for (int v = v2 + 1; v < NL2; v++) gt += sAll[256 + lane * 16 + v];
                    eq = sAll[256 + lane * 16 + v2];
                }
            }
            finish_threshold(Tthr, quota, gt, eq);
            if (lane == 0 && rank == 0) a.cand_count[u] = Cp;
        }
        __syncthreads();
    }
    const int u1 = sMisc[M_U1];
    const bool local = sMisc[M_LOCAL] != 0;

    // ---------------------------------------------------------------- P3
    const int Tthr = sMisc[M_T];
    int32_t *cidx = a.cand_idx + (size_t)u * a.C;
    {
        const int64_t nbc = blk1 - blk0;
        const int64_t bpt = (nbc + kSelThreads - 1) / kSelThreads;
        const int64_t my0 = blk0 + min((int64_t)tid * bpt, nbc);
        const int64_t my1 = blk0 + min((int64_t)(tid + 1) * bpt, nbc);
        int n_eq = 0, n_gt = 0;
        if (u1 >= 0)
#pragma unroll 1
            for (int64_t blk = my0; blk < my1; blk++) {
                uint32_t p[ACC], gt, eq;
#pragma unroll
                for (int j = 0; j < ACC; j++) p[j] = plane(j, blk);
                compare_planes<ACC>(p, Tthr, gt, eq);
                const uint32_t vm = pool_mask(blk, p0, pool);
                n_eq += __popc(eq & vm);
                n_gt += __popc(gt & vm);
            }
        // one scan of both counts: the ties taken before this thread are the
        // first `take` ties in order, min(take, eq_before) of them
        int eq_before, gt_before;
        block_exclusive_scan2(n_eq, n_gt, sScan, &eq_before, &gt_before);
        const int take = sMisc[M_TAKE];
        int allow = max(0, min(take - eq_before, n_eq));
        int pos = gt_before + min(take, eq_before) + sMisc[M_OFF];
        // owner CTA of list position pos and its slice [s_lo, s_hi), advanced
        // as pos grows (positions only increase); in the local mode this CTA
        int r2 = local ? rank : slice_owner(pos);
        int s_lo = sMisc[M_BOUND + r2], s_hi = sMisc[M_BOUND + r2 + 1];
#pragma unroll 1
        for (int64_t blk = my0; blk < my1; blk++) {
            uint32_t p[ACC], gt = 0, eq = 0;
#pragma unroll
            for (int j = 0; j < ACC; j++) p[j] = plane(j, blk);
            const uint32_t vm = pool_mask(blk, p0, pool);
            if (u1 >= 0) {
                compare_planes<ACC>(p, Tthr, gt, eq);
                gt &= vm;
                eq &= vm;
                uint32_t te = 0;
#pragma unroll 1
                for (uint32_t m = eq; m && allow > 0; m &= m - 1, allow--) te |= m & (0u - m);
#pragma unroll 1
                for (uint32_t m = gt | te; m; m &= m - 1) {
                    const int32_t id = (int32_t)(blk * 32 + __ffs(m) - 1);
                    // the row (or record) is read in P4: start it now
                    if (EXT && a.rsq) {
                        constexpr int RBQ = 6 * (D / 8);
                        const uint8_t *rp = a.rsq + ((size_t)u * a.cap + id) * RBQ;
                        prefetch_l2_line(rp);
                        prefetch_l2_line(rp + RBQ - 1);
                    } else {
                        prefetch_l2(static_cast<const uint8_t *>(a.K) + ((size_t)u * a.cap + id) * RB, RB);
                    }
                    cidx[pos] = id;
                    if (local) {
                        sI[pos - s_lo] = id;
                    } else {
                        // straight into the shared memory of the CTA whose P4
                        // slice [r*C'/CS, (r+1)*C'/CS) holds list position pos
                        while (r2 + 1 < CS && pos >= s_hi) {
                            r2++;
                            s_lo = s_hi;
                            s_hi = sMisc[M_BOUND + r2 + 1];
                        }
                        *cluster.map_shared_rank(&sI[pos - s_lo], r2) = id;
                    }
                    pos++;
                }
            }
            if (a.coarse) {
                uint8_t *co = a.coarse + (size_t)u * a.cap_pad + blk * 32;
#pragma unroll 1
                for (int i = 0; i < 32; i++) {
                    if (!((vm >> i) & 1u)) continue;
                    int s = 0;
#pragma unroll
                    for (int j = 0; j < ACC; j++) s |= (int)((p[j] >> i) & 1u) << j;
                    co[i] = (uint8_t)s;
                }
            }
        }
    }
    __syncthreads();
    if (!local) cluster.sync();  // #3: the unit's candidate list is complete

    // ---------------------------------------------------------------- P4
    // this CTA's slice of the candidate list: its own segment (local mode)
    // or an equal share (<= kMaxSlice: the host picks CS so); sI filled in P3
    const int lo = sMisc[M_BOUND + rank], hi = sMisc[M_BOUND + rank + 1];
    const int n = hi - lo;
    if (tid == 0) {  // P5 accumulators, ordered by the barrier below
        sMisc[M_KMIN] = (int)0xffffffffu;
        sMisc[M_KMAX] = 0;
        sMisc[M_AOWN] = 0;
    }
    if (EXT && a.rsq) {
        // Calibrated estimate from the records, no K rows: lane gl of a
        // half-warp is block slot gl (slots past d/8 add +0), zq of its block
        // is in sQbar; e = fma chain over the block's 8 coordinates of
        // (+-level) * zq, the signed level looked up by the coordinate's
        // nibble; t = w * e, then butterfly sums over spans 8..1.
        constexpr int NB = D / 8, RBQ = 6 * NB, NHW = kSelThreads / 16, RR = 8;
        const int hw = tid >> 4, gl = tid & 15;
        const float *sLev = reinterpret_cast<const float *>(smem + SM::oLev);
        float zqv[8];
#pragma unroll
        for (int e = 0; e < 8; e++) zqv[e] = (gl < NB) ? sQbar[gl * 8 + e] : 0.0f;
        const uint8_t *recu = a.rsq + (size_t)u * a.cap * RBQ;
        __syncthreads();  // sI complete (filled in P3)
#pragma unroll 1
        for (int base = 0; base < n; base += NHW * RR) {
            uint32_t wd[RR];
            uint32_t ws[RR];
            // branch-free (clamped index, then masked): the warp stays converged
            // for the butterflies below
#pragma unroll
            for (int r = 0; r < RR; r++) {
                const int j = base + r * NHW + hw;
                const bool live = j < n && gl < NB;
                const uint8_t *rp = recu + (size_t)sI[j < n ? j : n - 1] * RBQ;
                const int gs = gl < NB ? gl : 0;
                const uint32_t w0 = *reinterpret_cast<const uint32_t *>(rp + 4 * gs);
                const uint32_t s0 = *reinterpret_cast<const uint16_t *>(rp + 4 * NB + 2 * gs);
                wd[r] = live ? w0 : 0u;
                ws[r] = live ? s0 : 0u;
            }
#pragma unroll
            for (int r = 0; r < RR; r++) {
                float e = 0.0f;
#pragma unroll
                for (int jj = 0; jj < 8; jj++) e = __fmaf_rn(sLev[(wd[r] >> (4 * jj)) & 15u], zqv[jj], e);
                float t = (gl < NB) ? __uint_as_float(ws[r] << 16) * e : 0.0f;
#pragma unroll
                for (int span = 8; span >= 1; span >>= 1) t = t + __shfl_xor_sync(kFull, t, span);
                const int j = base + r * NHW + hw;
                if (gl == 0 && j < n) {
                    if (t != t) set_err(a.err, KVR_DEVERR_NONFINITE);
                    sS[j] = t;
                    a.cand_score[(size_t)u * a.C + lo + j] = t;
                }
            }
        }
    } else {
        float qv[P];
#pragma unroll
        for (int e = 0; e < P; e++) qv[e] = sQbar[(tid & 15) * P + e];
        // Rows go straight into registers: lane gl of a half-warp loads the
        // 16-byte-aligned dims [gl*P, gl*P+P) of its row (16 lanes = one
        // coalesced row), R rows in flight per half-warp (32 registers). The
        // rows were prefetched into L2 in P3, so fewer in flight suffice; the
        // smaller loop also costs less instruction fetch (measured faster
        // than 64 registers' worth).
        constexpr int WPR = P * (int)sizeof(T) / 4;  // 32-bit words per lane per row
        constexpr int R = 32 / WPR;
        constexpr int NHW = kSelThreads / 16;
        const uint32_t *Kw = reinterpret_cast<const uint32_t *>(static_cast<const uint8_t *>(a.K) +
                                                               (size_t)u * a.cap * RB);
        const int hw = tid >> 4, gl = tid & 15;
        __syncthreads();  // sI complete (filled in P3)
#pragma unroll 1
        for (int base = 0; base < n; base += NHW * R) {
            uint32_t raw[R][WPR];
#pragma unroll
            for (int r = 0; r < R; r++) {
                const int j = base + r * NHW + hw;
                if (j < n) {
                    const uint32_t *src = Kw + (size_t)sI[j] * (RB / 4) + gl * WPR;
#pragma unroll
                    for (int w = 0; w < WPR; w += (WPR >= 4 ? 4 : 2)) {
                        if constexpr (WPR >= 4) {
                            const uint4 v = __ldg(reinterpret_cast<const uint4 *>(src + w));
                            raw[r][w] = v.x;
                            raw[r][w + 1] = v.y;
                            raw[r][w + 2] = v.z;
                            raw[r][w + 3] = v.w;
                        } else {
                            const uint2 v = __ldg(reinterpret_cast<const uint2 *>(src + w));
                            raw[r][w] = v.x;
                            raw[r][w + 1] = v.y;
                        }
                    }
                } else {
#pragma unroll
                    for (int w = 0; w < WPR; w++) raw[r][w] = 0u;
                }
            }
#pragma unroll
            for (int r = 0; r < R; r++) {
                float kv[P];
#pragma unroll
                for (int e = 0; e < P; e++) {
                    if constexpr (sizeof(T) == 2)
                        kv[e] = (e & 1) ? bf16_hi(raw[r][e >> 1]) : bf16_lo(raw[r][e >> 1]);
                    else
                        kv[e] = __uint_as_float(raw[r][e]);
                }
                float acc = 0.0f;
#pragma unroll
                for (int e = 0; e < P; e++) acc = __fmaf_rn(qv[e], kv[e], acc);
#pragma unroll
                for (int span = 8; span >= 1; span >>= 1)
                    acc = acc + __shfl_xor_sync(kFull, acc, span);
                const int j = base + r * NHW + hw;
                if (gl == 0 && j < n) {
                    if (acc != acc) set_err(a.err, KVR_DEVERR_NONFINITE);
                    sS[j] = acc;
                    a.cand_score[(size_t)u * a.C + lo + j] = acc;
                }
            }
        }
    }
    __syncthreads();

    // ---------------------------------------------------------------- P5
    // Top-k over the cluster in three small exchanges: (1) the score range
    // (every CTA's min and max pushed into every CTA); (2) a 256-bin linear
    // histogram of every slice over that range, 16 bits per bin (the bin map
    // is monotone, so the k'-th largest key sits in one boundary bin); (3)
    // the counts above and in the boundary bin (pushed) and the bin's keys
    // (gathered), ranked by counting (past 32 of them inside one of 256
    // sub-bins of the bin; past 256 in that sub-bin, by one warp's 8-bit
    // radix passes). A boundary bin too large to gather (massive ties) falls
    // back to every CTA gathering all C' keys.
    static_assert(kSelThreads == 256, "one histogram bin per thread");
    int *sWH = reinterpret_cast<int *>(smem + SM::oWH);
    uint32_t *sPub = reinterpret_cast<uint32_t *>(ring);  // own boundary keys, published
    // 256-bin histogram of `bin(i)` over the items i < n with `take(i)`:
    // per-warp counters, then thread b sums bin b into sRad[b]
    auto histogram = [&](int nitems, auto &&take, auto &&bin) {
#pragma unroll 1
        for (int i = tid; i < kSelWarps * 256; i += kSelThreads) sWH[i] = 0;
        __syncthreads();
#pragma unroll 1
        for (int i = tid; i < nitems; i += kSelThreads)
            if (take(i)) atomicAdd(&sWH[warp * 256 + bin(i)], 1);
        __syncthreads();
        int c = 0;
#pragma unroll
        for (int w = 0; w < kSelWarps; w++) c += sWH[w * 256 + tid];
        sRad[tid] = c;
        __syncthreads();
    };
    // the bin of hist[256] holding the rem-th largest item, and how many lie
    // above it (computed by every calling warp alike, no barrier needed)
    auto find_bin_in = [&](const int *hist, int rem, int &bin, int &before) {
        int cnt[8], sum = 0;
#pragma unroll
        for (int r = 0; r < 8; r++) {
            cnt[r] = hist[255 - (lane * 8 + r)];
            sum += cnt[r];
        }
        int incl = sum;
        __syncwarp();
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(kFull, incl, o);
            incl += (lane >= o) ? y : 0;
        }
        const int run0 = incl - sum;
        const bool mine = run0 < rem && rem <= incl;
        int bn = 0, bf = 0;
        if (mine) {
            int run = run0;
#pragma unroll
            for (int r = 0; r < 8; r++) {
                if (run + cnt[r] >= rem) {
                    bn = 255 - (lane * 8 + r);
                    bf = run;
                    break;
                }
                run += cnt[r];
            }
        }
        __syncwarp();
        const int src = __ffs(__ballot_sync(kFull, mine)) - 1;
        bin = __shfl_sync(kFull, bn, src);
        before = __shfl_sync(kFull, bf, src);
    };
    // warp 0 only: the rem-th largest of keys[0..nk) by four 8-bit passes;
    // writes the key and how many copies of it are taken (ties) to sMisc
    auto radix_warp = [&](const uint32_t *keys, int nk, int rem) {
        int *wh = sRad + 256;
        uint32_t prefix = 0, mask = 0;
#pragma unroll 1
        for (int pass = 0; pass < 4; pass++) {
            const int shift = 24 - 8 * pass;
#pragma unroll 1
            for (int i = lane; i < 256; i += 32) wh[i] = 0;
            __syncwarp();
#pragma unroll 1
            for (int i = lane; i < nk; i += 32) {
                const uint32_t k = keys[i];
                if ((k & mask) == prefix) atomicAdd(&wh[(k >> shift) & 255u], 1);
            }
            __syncwarp();
            int dg, before;
            find_bin_in(wh, rem, dg, before);
            rem -= before;
            prefix |= (uint32_t)dg << shift;
            mask |= 255u << shift;
            __syncwarp();
        }
        if (lane == 0) {
            sMisc[M_KEYT] = (int)prefix;
            sMisc[M_QUOTA] = rem;
        }
    };

    // (1) the score range of this slice, then of the unit
    {
        uint32_t lmin = 0xffffffffu, lmax = 0u;
#pragma unroll 1
        for (int j = tid; j < n; j += kSelThreads) {
            const uint32_t k = order_key(sS[j]);
            lmin = min(lmin, k);
            lmax = max(lmax, k);
        }
        __syncwarp();
        lmin = __reduce_min_sync(kFull, lmin);
        lmax = __reduce_max_sync(kFull, lmax);
        if (lane == 0) {  // slots set before P4
            atomicMin(reinterpret_cast<unsigned *>(&sMisc[M_KMIN]), lmin);
            atomicMax(reinterpret_cast<unsigned *>(&sMisc[M_KMAX]), lmax);
        }
    }
    sRad[tid] = 0;
    __syncthreads();
    // pushed into slot `rank` of every CTA (the first-level histogram slots,
    // free since barrier #2): min in sH1, max in sH2
    if (tid < CS) {
        *cluster.map_shared_rank(&sH1[rank], tid) = sMisc[M_KMIN];
        *cluster.map_shared_rank(&sH2[rank], tid) = sMisc[M_KMAX];
    }
    cluster.sync();  // #4: slice ranges published
    // every warp reduces the ranges itself (empty slices: ~0 / 0)
    const uint32_t g0 = __reduce_min_sync(kFull, lane < CS ? (uint32_t)sH1[lane] : 0xffffffffu);
    const uint32_t g1 = __reduce_max_sync(kFull, lane < CS ? (uint32_t)sH2[lane] : 0u);
    const float fmin = key_float(g0);
    float scale = 256.0f / (key_float(g1) - fmin);
    if (!(scale < INFINITY) || !(scale > 0.0f)) scale = 0.0f;  // one value, or no spread
    // the position of a key in the linear bin map, in bin units; the bin is
    // its integer part (clamped), a sub-bin of it 1/256 of that unit
    // (rounded operations: never contracted, so every use maps a key alike)
    auto lin_pos = [&](uint32_t key) { return __fmul_rn(__fsub_rn(key_float(key), fmin), scale); };
    auto lin_bin = [&](uint32_t key) {
        const int x = (int)lin_pos(key);
        return min(255, max(0, x));
    };
    // (2) this slice's linear histogram, two 16-bit bins per word (a slice
    // holds at most 2048 keys): reading every slice's histogram is bound by
    // the bytes moved between the CTAs, so they move half as many
    uint32_t *sHist = reinterpret_cast<uint32_t *>(sRad);
    if (kp > 0)
#pragma unroll 1
        for (int j = tid; j < n; j += kSelThreads) {
            const int bn = lin_bin(order_key(sS[j]));
            atomicAdd(&sHist[bn >> 1], 1u << ((bn & 1) * 16));
        }
    __syncthreads();
    cluster.sync();  // #5: slice histograms published
    int b_lin = 0, rem = 0;
    if (kp > 0 && tid < 128) {
        uint32_t w[16];
#pragma unroll
        for (int r = 0; r < 16; r++) w[r] = (r < CS) ? *cluster.map_shared_rank(&sHist[tid], r) : 0u;
        int lo16 = 0, hi16 = 0;
#pragma unroll
        for (int r = 0; r < 16; r++) {
            lo16 += (int)(w[r] & 0xffffu);
            hi16 += (int)(w[r] >> 16);
        }
        sRad[256 + 2 * tid] = lo16;
        sRad[256 + 2 * tid + 1] = hi16;
    }
    if (tid == 0) sMisc[M_CNT] = 0;
    __syncthreads();
    if (kp > 0) {
        int above;
        find_bin_in(sRad + 256, kp, b_lin, above);
        rem = kp - above;  // rank of the k'-th key inside the boundary bin
    }
    // this slice's keys above the boundary bin, and its boundary keys
    int a_own = 0;
    if (kp > 0)
#pragma unroll 1
        for (int j = tid; j < n; j += kSelThreads) {
            const uint32_t k = order_key(sS[j]);
            const int bn = lin_bin(k);
            if (bn > b_lin) a_own++;
            else if (bn == b_lin) sPub[atomicAdd(&sMisc[M_CNT], 1)] = k;
        }
    {
        const int s = warp_sum(a_own);
        if (lane == 0 && s) atomicAdd(&sMisc[M_AOWN], s);  // slot cleared before P4
    }
    __syncthreads();
    // the counts pushed into slot `rank` of every CTA (the first rows of the
    // P2 table, free since P2)
    if (tid < CS) {
        *cluster.map_shared_rank(&sAll[rank], tid) = sMisc[M_AOWN];
        *cluster.map_shared_rank(&sAll[16 + rank], tid) = sMisc[M_CNT];
    }
    cluster.sync();  // #6: above counts and boundary keys published

    uint32_t keyT = 0;
    if (kp > 0) {
        // boundary segments in cluster (= index) order
        if (warp == 0) {
            int ab = 0, nb = 0;
            if (lane < CS) {
                ab = sAll[lane];
                nb = sAll[16 + lane];
            }
            const int ab_before = warp_exclusive_scan(ab);
            const int nb_before = warp_exclusive_scan(nb);
            if (lane <= CS) sMisc[M_SEG + lane] = nb_before;  // lane CS: the total
            if (lane == rank) sMisc[M_ABOVEB] = ab_before;
        }
        __syncthreads();
        const int NB = sMisc[M_SEG + CS];
        uint32_t *sB = reinterpret_cast<uint32_t *>(sWH);
        if (NB <= kSelWarps * 256) {
            auto seg_owner = [&](int t) {
                int r = 0;
#pragma unroll
                for (int s2 = 8; s2 >= 1; s2 >>= 1)
                    if (r + s2 < CS && sMisc[M_SEG + r + s2] <= t) r += s2;
                return r;
            };
#pragma unroll 1
            for (int base = 0; base < NB; base += 8 * kSelThreads) {
                uint32_t v[8];
#pragma unroll
                for (int i = 0; i < 8; i++) {
                    const int t = base + i * kSelThreads + tid;
                    v[i] = 0u;
                    if (t < NB) {
                        const int r2 = seg_owner(t);
                        v[i] = *cluster.map_shared_rank(&sPub[t - sMisc[M_SEG + r2]], r2);
                    }
                }
#pragma unroll
                for (int i = 0; i < 8; i++) {
                    const int t = base + i * kSelThreads + tid;
                    if (t < NB) sB[t] = v[i];
                }
            }
            if (tid < 3) sScan[tid] = 0;
            __syncthreads();
            // rank by counting: thread t < nk ranks keys[t] against all nk keys
            // (keys 16-byte aligned); the copy of the rk-th largest key sets it
            auto rank_count = [&](const uint32_t *keys, int nk, int rk) {
                if (tid < nk) {
                    const uint32_t k = keys[tid];
                    int gt = 0, eq = 0, j = 0;
                    // independent 16-byte broadcast loads, several in flight
#pragma unroll 4
                    for (; j + 4 <= nk; j += 4) {
                        const uint4 v = *reinterpret_cast<const uint4 *>(keys + j);
                        gt += (int)(v.x > k) + (int)(v.y > k) + (int)(v.z > k) + (int)(v.w > k);
                        eq += (int)(v.x == k) + (int)(v.y == k) + (int)(v.z == k) + (int)(v.w == k);
                    }
#pragma unroll 1
                    for (; j < nk; j++) {
                        const uint32_t kj = keys[j];
                        gt += kj > k;
                        eq += kj == k;
                    }
                    if (gt < rk && rk <= gt + eq) {  // every copy of the key agrees
                        sMisc[M_KEYT] = (int)k;
                        sMisc[M_QUOTA] = rk - gt;
                    }
                }
            };
            if (NB <= 32) {
                rank_count(sB, NB, rem);
            } else {
                // 256 sub-bins of the boundary bin (a monotone refinement of
                // the bin map): the sub-bin of the k'-th key, then its keys
                // gathered and ranked by counting (past 256 of them, by one
                // warp's radix passes). The unit's histogram in sRad + 256 has
                // been read; the gathered keys follow the published ones.
                int *sSub = sRad + 256;
                uint32_t *sC = reinterpret_cast<uint32_t *>(ring) + kMaxSlice;
                auto sub_bin = [&](uint32_t key) {
                    const int x = (int)__fmul_rn(__fsub_rn(lin_pos(key), (float)b_lin), 256.0f);
                    return min(255, max(0, x));
                };
                sSub[tid] = 0;
                if (tid == 0) sMisc[M_NSUB] = 0;
                __syncthreads();
#pragma unroll 1
                for (int t = tid; t < NB; t += kSelThreads) atomicAdd(&sSub[sub_bin(sB[t])], 1);
                __syncthreads();
                int sbin, sabove;
                find_bin_in(sSub, rem, sbin, sabove);
                const int rem2 = rem - sabove;
#pragma unroll 1
                for (int t = tid; t < NB; t += kSelThreads) {
                    const uint32_t k = sB[t];
                    if (sub_bin(k) == sbin) sC[atomicAdd(&sMisc[M_NSUB], 1)] = k;
                }
                __syncthreads();
                const int NC = sMisc[M_NSUB];
                if (NC <= kSelThreads) rank_count(sC, NC, rem2);
                else if (warp == 0) radix_warp(sC, NC, rem2);
            }
            __syncthreads();
            keyT = (uint32_t)sMisc[M_KEYT];
            const int quota = sMisc[M_QUOTA];
            // ties at keyT go to the lowest indices: boundary keys of earlier
            // slices (up to 256 keys: one per thread, counted by the barrier)
            int gt_before, eq_before, eq_mine;
            if (NB <= kSelThreads) {
                bool gtb = false, eqb = false, eqm = false;
                if (tid < NB) {
                    const int r2 = seg_owner(tid);
                    const uint32_t k = sB[tid];
                    gtb = r2 < rank && k > keyT;
                    eqb = r2 < rank && k == keyT;
                    eqm = r2 == rank && k == keyT;
                }
                gt_before = __syncthreads_count(gtb);
                eq_before = __syncthreads_count(eqb);
                eq_mine = __syncthreads_count(eqm);
            } else {
                int gt_b = 0, eq_b = 0, eq_m = 0;
#pragma unroll 1
                for (int t = tid; t < NB; t += kSelThreads) {
                    const int r2 = seg_owner(t);
                    const uint32_t k = sB[t];
                    if (r2 < rank) {
                        gt_b += k > keyT;
                        eq_b += k == keyT;
                    } else if (r2 == rank) {
                        eq_m += k == keyT;
                    }
                }
                gt_b = warp_sum(gt_b);
                eq_b = warp_sum(eq_b);
                eq_m = warp_sum(eq_m);
                if (lane == 0) {
                    if (gt_b) atomicAdd(&sScan[0], gt_b);
                    if (eq_b) atomicAdd(&sScan[1], eq_b);
                    if (eq_m) atomicAdd(&sScan[2], eq_m);
                }
                __syncthreads();
                gt_before = sScan[0];
                eq_before = sScan[1];
                eq_mine = sScan[2];
            }
            if (tid == 0) {
                sMisc[M_KTAKE] = max(0, min(quota - eq_before, eq_mine));
                sMisc[M_KOFF] = sMisc[M_ABOVEB] + gt_before + min(eq_before, quota);
            }
            __syncthreads();
        } else {
            // fallback: every CTA gathers all C' keys and selects within the bin
            uint32_t *sKey = reinterpret_cast<uint32_t *>(ring);
            const int per = (Cp + kSelThreads - 1) / kSelThreads;
#pragma unroll 1
            for (int base = 0; base < per; base += 8) {
                float v[8];
#pragma unroll
                for (int i = 0; i < 8; i++) {
                    const int t = (base + i) * kSelThreads + tid;
                    v[i] = 0.0f;
                    if (base + i < per && t < Cp) {
                        const int r2 = slice_owner(t);
                        v[i] = *cluster.map_shared_rank(&sS[t - sMisc[M_BOUND + r2]], r2);
                    }
                }
#pragma unroll
                for (int i = 0; i < 8; i++) {
                    const int t = (base + i) * kSelThreads + tid;
                    if (base + i < per && t < Cp) sKey[t] = order_key(v[i]);
                }
            }
            __syncthreads();
            uint32_t prefix = 0, mask = 0;
#pragma unroll 1
            for (int pass = 0; pass < 4; pass++) {
                const int shift = 24 - 8 * pass;
                histogram(Cp,
                          [&](int t) {
                              return lin_bin(sKey[t]) == b_lin && (sKey[t] & mask) == prefix;
                          },
                          [&](int t) { return (int)((sKey[t] >> shift) & 255u); });
                int dg, before;
                find_bin_in(sRad, rem, dg, before);
                rem -= before;
                prefix |= (uint32_t)dg << shift;
                mask |= 255u << shift;
            }
            keyT = prefix;
            int gt_b = 0, eq_b = 0, eq_m = 0;
#pragma unroll 1
            for (int t = tid; t < hi; t += kSelThreads) {
                const uint32_t key = sKey[t];
                if (t < lo) {
                    gt_b += key > keyT;
                    eq_b += key == keyT;
                } else {
                    eq_m += key == keyT;
                }
            }
            int gt_before, eq_before, eq_mine;
            block_exclusive_scan(gt_b, sScan, &gt_before);
            block_exclusive_scan(eq_b, sScan, &eq_before);
            block_exclusive_scan(eq_m, sScan, &eq_mine);
            if (tid == 0) {
                sMisc[M_KTAKE] = max(0, min(rem - eq_before, eq_mine));
                sMisc[M_KOFF] = gt_before + min(eq_before, rem);
            }
            __syncthreads();
        }
    }

    // With the fused attention, P7 stages rows over the code ring and the
    // candidate arrays, which the other CTAs read until they have finished
    // P5 (published boundary keys, and scores in the all-keys path): arrive
    // here, after this CTA's last read of another's shared memory, and wait
    // before the first staging write.
    if constexpr (GA > 0) {
        __syncwarp();
        cluster_arrive_release();
    }

    // ---------------------------------------------------------------- P6
    // winners of this slice, ascending by index; with the fused attention
    // they are also listed (in the plane area, free since P3) for P7
    int32_t *sWin = reinterpret_cast<int32_t *>(smem + SM::oPl);
    static_assert(8 * kPlaneCap >= kMaxSlice, "the winner list fits the plane area");
    if (GA > 0 && tid == 0 && kp == 0) sMisc[M_NW] = 0;
    if (kp > 0) {
        const int spt = (n + kSelThreads - 1) / kSelThreads;
        const int j0 = min(tid * spt, n), j1 = min(j0 + spt, n);
        int n_eq = 0, n_gt = 0;
#pragma unroll 1
        for (int j = j0; j < j1; j++) {
            const uint32_t key = order_key(sS[j]);
            n_eq += key == keyT;
            n_gt += key > keyT;
        }
        // one scan of both counts: the ties taken before this thread are the
        // first `ktake` ties in order, min(ktake, eq_before) of them
        int eq_before, gt_before;
        block_exclusive_scan2(n_eq, n_gt, sScan, &eq_before, &gt_before);
        const int ktake = sMisc[M_KTAKE];
        const int allow0 = max(0, min(ktake - eq_before, n_eq));
        int pos = gt_before + min(ktake, eq_before) + sMisc[M_KOFF];
        int32_t *orow = a.out_idx + (size_t)u * a.k;
        const int koff = sMisc[M_KOFF];
        int allow = allow0;
#pragma unroll 1
        for (int j = j0; j < j1; j++) {
            const uint32_t key = order_key(sS[j]);
            bool take = key > keyT;
            if (key == keyT && allow > 0) {
                take = true;
                allow--;
            }
            if (take) {
                if constexpr (GA > 0) sWin[pos - koff] = sI[j];
                // the attention reads the winner's V row next: start it into L2
                if (a.V)
                    prefetch_l2(static_cast<const uint8_t *>(a.V) + ((size_t)u * a.cap + sI[j]) * RB,
                                RB);
                orow[pos++] = sI[j];
            }
        }
        // the last thread's end position closes this CTA's winner segment
        if (GA > 0 && tid == kSelThreads - 1) sMisc[M_NW] = pos - koff;
    }
    if (rank == 0) {
        int32_t *orow = a.out_idx + (size_t)u * a.k;
#pragma unroll 1
        for (int j = kp + tid; j < a.k; j += kSelThreads) orow[j] = -1;
        if (tid == 0) a.out_count[u] = kp;
    }
    if constexpr (GA > 0) {
        __syncthreads();  // sWin and its length complete; sS / sI no longer read
        attend_tail<D, T, GA>(a, smem, sWin, sMisc[M_NW], b, h, N, p0, pool, rank, CS);
    }
    __syncthreads();
    cluster.sync();  // exit: no CTA leaves while another may read its shared memory
}

// ------------------------------------------------------------------ host side
//
// This file is compiled three times: as itself (the common kernels, EXT =
// false, GA = 0, and the host code), through kvr_select_ext.cu with
// KVR_SELECT_EXT_TU defined (the EXT = true kernels: reranker records and
// magnitude-aware votes) and through kvr_select_att.cu with
// KVR_SELECT_ATT_TU defined (the GA = 4 kernels: selection + attention), so
// the three sets of instantiations build in parallel.

// Long contexts: the scan and the rescoring dominate, and a CTA that shares
// its SM with another runs them at about half speed while every cluster
// barrier waits for it (two CTAs of this kernel fit an SM, and 16-CTA
// clusters cannot all take SMs of their own). There, the largest cluster
// size (16 down to 8, even, at least C / kMaxSlice) whose U clusters can all
// be resident at one CTA per SM is used, the shared memory padded past half
// an SM. Measured on the Llama-3-8B-shaped layer (8 units): 12 CTAs per unit
// on SMs of their own took the million-token step from 116.6 to 109.1 us;
// at 128K (16 half-tiles per CTA) the same took it from 39.8 to 41.7 us, so
// the spread form starts at kSpreadCap tokens of capacity.
constexpr int64_t kSpreadCap = 1 << 19;
constexpr int kSpreadSmem = 120 * 1024;

template <int D, typename T, int VB, bool EXT, int GA>
static kvr_status launch_select_t(const LaunchCtx &c, const SelArgs &a, int cs)
{
    auto kern = select_kernel<D, T, VB, EXT, GA>;
    int smem = SelSmem<D, T>::bytes;
    static_assert(SelSmem<D, T>::bytes <= kSpreadSmem, "the padded form holds the layout");
    if (c.shape.cap >= kSpreadCap) {
        const int U = c.shape.B * c.shape.Hkv;
        const int cmin = (a.C + kMaxSlice - 1) / kMaxSlice;
        if (prepare_cluster_kernel(reinterpret_cast<const void *>(kern), kSpreadSmem) == KVR_OK)
            for (int cs1 = 16; cs1 >= 8 && cs1 >= cmin; cs1 -= 2)
                if (max_active_clusters(reinterpret_cast<const void *>(kern), cs1, kSelThreads,
                                        kSpreadSmem) >= U) {
                    cs = cs1;
                    smem = kSpreadSmem;
                    break;
                }
    }
    kvr_status st = prepare_cluster_kernel(reinterpret_cast<const void *>(kern), smem);
    if (st != KVR_OK) return st;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cs, c.shape.B * c.shape.Hkv, 1);
    cfg.blockDim = dim3(kSelThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = c.stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    if (cudaLaunchKernelEx(&cfg, kern, a) != cudaSuccess) return KVR_ERR_CUDA;
    return check_launch();
}

template <int D, typename T, bool EXT, int GA>
static kvr_status launch_select_vb(const LaunchCtx &c, const SelArgs &a, int cs, int vb)
{
    switch (vb) {
    case 1: return launch_select_t<D, T, 1, EXT, GA>(c, a, cs);
    case 2: return launch_select_t<D, T, 2, EXT, GA>(c, a, cs);
    case 3: return launch_select_t<D, T, 3, EXT, GA>(c, a, cs);
    default: return launch_select_t<D, T, 4, EXT, GA>(c, a, cs);
    }
}

template <bool EXT, int GA>
static kvr_status launch_select(const LaunchCtx &c, const SelArgs &a, int cs, int vb)
{
    const bool bf = c.shape.dtype == KVR_BF16;
    if (c.shape.d == 128)
        return bf ? launch_select_vb<128, __nv_bfloat16, EXT, GA>(c, a, cs, vb)
                  : launch_select_vb<128, float, EXT, GA>(c, a, cs, vb);
    return bf ? launch_select_vb<64, __nv_bfloat16, EXT, GA>(c, a, cs, vb)
              : launch_select_vb<64, float, EXT, GA>(c, a, cs, vb);
}

#if defined(KVR_SELECT_EXT_TU)

kvr_status select_launch_ext(const LaunchCtx &c, const SelArgs &a, int cs, int vb)
{
    return launch_select<true, 0>(c, a, cs, vb);
}

#elif defined(KVR_SELECT_ATT_TU)

kvr_status select_launch_att(const LaunchCtx &c, const SelArgs &a, int cs, int vb)
{
    return launch_select<false, 4>(c, a, cs, vb);
}

#else

// defined in the KVR_SELECT_EXT_TU / KVR_SELECT_ATT_TU compilations of this file
kvr_status select_launch_ext(const LaunchCtx &c, const SelArgs &a, int cs, int vb);
kvr_status select_launch_att(const LaunchCtx &c, const SelArgs &a, int cs, int vb);

int select_cluster_size(int U, int C)
{
    int cs = 16;
    while (cs > 1 && (int64_t)U * cs > 2 * sm_count()) cs >>= 1;
    while (cs < 16 && (int64_t)cs * kMaxSlice < C) cs <<= 1;
    return cs;
}

bool select_attend_fusable(const kvr_shape &s, const kvr_select_params &p)
{
    return s.Hq / s.Hkv <= 4 && !p.rsq_records && !(p.flags & KVR_SELECT_MAGNITUDE_VOTES);
}

kvr_status select_dispatch(const LaunchCtx &c, const kvr_select_params &p, const SelectPlan &plan,
                           const void *q, const void *K, const uint8_t *codes,
                           const int32_t *seq_len, const int8_t *sgn, int32_t *out_idx,
                           int32_t *out_count, uint8_t *ws, int32_t *err, const FusedAttend *att)
{
    SelArgs a;
    a.Hq = c.shape.Hq;
    a.Hkv = c.shape.Hkv;
    a.G = c.shape.Hq / c.shape.Hkv;
    a.cap = c.shape.cap;
    a.C = p.C;
    a.k = p.k;
    a.W = p.W;
    int maxw = 0;
    for (int m = 0; m < 9; m++) maxw = p.lut[m] > maxw ? p.lut[m] : maxw;
    const int vb = maxw > 0 ? bit_width(maxw) : 1;
    for (int j = 0; j < 4; j++) {
        uint32_t bits = 0;
        for (int m = 0; m < 9; m++) bits |= (uint32_t)((p.lut[m] >> j) & 1) << m;
        a.leaf[j] = bits;
    }
    a.q = q;
    a.K = K;
    a.V = att ? att->V : p.V_prefetch;
    a.early = (p.flags & KVR_SELECT_EARLY_INPUTS) != 0;
    a.rsq = p.rsq_records;
    a.sink = p.sink;
    a.region_end = p.region_end;
    a.votes = plan.has_votes ? reinterpret_cast<const uint16_t *>(ws + plan.off_votes) : nullptr;
    for (int i = 0; i < 8; i++) a.lev[i] = rsq_tables().lev[i];
    a.codes = codes;
    a.seq_len = seq_len;
    a.sgn = sgn;
    a.out_idx = out_idx;
    a.out_count = out_count;
    a.planes = reinterpret_cast<uint32_t *>(ws + plan.off_planes);
    a.cand_idx = reinterpret_cast<int32_t *>(ws + plan.off_cand_idx);
    a.cand_score = reinterpret_cast<float *>(ws + plan.off_cand_score);
    a.cand_count = reinterpret_cast<int32_t *>(ws + plan.off_cand_count);
    a.qbar = reinterpret_cast<float *>(ws + plan.off_qbar);
    a.coarse = plan.has_coarse ? ws + plan.off_coarse : nullptr;
    a.nblk = plan.nblk;
    a.cap_pad = plan.cap_pad;
    a.tiles = plan.tiles;
    a.err = err;
    a.att_out = att ? att->out : nullptr;
    a.att_scale_log2 = att ? att->scale * 1.4426950408889634f : 0.0f;
    if (att && !select_attend_fusable(c.shape, p)) return KVR_ERR_UNSUPPORTED;
    if (plan.has_votes) {
        const kvr_status st = vote_list_dispatch(c, q, sgn, p.lut,
                                                 reinterpret_cast<uint16_t *>(ws + plan.off_votes));
        if (st != KVR_OK) return st;
    }
    const int cs = select_cluster_size(c.shape.B * c.shape.Hkv, p.C);
    if (att) return select_launch_att(c, a, cs, vb);
    if (a.rsq || a.votes) return select_launch_ext(c, a, cs, vb);
    return launch_select<false, 0>(c, a, cs, vb);
}

#endif  // KVR_SELECT_EXT_TU / KVR_SELECT_ATT_TU

}  // namespace kvr
