// verify.cu -- recursive tree speculative sampling and greedy verification (sm_103a).
//
// Pages: "EAGLE: Speculative Sampling Requires Rethinking Feature Uncertainty" (papercache.org)
// section A3 (accept a draft token with probability min(1, p/q); on rejection resample from
// norm(max(0, p - q))), section 3.3 and appendix A.2 (multi-round speculative sampling: after a
// rejection the next candidate is tested against the adjusted distribution; only when every
// candidate is rejected is a token drawn from it); "LLM speculative decoding explained"
// (hubwiz.com) sections 1-2 (p = target, q = draft; a bonus token when all are accepted;
// temperature applied to both distributions).
//
// GPU design.  The accept tests at a node never depend on the uniforms of earlier tests, only on
// how many siblings were rejected before.  After j rejections at a node with normalised target
// p0 and draft q the adjusted distribution is
//     p_j = (p0 - c_j q)+ / S_j,   S_j = sum_t (p0(t) - c_j q(t))+,   c_0 = 0, S_0 = 1,
//     c_{j+1} = c_j + S_j                         (a rejection with S_{j+1} = 0 keeps p_j),
// because max(0, (p0 - c_j q)+ / S_j - q) = (p0 - (c_j + S_j) q)+ / S_j.  So every node's whole
// rejection chain and its final draw (the walk stops at a node only after all of its children
// were rejected) can be computed for all nodes at once, in parallel, and the sequential walk over
// the tree reduces to comparisons of uniforms with precomputed ratios.
//
//   verify_prep_kernel  one cluster of CL CTAs (8, or 16 for vocabularies above 131072) per node
//                       with children (sampling, working nodes first; greedy: per pair of nodes).
//                       Each CTA bulk-copies its slices of the node's target and draft rows into
//                       shared memory; thread t takes 8 chunks of 4 tokens, chunk e at token 4 (t +
//                       512 e) of the slice, into registers.  Log-sum-exp, the S_j passes and the
//                       inverse-CDF scan are register loops; each CTA reduces a pass to one record
//                       and pushes it to every peer (st.async completing on the receiver's
//                       mbarrier), so a pass costs one point-to-point exchange, not a cluster-wide
//                       barrier.  A chain stops at its first accepted child.  When that child is a
//                       leaf the walk may end there, so the cluster also draws the leaf's bonus
//                       token from the leaf's target row (the first child's row slice is prefetched
//                       with the node's own rows, as it is the one usually accepted); the root
//                       without children draws its own final token.  Per-node statistics (row
//                       maxima, log normalisers, each child's c_j and S_j with the prep's verdict)
//                       and the draws go to the workspace.
//   verify_walk_kernel  one CTA per sequence: validates the tree and walks it over the prep's
//                       verdicts, committing the draft tokens of the accepted path and the final
//                       or bonus token the prep drew where the walk stops.  With every child's
//                       ratio wanted (out_ratio) the chains run to the end, the walk makes every
//                       test itself in double precision (one thread per node), and a walk that
//                       ends at a leaf leaves the bonus token's slot to a third launch: the prep
//                       kernel in bonus mode, one cluster per sequence, draws it from that leaf's
//                       target distribution.
#include <atomic>
#include <cooperative_groups.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "common.cuh"

namespace cg = cooperative_groups;

namespace eagle {

namespace {

constexpr int kPrepThreads = 512;
constexpr int kWarpsPrep = kPrepThreads / 32;
constexpr int kE = 32;                       // tokens per thread and row, in kChunks chunks of 4
constexpr int kChunks = kE / 4;
constexpr int kSliceMax = kPrepThreads * kE;  // one CTA's slice of a row (16384 tokens)
// the node's two rows' slices and a prefetched slice of its first child's row, 192 KB
constexpr size_t kPrepSmem = 3 * size_t(kSliceMax) * sizeof(float);
constexpr int kMaxNodes = 64;
constexpr double kFxInv = 1.0 / 4503599627370496.0;  // fixed-point unit of weight sums: 2^-52

// Per-node statistics the prep kernel leaves for the walk.  Row statistics (mp, mq, lnsp, lnsq)
// belong to a node with children; (cj, sj) to a node as a child: its parent's rejection chain
// state when this child is tested.  Child j (sibling index) is accepted when
// u < (p0/q0 - c_j)+ / S_j at its token, i.e. u S_j + c_j < p0/q0 (S_j = 0 accepts), decided
// exactly in 2^-52 units.  When a chain stops at the first accepted child, the prep makes the
// tests itself and leaves each child's verdict in the top bits of sj.
struct NodeStat {
    float mp, mq;      // row maxima (logit units)
    float lnsp, lnsq;  // ln of the normaliser sum_t exp((x_t - max) / T), target and draft rows
    uint64_t cj, sj;   // c_j, S_j (<= 2^52) in 2^-52 units; sj bits 62-63: the prep's verdict
};
constexpr int kVerdictShift = 62;  // 0: not tested by the prep, 1: rejected, 2: accepted
constexpr uint64_t kSjMask = (1ull << kVerdictShift) - 1;
static_assert(sizeof(NodeStat) == 32, "NodeStat layout");

struct VerifyArgs {
    const float *target;    // [B][n][V]
    const float *draft;     // [B][R][V]
    const int32_t *tokens;  // [B][n]
    const int32_t *parents;
    const int32_t *node_row;
    const float *uniforms;  // [B][n]
    NodeStat *stat;         // [B][n] workspace
    int32_t *final_tok;     // [B][n] workspace
    int32_t *bonus;         // [B] workspace: leaf | out slot << 8 for the bonus draw, or -1
    float *out_ratio;       // optional
    int32_t *out_tokens, *out_len, *out_path;
    int32_t *status;
    // Per-call failure tag (a word of the workspace header): a prep CTA whose wait ran out stores
    // this call's `gen` there, and the walk then commits nothing (out_len = 0) for any sequence.
    // Tags are unique per call in a process, so a tag left by an earlier call never matches.
    int32_t *fail_tag;
    int32_t gen;
    int B, n, V, R, D, slice;
    float inv_t;    // 1/T (T > 0)
    double inv_td;  // 1/T in double
    float c;        // log2(e)/T
    int greedy;
    int bonus_mode;  // the prep kernel draws the bonus token of the leaf in `bonus`
    int full_chain;  // every child tested (its ratio is an output); else a chain stops at the
                     // first accepted child
};

// ---- cluster record exchange.  Each CTA reduces a pass to one 16-byte record and pushes it into
// every peer's receive slot with st.async, whose bytes complete on the receiver's own mbarrier; a
// CTA then reads the CL records of the exchange from its own shared memory, in rank order, so all
// CTAs of the cluster derive bit-identical totals without a cluster-wide barrier per pass.  Receive
// slots alternate by exchange parity: a CTA can only send exchange e + 2 after receiving every
// record of e + 1, which each peer sends after it has consumed exchange e.
__device__ __forceinline__ uint32_t mapa_u32(uint32_t local, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
    return r;
}
__device__ __forceinline__ void st_async_v4(uint32_t raddr, float4 v, uint32_t rbar) {
    asm volatile(
        "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(raddr),
        "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(rbar)
        : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {  // release, CTA scope
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(bar)))
                 : "memory");
}
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

// ---- token layout.  Thread t of a CTA holds chunk e (e < kChunks) of its slice at tokens
// 4 (t + 512 e) .. 4 (t + 512 e) + 3, in registers v[4 e] .. v[4 e + 3]: a warp's accesses to a
// row are 16-byte contiguous per lane, so shared-memory reads are conflict-free and global reads
// coalesce.  Ascending token order is chunk column e first, then thread.
__device__ __forceinline__ int chunk_tok(int e) { return 4 * (int(threadIdx.x) + kPrepThreads * e); }

// This thread's chunks of a row slice from shared memory (cnt a multiple of 4; -inf past the end).
__device__ __forceinline__ void read_chunks(float (&v)[kE], const float *srow, int cnt) {
#pragma unroll
    for (int e = 0; e < kChunks; ++e) {
        const int t = chunk_tok(e);
        const float4 w = t < cnt ? *reinterpret_cast<const float4 *>(srow + t)
                                 : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        v[4 * e] = w.x;
        v[4 * e + 1] = w.y;
        v[4 * e + 2] = w.z;
        v[4 * e + 3] = w.w;
    }
}
// The same from global memory, one value at a time (rows that a bulk copy cannot take).
__device__ __forceinline__ void load_chunks(float (&v)[kE], const float *src, int cnt) {
#pragma unroll
    for (int e = 0; e < kChunks; ++e)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int t = chunk_tok(e) + i;
            v[4 * e + i] = t < cnt ? __ldg(src + t) : -INFINITY;
        }
}

// In place: v <- 2^((v - m) c) against the thread's max m (0 past the end); returns the sum.
__device__ __forceinline__ float exp_run(float (&v)[kE], float &m, float c) {
    m = -INFINITY;
#pragma unroll
    for (int j = 0; j < kE; ++j) m = fmaxf(m, v[j]);
    const float mc = m == -INFINITY ? 0.f : m * c;
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < kE; ++j) {
        v[j] = v[j] == -INFINITY ? 0.f : fast_exp2(fmaf(v[j], c, -mc));
        s += v[j];
    }
    return s;
}

// ---- fixed point.  Weight sums (probabilities, residuals) are carried as integers in units of
// 2^-52, so every sum above the chunk level is exact: the same in every thread and CTA that forms
// it, whatever the order, and consistent between the per-rank totals and a CTA's own scan.
// A chunk's weight (<= 4 values in [0, 1]) is clamped to [0, 2); NaN maps to 0.  Conversions in
// both directions use 32-bit integer arithmetic only: 64-bit conversions and doubles run on the
// (slow) FP64 pipe.
__device__ __forceinline__ uint64_t to_fx(float x) {
    if (!(x > 0.f)) return 0ull;
    const uint32_t bits = __float_as_uint(fminf(x, 1.99999988f));
    const int ex = int(bits >> 23);  // biased exponent, <= 127
    if (ex == 0) return 0ull;        // below 2^-126
    const uint32_t m = (bits & 0x7fffffu) | 0x800000u;  // x = m 2^(ex - 150), fx = m 2^(ex - 98)
    return ex >= 98 ? (uint64_t(m) << (ex - 98)) : (ex > 74 ? uint64_t(m >> (98 - ex)) : 0ull);
}
// A fixed-point value as a float (within 1.5 float ulps; every caller forms a given c the same way).
__device__ __forceinline__ float fx_to_float(uint64_t v) {
    return fmaf(__uint2float_rn(uint32_t(v >> 32)), 9.5367431640625e-07f /* 2^-20 */,
                __uint2float_rn(uint32_t(v)) * 2.220446049250313e-16f /* 2^-52 */);
}
__device__ __forceinline__ float4 fx_rec(uint64_t v) {
    return make_float4(__uint_as_float(uint32_t(v)), __uint_as_float(uint32_t(v >> 32)), 0.f, 0.f);
}
__device__ __forceinline__ uint64_t rec_fx(float4 r) {
    return (uint64_t(__float_as_uint(r.y)) << 32) | __float_as_uint(r.x);
}
// A chunk's weight: its four weights summed in this order in float, then in fixed point.
__device__ __forceinline__ uint64_t chunk_weight(float w0, float w1, float w2, float w3) {
    return to_fx(((w0 + w1) + w2) + w3);
}
__device__ __forceinline__ uint64_t clamp53(uint64_t t) { return t < (1ull << 53) ? t : (1ull << 53) - 1; }
// This thread's weight of (p - c q)+ (a pass of the rejection chain) or of w itself (q == nullptr).
__device__ __forceinline__ uint64_t residual_fx(const float (&p)[kE], const float (&q)[kE], float c) {
    uint64_t t = 0;
#pragma unroll
    for (int e = 0; e < kChunks; ++e)
        t += chunk_weight(fmaxf(fmaf(-c, q[4 * e], p[4 * e]), 0.f), fmaxf(fmaf(-c, q[4 * e + 1], p[4 * e + 1]), 0.f),
                          fmaxf(fmaf(-c, q[4 * e + 2], p[4 * e + 2]), 0.f), fmaxf(fmaf(-c, q[4 * e + 3], p[4 * e + 3]), 0.f));
    return clamp53(t);
}
__device__ __forceinline__ uint64_t weight_fx(const float (&w)[kE]) {
    uint64_t t = 0;
#pragma unroll
    for (int e = 0; e < kChunks; ++e) t += chunk_weight(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
    return clamp53(t);
}

// p0/q0 in 2^-52 units, clamped at 2^11 (c_j <= 64 and u S_j < 1, so the clamp never decides a
// test); NaN and non-positive ratios give 0.
__device__ __forceinline__ uint64_t ratio_fx(double rr) {
    const double v = rr * 4503599627370496.0;  // 2^52
    return v >= 9223372036854775808.0 ? (1ull << 63) : (v > 0.0 ? __double2ull_rz(v) : 0ull);
}
// The accept test u < (p0/q0 - c)+ / S, as u S + c < p0/q0 in 2^-52 units (S = 0 accepts).
__device__ __forceinline__ bool accept_fx(float u, uint64_t c, uint64_t S, uint64_t rrfx) {
    return S == 0 || scale_fx(S, u) + c < rrfx;
}

// Warp-wide merge of (max, scaled sum) pairs: M = max over the lanes, S = sum of s 2^((m - M) c)
// (the same in every lane: one max reduction, one exponential per lane, a butterfly sum).
__device__ __forceinline__ float2 ms_fold(float m, float s, float c) {
    const float M = float_from_order_key(__reduce_max_sync(0xffffffffu, float_order_key(m)));
    float t = m == -INFINITY ? 0.f : s * fast_exp2((m - M) * c);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) t += __shfl_xor_sync(0xffffffffu, t, off);
    return make_float2(M, t);
}
__device__ __forceinline__ float4 ms_fold2(float4 v, float c) {
    const float2 a = ms_fold(v.x, v.y, c), b = ms_fold(v.z, v.w, c);
    return make_float4(a.x, a.y, b.x, b.y);
}

// Owner of a final draw, warp-parallel: lane r < CL holds rank r's weight total (fixed point, 0
// in the other lanes; ascending rank = ascending token id).  The owner is the rank holding the
// first cumulative step above u * total; owner = -1 when there is no mass at all; local = the
// target minus the owner's starting sum.  Same result in every lane.
template <int CL>
__device__ __forceinline__ void decide_owner_warp(uint64_t t, float u, int &owner, uint64_t &local) {
    const int lane = threadIdx.x & 31;
    uint64_t incl = t;
#pragma unroll
    for (int off = 1; off < CL; off <<= 1) {
        const uint64_t o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
    }
    const uint64_t total = __shfl_sync(0xffffffffu, incl, CL - 1);
    owner = -1;
    local = 0;
    if (total == 0) return;
    const uint64_t tgt = scale_fx(total, u);  // < total
    const uint64_t excl = incl - t;
    const unsigned m = __ballot_sync(0xffffffffu, lane < CL && excl <= tgt && tgt < incl);
    owner = __ffs(m) - 1;  // exactly one lane: the steps tile [0, total)
    local = __shfl_sync(0xffffffffu, tgt - excl, owner);
}

// Final draw over this CTA's slice (CTA-uniform call): w holds this thread's weights; the draw
// takes the first token, in ascending id order, whose cumulative weight exceeds `local` (fixed
// point, relative to the slice).  Column totals and the warp's lane scan are exact; inside the
// chosen chunk the float partial sums are the ones its chunk weight was formed from.  If `local`
// lies at or beyond the slice's total (per-rank totals formed from other sums), the last token of
// positive weight is taken.  Returns the token's offset in the slice in one thread, -1 elsewhere.
struct DrawSmem {
    uint64_t col[kWarpsPrep][kChunks];  // per-warp totals of every chunk column
    uint64_t rem;
    int pick_col, pick_warp, last;
};
__device__ __forceinline__ int draw_in_slice(const float (&w)[kE], uint64_t local, DrawSmem &ds) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int tlast = -1;
#pragma unroll
    for (int e = 0; e < kChunks; ++e) {
        const uint64_t t = warp_sum_fx(chunk_weight(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]));
        if (lane == 0) ds.col[warp][e] = t;
#pragma unroll
        for (int i = 0; i < 4; ++i)
            if (w[4 * e + i] > 0.f) tlast = max(tlast, chunk_tok(e) + i);
    }
    tlast = __reduce_max_sync(0xffffffffu, tlast + 1) - 1;
    if (tid == 0) ds.last = -1;
    __syncthreads();
    if (lane == 0 && tlast >= 0) atomicMax(&ds.last, tlast);
    if (warp == 0) {
        // the chunk column holding the target, then the warp within it (same in every lane)
        uint64_t base = 0, colbase = 0;
        int col = -1;
#pragma unroll
        for (int e = 0; e < kChunks; ++e) {
            uint64_t t = 0;
            for (int w2 = 0; w2 < kWarpsPrep; ++w2) t += ds.col[w2][e];
            if (col < 0 && local < base + t) {
                col = e;
                colbase = base;
            }
            base += t;
        }
        int wsel = -1;
        uint64_t rem = 0;
        if (col >= 0) {
            uint64_t acc = colbase;
            for (int w2 = 0; w2 < kWarpsPrep; ++w2) {
                const uint64_t t = ds.col[w2][col];
                if (wsel < 0 && local < acc + t) {
                    wsel = w2;
                    rem = local - acc;
                }
                acc += t;
            }
        }
        if (lane == 0) {
            ds.pick_col = col;
            ds.pick_warp = wsel;
            ds.rem = rem;
        }
    }
    __syncthreads();
    const int col = ds.pick_col;
    int found = -1;
    if (col < 0) {
        if (tid == 0) found = max(ds.last, 0);
    } else if (warp == ds.pick_warp) {
        float c0 = 0.f, c1 = 0.f, c2 = 0.f, c3 = 0.f;
#pragma unroll
        for (int e = 0; e < kChunks; ++e)
            if (e == col) {
                c0 = w[4 * e];
                c1 = w[4 * e + 1];
                c2 = w[4 * e + 2];
                c3 = w[4 * e + 3];
            }
        const uint64_t mine = chunk_weight(c0, c1, c2, c3);
        uint64_t incl = mine;  // inclusive scan over the lanes
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const uint64_t o = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += o;
        }
        const uint64_t rem = ds.rem, excl = incl - mine;
        const unsigned claim = __ballot_sync(0xffffffffu, excl <= rem && rem < incl);
        if (claim && lane == __ffs(claim) - 1) {
            // inside the chunk: the float partial sums of its weight, against the remainder
            const float r = fx_to_float(rem - excl);
            const float a1 = c0 + c1, a2 = a1 + c2, a3 = a2 + c3;
            const int t0 = chunk_tok(col);
            int lastp = -1;
            if (c0 > 0.f) lastp = 0;
            if (c1 > 0.f) lastp = 1;
            if (c2 > 0.f) lastp = 2;
            if (c3 > 0.f) lastp = 3;
            int i = (c0 > 0.f && c0 > r) ? 0 : (c1 > 0.f && a1 > r) ? 1 : (c2 > 0.f && a2 > r) ? 2 : (c3 > 0.f && a3 > r) ? 3 : lastp;
            found = t0 + max(i, 0);
        } else if (!claim && lane == 0) {
            found = max(ds.last, 0);  // cannot happen with exact sums; kept as a guard
        }
    }
    return found;
}

template <int CL>
__global__ void __launch_bounds__(kPrepThreads, 1) verify_prep_kernel(VerifyArgs a) {
    pdl_wait();
    pdl_launch_next();
    extern __shared__ __align__(16) float s_rows[];  // [2][kSliceMax]: the two held rows' slices
    __shared__ float4 s_wp[kWarpsPrep];              // per-warp partials of the current pass
    __shared__ float4 s_recv[2][CL];                 // the cluster's records of an exchange, by parity
    __shared__ __align__(8) uint64_t s_rbar[2];
    __shared__ __align__(8) uint64_t s_pbar;     // every warp's partial of the current pass posted
    __shared__ __align__(8) uint64_t s_lbar[3];  // a row slice landed
    __shared__ int s_kid[kMaxNodes];             // children of the node (sampling), ascending
    __shared__ uint64_t s_rrfx[kMaxNodes];       // each child's p0/q0 at its token, 2^-52 units
    __shared__ float s_uk[kMaxNodes];            // each child's uniform
    __shared__ int s_dec[2];                     // the accept test of the current child, by parity
    __shared__ __align__(8) uint64_t s_decbar;   // s_dec written
    __shared__ int s_nk, s_fail, s_second, s_y;
    __shared__ uint64_t s_leaves;  // the tree's leaves (nodes without children), one bit each
    __shared__ int s_acc;          // the child at which the chain stopped (accepted)
    __shared__ int s_pre;          // the child whose target row slice was prefetched, or -1
    __shared__ int s_own[1];
    __shared__ uint64_t s_local[1];
    __shared__ DrawSmem s_draw;

    cg::cluster_group cluster = cg::this_cluster();
    const int rank = int(cluster.block_rank());
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n = a.n, V = a.V, b = blockIdx.y;
    const int lo = rank * a.slice;
    const int hi = min(V, lo + a.slice);
    const int cnt = hi > lo ? hi - lo : 0;
    const int32_t *par = a.parents + size_t(b) * n;

    // ---- work of this cluster (cluster index s = blockIdx.z, sequence b = blockIdx.y).  Greedy:
    // nodes 2s and 2s + 1 (argmax of two target rows).  Sampling: the s-th working node in index
    // order, a node with children or the root (found by the tree scan below; clusters past the
    // last working node exit), so that the clusters with work are the first ones the GPU places.
    // Bonus mode: the leaf the walk ended at, if any (written by the walk, the launch before this).
    const int breq = a.bonus_mode ? __ldg(a.bonus + blockIdx.y) : -1;
    if (a.bonus_mode && breq < 0) return;  // uniform for the cluster: nothing has started
    const int cs = int(blockIdx.z);
    // The barriers exist before anything else, and the cluster barrier that publishes them to the
    // peers is arrived at now and waited on only before the first exchange, so its latency hides
    // behind the tree scan, the slice copies and the first register pass.
    if (tid == 0) {
        mbar_init(&s_rbar[0], 1);
        mbar_init(&s_rbar[1], 1);
        mbar_init(&s_pbar, kWarpsPrep);
        mbar_init(&s_lbar[0], 1);
        mbar_init(&s_lbar[1], 1);
        mbar_init(&s_lbar[2], 1);
        mbar_init(&s_decbar, 1);
        fence_barrier_init();
    }
    cluster_arrive();
    if (a.bonus_mode) {  // the leaf's own target row only: no tree to scan
        if (tid == 0) {
            s_nk = 0;
            s_second = -1;
            s_fail = 0;
            s_own[0] = -1;
            s_y = breq & 255;
        }
    } else if (warp == 0) {
        // every node's "has children" bit, this cluster's node y, and its children, from the <= 64
        // parents
        const int p0 = lane < n ? __ldg(par + lane) : -1;
        const int p1 = lane + 32 < n ? __ldg(par + lane + 32) : -1;
        uint64_t mine = 0;
        if (lane > 0 && p0 >= 0 && p0 < n) mine |= 1ull << p0;
        if (p1 >= 0 && p1 < n) mine |= 1ull << p1;
        const unsigned ml = __reduce_or_sync(0xffffffffu, uint32_t(mine));
        const unsigned mh = __reduce_or_sync(0xffffffffu, uint32_t(mine >> 32));
        const uint64_t internal = (uint64_t(mh) << 32) | ml;
        const uint64_t all = n >= 64 ? ~0ull : ((1ull << n) - 1ull);
        const uint64_t leaves = all & ~internal;
        int y = a.greedy ? cs : -1;
        if (!a.greedy) {
            // working nodes: those with children, and the root unless every ratio is wanted (it
            // then has its own draw only when it has children)
            uint64_t work = internal | (a.full_chain ? 0ull : 1ull);
            if (cs < __popcll(work)) {
                for (int i = 0; i < cs; ++i) work &= work - 1ull;  // drop the cs lowest working nodes
                y = __ffsll(static_cast<long long>(work)) - 1;
            }
        }
        const bool k0 = y >= 0 && lane > 0 && p0 == y, k1 = y >= 0 && p1 == y;
        const unsigned b0 = __ballot_sync(0xffffffffu, k0), b1 = __ballot_sync(0xffffffffu, k1);
        if (k0) s_kid[__popc(b0 & ((1u << lane) - 1u))] = lane;
        if (k1) s_kid[__popc(b0) + __popc(b1 & ((1u << lane) - 1u))] = lane + 32;
        if (lane == 0) {
            s_nk = __popc(b0) + __popc(b1);
            int second = -1;  // greedy: the paired node (-2: this cluster has no work)
            if (!a.greedy && y < 0) second = -2;  // past the last working node
            s_leaves = leaves;
            s_y = y < 0 ? 0 : y;
            if (a.greedy) second = 2 * y + 1 < n ? 2 * y + 1 : -1;
            s_second = second;
            s_fail = 0;
            s_own[0] = -1;
        }
    }
    __syncthreads();
    const int second = s_second;
    if (second == -2) return;  // uniform for the cluster: no exchange or copy has started
    const int nodeA = a.greedy ? 2 * cs : s_y;
    const int nrow = a.greedy ? -1 : __ldg(a.node_row + size_t(b) * n + nodeA);
    const int J = a.greedy ? 0 : s_nk;
    const int nodeB = a.greedy ? second : -1;  // greedy: the paired node
    const int rowq = J > 0 ? nrow : -1;
    const bool has_q = J > 0 && rowq >= 0 && rowq < a.R;
    // warp 4: the children's logits at their tokens, loaded now for the accept tests
    float kx = 0.f, ky = 0.f;
    int ktok = -1;
    if (warp == 4 && has_q)
        for (int jj = lane; jj < J && jj < 32; jj += 32) {
            ktok = __ldg(a.tokens + size_t(b) * n + s_kid[jj]);
            if (ktok >= 0 && ktok < V) {
                kx = __ldg(a.target + (size_t(b) * n + nodeA) * V + ktok);
                ky = __ldg(a.draft + (size_t(b) * a.R + rowq) * V + ktok);
            }
        }
    const float *rowA = a.target + (size_t(b) * n + nodeA) * V + lo;
    const float *rowB = nullptr;
    if (nodeB >= 0) rowB = a.target + (size_t(b) * n + nodeB) * V + lo;
    else if (has_q) rowB = a.draft + (size_t(b) * a.R + rowq) * V + lo;
    // whole slices by bulk copy into shared memory (16-byte aligned rows of a multiple of 4 floats)
    auto bulk_ok = [&](const float *r) {
        return r && ((V & 3) == 0) && ((reinterpret_cast<uintptr_t>(r) & 15) == 0) && cnt > 0;
    };
    const bool bulkA = bulk_ok(rowA), bulkB = bulk_ok(rowB);
    // The first child is the one most often accepted; when it is a leaf the walk may end there
    // and need its bonus draw, so its target row's slice follows the node's own two rows in,
    // issued once those have landed so that it does not share their bandwidth (used only if that
    // child is accepted; the CTA waits for it before leaving either way).
    const float *rowP = nullptr;
    if (tid == 0) {
        const int pre = (!a.greedy && !a.bonus_mode && !a.full_chain && has_q && ((s_leaves >> s_kid[0]) & 1ull))
                            ? s_kid[0] : -1;
        rowP = pre >= 0 ? a.target + (size_t(b) * n + pre) * V + lo : nullptr;
        s_pre = bulk_ok(rowP) ? pre : -1;
        if (bulkA) {
            mbar_expect_tx(&s_lbar[0], uint32_t(cnt) * 4u);
            bulk_g2s(s_rows, rowA, uint32_t(cnt) * 4u, &s_lbar[0]);
        }
        if (bulkB) {
            mbar_expect_tx(&s_lbar[1], uint32_t(cnt) * 4u);
            bulk_g2s(s_rows + kSliceMax, rowB, uint32_t(cnt) * 4u, &s_lbar[1]);
        }
    }
    // every final draw uses the sequence's first uniform (the root's, which no accept test uses)
    const float uA = __ldg(a.uniforms + size_t(b) * n);
    float xp[kE], xq[kE];
    if (!bulkA) load_chunks(xp, rowA, cnt);
    if (rowB && !bulkB) load_chunks(xq, rowB, cnt);
    // A slice copy that does not land marks the CTA failed; the CTA still waits (bounded) for it
    // before it can leave, as the copy writes into its shared memory.
    auto wait_slice = [&](int i) {
        const bool got = mbar_warp_wait_bounded(&s_lbar[i], 0);
        if (!got && lane == 0) {
            s_fail = 1;
            set_status(a.status, EAGLE_ERR_TIMEOUT);
            atomicExch(a.fail_tag, a.gen);
        }
    };
    if (bulkA) {
        wait_slice(0);
        read_chunks(xp, s_rows, cnt);
    }
    if (bulkB) {
        wait_slice(1);
        read_chunks(xq, s_rows + kSliceMax, cnt);
    }
    if (tid == 0 && s_pre >= 0) {  // the first child's slice, now that the node's own have landed
        mbar_expect_tx(&s_lbar[2], uint32_t(cnt) * 4u);
        bulk_g2s(s_rows + 2 * kSliceMax, rowP, uint32_t(cnt) * 4u, &s_lbar[2]);
    }

    // One pass = one exchange.  Every warp leaves its partial in s_wp[warp] and arrives on s_pbar;
    // warp 0 waits for all sixteen, folds them into the CTA's record and pushes it to every CTA of
    // the cluster; then each warp that needs the pass's totals waits for the CL records itself and
    // folds them in rank order (identical in every thread of the cluster), so a pass costs no
    // CTA-wide barrier and no broadcast.  A wait that runs out marks the CTA failed (its results
    // are then not written) and later waits return at once.
    int xch = 0, nposts = 0;  // exchanges received, posts waited on
    auto failed = [&]() { return __any_sync(0xffffffffu, *reinterpret_cast<volatile int *>(&s_fail) != 0); };
    auto fail = [&]() {
        if (lane == 0) {
            s_fail = 1;
            set_status(a.status, EAGLE_ERR_TIMEOUT);
            atomicExch(a.fail_tag, a.gen);
        }
    };
    auto post = [&](float4 v) {  // lane 0's v: this warp's partial
        if (lane == 0) {
            s_wp[warp] = v;
            mbar_arrive(&s_pbar);
        }
    };
    auto wait_posts = [&]() -> bool {  // warp 0
        const bool got = !failed() && mbar_warp_wait_bounded(&s_pbar, nposts & 1);
        ++nposts;
        if (!got) fail();
        return got;
    };
    auto send = [&](float4 rec) {  // warp 0, rec the same in every lane
        const int slot = xch & 1;
        if (lane == 0) mbar_expect_tx(&s_rbar[slot], CL * 16);
        __syncwarp();
        if (lane < CL)
            st_async_v4(mapa_u32(static_cast<uint32_t>(__cvta_generic_to_shared(&s_recv[slot][rank])), lane), rec,
                        mapa_u32(static_cast<uint32_t>(__cvta_generic_to_shared(&s_rbar[slot])), lane));
    };
    auto wait_recv = [&]() -> bool {  // the CL records of the current exchange are in s_recv
        const int slot = xch & 1;
        const bool got = !failed() && mbar_warp_wait_cluster_bounded(&s_rbar[slot], (xch >> 1) & 1);
        ++xch;
        if (!got) fail();
        return got;
    };
    // exact sums of fixed-point records: the sixteen warp partials, the CL CTA records
    auto fold_posts = [&]() {
        uint64_t t = 0;
#pragma unroll
        for (int w2 = 0; w2 < kWarpsPrep; ++w2) t += rec_fx(s_wp[w2]);
        return t;
    };
    auto recv_fx = [&]() -> uint64_t {  // the exchange's total; its records stay in s_recv
        const int slot = xch & 1;
        uint64_t t = 0;
        if (wait_recv())
#pragma unroll
            for (int r = 0; r < CL; ++r) t += rec_fx(s_recv[slot][r]);
        return t;
    };

    if (a.greedy) {
        // argmax of the two target rows (ties to the lower id): thread, warp, CTA, cluster
        uint64_t ba = 0, bb = 0;
#pragma unroll
        for (int e = 0; e < kChunks; ++e)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int j = 4 * e + i;
                const uint32_t t = uint32_t(lo + chunk_tok(e) + i);
                const uint64_t ka = xp[j] == -INFINITY ? 0ull : topk_key(xp[j], t);
                ba = ka > ba ? ka : ba;
                if (nodeB >= 0) {
                    const uint64_t kb = xq[j] == -INFINITY ? 0ull : topk_key(xq[j], t);
                    bb = kb > bb ? kb : bb;
                }
            }
        ba = warp_max_u64(ba);
        bb = warp_max_u64(bb);
        cluster_wait();  // every peer's barriers exist
        post(make_float4(__uint_as_float(uint32_t(ba)), __uint_as_float(uint32_t(ba >> 32)),
                         __uint_as_float(uint32_t(bb)), __uint_as_float(uint32_t(bb >> 32))));
        if (warp == 0) {
            uint64_t ga = 0, gb = 0;
            if (wait_posts()) {
                if (lane < kWarpsPrep) {
                    const float4 v = s_wp[lane];
                    ga = (uint64_t(__float_as_uint(v.y)) << 32) | __float_as_uint(v.x);
                    gb = (uint64_t(__float_as_uint(v.w)) << 32) | __float_as_uint(v.z);
                }
                ga = warp_max_u64(ga);
                gb = warp_max_u64(gb);
                send(make_float4(__uint_as_float(uint32_t(ga)), __uint_as_float(uint32_t(ga >> 32)),
                                 __uint_as_float(uint32_t(gb)), __uint_as_float(uint32_t(gb >> 32))));
            }
            const int slot = xch & 1;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (wait_recv() && lane < CL) v = s_recv[slot][lane];
            ga = (uint64_t(__float_as_uint(v.y)) << 32) | __float_as_uint(v.x);
            gb = (uint64_t(__float_as_uint(v.w)) << 32) | __float_as_uint(v.z);
            ga = warp_max_u64(ga);
            gb = warp_max_u64(gb);
            if (rank == 0 && lane == 0 && !s_fail) {
                a.final_tok[size_t(b) * n + nodeA] = int32_t(topk_key_token(ga));
                if (nodeB >= 0) a.final_tok[size_t(b) * n + nodeB] = int32_t(topk_key_token(gb));
            }
        }
        cluster_arrive();
        cluster_wait();
        return;
    }

    // sampling from here on: the second held row is the node's draft row (no paired node)
    const float c = a.c;
    // ---- row statistics of both held rows.  Values become 2^((x - m) c) against the thread's max
    // m, so the probabilities later cost one multiply each (no second exponential).
    float mA, mB = -INFINITY, sB = 0.f;
    float4 gst;  // the rows' global (max, sum) statistics
    const float sA = exp_run(xp, mA, c);
    if (rowB) sB = exp_run(xq, mB, c);
    cluster_wait();  // every peer's barriers exist
    {
        const float4 neutral = make_float4(-INFINITY, 0.f, -INFINITY, 0.f);
        post(ms_fold2(make_float4(mA, sA, mB, sB), c));
        if (warp == 0 && wait_posts()) send(ms_fold2(lane < kWarpsPrep ? s_wp[lane] : neutral, c));
        const int slot = xch & 1;
        const bool ok = wait_recv();
        const float4 mine = ok && lane < CL ? s_recv[slot][lane] : neutral;  // lane r < CL: rank r's record
        const float4 g = ms_fold2(mine, c);
        const float l2A = g.y > 0.f ? log2f(g.y) : 0.f;
        const float l2B = g.w > 0.f ? log2f(g.w) : 0.f;
        // side work off warp 0 (which gathers the next pass): a node without a draft row (the
        // bonus launch's leaf, or the root without children) draws from its target
        // distribution: the draw's owner from the per-rank probability totals; and the node's row
        // statistics
        if (warp == 1 && !has_q) {
            const float tr = mine.x == -INFINITY ? 0.f : mine.y * fast_exp2((mine.x - g.x) * c - l2A);
            int own;
            uint64_t loc;
            decide_owner_warp<CL>(lane < CL ? to_fx(tr) : 0ull, uA, own, loc);
            if (lane == 0) {
                s_own[0] = own;
                s_local[0] = loc;
            }
        }
        gst = g;
        if (warp == 3 && lane == 0 && rank == 0 && J > 0 && !s_fail) {
            NodeStat *st = a.stat + size_t(b) * n + nodeA;
            st->mp = g.x;
            st->mq = g.z;
            st->lnsp = logf(g.y);
            st->lnsq = has_q && g.w > 0.f ? logf(g.w) : 0.f;
        }
        // probabilities: p = 2^((x - m) c) * 2^((m - M) c - log2 S), one exponential per thread
        const float fA = mA == -INFINITY ? 0.f : fast_exp2(fmaf(mA - g.x, c, -l2A));
#pragma unroll
        for (int j = 0; j < kE; ++j) xp[j] *= fA;
        if (rowB) {
            const float fB = mB == -INFINITY ? 0.f : fast_exp2(fmaf(mB - g.z, c, -l2B));
#pragma unroll
            for (int j = 0; j < kE; ++j) xq[j] *= fB;
        }
    }

    // ---- rejection chain of a node with children: c_0 = 0, S_0 = 1; after rejecting child j:
    // c_{j+1} = c_j + S_j and S_{j+1} = sum (p0 - c_{j+1} q)+ (a zero sum keeps the previous
    // distribution).  c_j and S_j are fixed-point integers, the same in every thread; each pass
    // uses c_{j+1} rounded to float.  When the last pass moves c, its per-rank sums are exactly
    // the final draw's per-rank weights: the residual below is formed with the same float c.
    // Child j is tested with c_j and S_j, known before pass j; pass j is issued first and the
    // test is made while its exchange is in flight.  Unless every ratio is wanted, the chain stops
    // at the first accepted child: the walk takes that child, and the node's final draw (made
    // only when every child is rejected) is not needed.
    // warp 4: every child's p0/q0 at its token, in double precision from the row statistics:
    // exp(((x - Mp) / T - ln Sp) - ((y - Mq) / T - ln Sq)), its fixed-point image, and its uniform
    // (lanes past 32 children load their logits here)
    auto child_ratios = [&]() {
        const double lnsp = double(logf(gst.y)), lnsq = gst.w > 0.f ? double(logf(gst.w)) : 0.0;
        for (int jj = lane; jj < J; jj += 32) {
            const int kid = s_kid[jj];
            if (jj >= 32) {
                ktok = __ldg(a.tokens + size_t(b) * n + kid);
                if (ktok >= 0 && ktok < V) {
                    kx = __ldg(a.target + (size_t(b) * n + nodeA) * V + ktok);
                    ky = __ldg(a.draft + (size_t(b) * a.R + rowq) * V + ktok);
                }
            }
            double rr = NAN;
            if (ktok >= 0 && ktok < V)
                rr = exp(((double(kx) - double(gst.x)) * a.inv_td - lnsp) - ((double(ky) - double(gst.z)) * a.inv_td - lnsq));
            s_rrfx[jj] = ratio_fx(rr);
            s_uk[jj] = __ldg(a.uniforms + size_t(b) * n + kid);
        }
        __syncwarp();
    };
    uint64_t cj = 0, Sj = 1ull << 52;
    float cnf = 1.f;  // c_1 = c_0 + S_0
    bool decided = !has_q;
    bool accepted = false;  // a child was accepted and the chain stopped there (s_acc)
    for (int j = 0; j < J && has_q; ++j) {
        // the last pass forms exact chunk weights (they may become the final draw's); earlier
        // passes need only the sum: one float sum per thread
        uint64_t part;
        if (j == J - 1) {
            part = residual_fx(xp, xq, cnf);
        } else {
            float t0 = 0.f, t1 = 0.f, t2 = 0.f, t3 = 0.f;  // four chains of dependent adds
#pragma unroll
            for (int e = 0; e < kE; e += 4) {
                t0 += fmaxf(fmaf(-cnf, xq[e], xp[e]), 0.f);
                t1 += fmaxf(fmaf(-cnf, xq[e + 1], xp[e + 1]), 0.f);
                t2 += fmaxf(fmaf(-cnf, xq[e + 2], xp[e + 2]), 0.f);
                t3 += fmaxf(fmaf(-cnf, xq[e + 3], xp[e + 3]), 0.f);
            }
            part = to_fx((t0 + t1) + (t2 + t3));
        }
        post(fx_rec(warp_sum_fx(part)));
        // The accept test of child j, made by one lane of warp 4 while the pass's exchange runs
        // (double precision stays off the other warps: the FP64 pipe is narrow), published
        // through s_dec and s_decbar; every warp reads it after the exchange.  The inputs are the
        // same in every CTA, so every CTA of the cluster takes the same decision.
        if (warp == 4) {
            if (j == 0 && !a.full_chain) child_ratios();
            if (lane == 0 && a.full_chain) {  // the walk makes every test
                if (rank == 0 && !s_fail) {
                    NodeStat *st = a.stat + size_t(b) * n + s_kid[j];
                    st->cj = cj;
                    st->sj = Sj;
                }
            } else if (lane == 0) {
                // u < (p0/q0 - c_j)+ / S_j, i.e. u S_j + c_j < p0/q0, exactly in 2^-52 units (an
                // empty residual, S_j = 0, accepts)
                const bool acc = accept_fx(s_uk[j], cj, Sj, s_rrfx[j]);
                s_dec[j & 1] = acc;
                if (rank == 0 && !s_fail) {
                    NodeStat *st = a.stat + size_t(b) * n + s_kid[j];
                    st->cj = cj;
                    st->sj = Sj | (uint64_t(acc ? 2 : 1) << kVerdictShift);
                    if (acc)
                        for (int k2 = j + 1; k2 < J; ++k2) a.stat[size_t(b) * n + s_kid[k2]].sj = 0;  // not tested
                }
                mbar_arrive(&s_decbar);
            }
            __syncwarp();
        }
        if (warp == 0 && wait_posts()) send(fx_rec(fold_posts()));
        const int slot = xch & 1;
        const uint64_t g = recv_fx();  // received in every case: the exchanges stay paired
        if (!a.full_chain) {
            if (!mbar_warp_wait_bounded(&s_decbar, j & 1)) fail();
            if (*reinterpret_cast<volatile int *>(&s_dec[j & 1])) {
                accepted = true;
                if (tid == 0) s_acc = s_kid[j];
                break;
            }
        }
        const bool moved = g > 0;
        if (moved) {
            cj += Sj;
            Sj = g;
        }
        cnf = fx_to_float(cj + Sj);
        if (j == J - 1) {
            decided = moved;
            if (moved && warp == 0) {
                int own;
                uint64_t loc;
                decide_owner_warp<CL>(lane < CL ? rec_fx(s_recv[slot][lane]) : 0ull, uA, own, loc);
                if (lane == 0) {
                    s_own[0] = own;
                    s_local[0] = loc;
                }
            }
        }
    }
    // residual weights of a node with children: (p0 - c_J q)+, with c_J as the pass that set it
    // rounded it
    if (has_q && !accepted) {
        const float cjf = fx_to_float(cj);
#pragma unroll
        for (int e = 0; e < kE; ++e) xp[e] = fmaxf(fmaf(-cjf, xq[e], xp[e]), 0.f);
    }
    if (has_q && !decided && !accepted) {
        // the last pass left c unchanged: one more exchange for the residual's per-rank weights
        post(fx_rec(warp_sum_fx(weight_fx(xp))));
        if (warp == 0) {
            if (wait_posts()) send(fx_rec(fold_posts()));
            const int slot = xch & 1;
            recv_fx();
            int own;
            uint64_t loc;
            decide_owner_warp<CL>(lane < CL ? rec_fx(s_recv[slot][lane]) : 0ull, uA, own, loc);
            if (lane == 0) {
                s_own[0] = own;
                s_local[0] = loc;
            }
        }
    }
    // ---- an accepted child that is a leaf: the walk may end there, with a bonus token drawn from
    // the leaf's own target distribution (inverse CDF with the sequence's first uniform).  It is
    // drawn here, while the other nodes' chains still run, instead of in a launch after the walk
    // (unless every ratio is wanted: the walk then makes the tests and the bonus launch the draw).
    // The decision is the same in every CTA of the cluster, so the exchanges stay paired.
    if (accepted) __syncthreads();  // s_acc is visible; every thread has read its row A chunks
    const int spec = (accepted && !a.full_chain && ((s_leaves >> s_acc) & 1ull)) ? s_acc : -1;
    if (spec >= 0) {
        const float *rowL = a.target + (size_t(b) * n + spec) * V + lo;
        const bool pref = spec == s_pre;              // prefetched into the third slice buffer
        const bool copy = !pref && bulk_ok(rowL);     // else copied now into the first one
        if (copy && tid == 0) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // generic reads before the copy
            mbar_expect_tx(&s_lbar[0], uint32_t(cnt) * 4u);
            bulk_g2s(s_rows, rowL, uint32_t(cnt) * 4u, &s_lbar[0]);
        }
        if (pref || copy) {
            // the first buffer's barrier is in its phase 1 after the row A copy, else 0
            const bool got = mbar_warp_wait_bounded(&s_lbar[pref ? 2 : 0], pref ? 0u : (bulkA ? 1u : 0u));
            if (!got && lane == 0) {
                s_fail = 1;
                set_status(a.status, EAGLE_ERR_TIMEOUT);
                atomicExch(a.fail_tag, a.gen);
            }
            read_chunks(xp, s_rows + (pref ? 2 * kSliceMax : 0), cnt);
        } else {
            load_chunks(xp, rowL, cnt);
        }
        float mL;
        const float sL = exp_run(xp, mL, c);
        const float4 neutral = make_float4(-INFINITY, 0.f, -INFINITY, 0.f);
        post(ms_fold2(make_float4(mL, sL, -INFINITY, 0.f), c));
        if (warp == 0 && wait_posts()) send(ms_fold2(lane < kWarpsPrep ? s_wp[lane] : neutral, c));
        const int slot = xch & 1;
        const bool ok = wait_recv();
        const float4 mine = ok && lane < CL ? s_recv[slot][lane] : neutral;  // lane r < CL: rank r's record
        const float4 gl = ms_fold2(mine, c);
        const float l2 = gl.y > 0.f ? log2f(gl.y) : 0.f;
        if (warp == 1) {  // the draw's owner from the per-rank probability totals
            const float tr = mine.x == -INFINITY ? 0.f : mine.y * fast_exp2((mine.x - gl.x) * c - l2);
            int own;
            uint64_t loc;
            decide_owner_warp<CL>(lane < CL ? to_fx(tr) : 0ull, uA, own, loc);
            if (lane == 0) {
                s_own[0] = own;
                s_local[0] = loc;
            }
        }
        const float fL = mL == -INFINITY ? 0.f : fast_exp2(fmaf(mL - gl.x, c, -l2));
#pragma unroll
        for (int j = 0; j < kE; ++j) xp[j] *= fL;
    }
    // every record this CTA sends has been sent: the closing cluster barrier can start
    cluster_arrive();
    __syncthreads();  // the draw decisions are visible

    // ---- the final draw, over xp: node A's probabilities or residual (every child rejected), or
    // the accepted leaf's probabilities
    if (!accepted || spec >= 0) {
        const int owner = s_own[0];
        const int node = spec >= 0 ? spec : nodeA;
        int32_t *slot = a.bonus_mode ? a.out_tokens + size_t(b) * (a.D + 1) + (breq >> 8) : nullptr;
        if (owner < 0) {
            if (rank == 0 && tid == 0 && !s_fail) {  // no positive mass
                a.final_tok[size_t(b) * n + node] = 0;
                if (slot) *slot = 0;
            }
        } else if (rank == owner) {
            const int found = draw_in_slice(xp, s_local[0], s_draw);
            if (found >= 0 && !s_fail) {
                a.final_tok[size_t(b) * n + node] = lo + found;
                if (slot) *slot = lo + found;
            }
        }
    }
    // a bonus draw that could not be made: nothing of this sequence is committed
    if (a.bonus_mode && tid == 0 && *reinterpret_cast<volatile int *>(&s_fail)) a.out_len[b] = 0;
    // an unused prefetch has landed before the shared memory is released (bounded)
    if (s_pre >= 0 && spec != s_pre) mbar_warp_wait_bounded(&s_lbar[2], 0);
    cluster_wait();  // no peer leaves while records it sent may still be landing here, or vice versa
}

__global__ void __launch_bounds__(64) verify_walk_kernel(VerifyArgs a) {
    pdl_wait();
    pdl_launch_next();
    __shared__ int s_tok[64], s_row[64], s_fin[64], s_next[64], s_kids[64];
    __shared__ int s_bad;
    const int b = blockIdx.x, tid = threadIdx.x;
    const int n = a.n, D = a.D;
    int t = 0, p = -1;
    float u = 0.f;
    NodeStat cs = {};
    if (tid < n) {  // every load of the node's own inputs at once
        const size_t o = size_t(b) * n + tid;
        t = a.tokens[o];
        p = a.parents[o];
        u = a.uniforms[o];
        s_row[tid] = a.node_row[o];
        s_fin[tid] = a.final_tok[o];
        if (!a.greedy && tid > 0) cs = a.stat[o];
    }
    s_next[tid] = n;  // no accepted child (yet)
    s_kids[tid] = 0;
    if (tid == 0) s_bad = 0;
    __syncthreads();
    bool bad = false;
    if (tid < n) {
        s_tok[tid] = t;
        bad = t < 0 || t >= a.V;
        bad |= tid == 0 ? p != -1 : (p < 0 || p >= tid);
    }
    if (bad) s_bad = 1;
    if (!bad && tid > 0 && tid < n) s_kids[p] = 1;
    __syncthreads();
    if (!a.greedy && tid > 0 && tid < n && !s_bad && (s_row[p] < 0 || s_row[p] >= a.R)) s_bad = 1;
    __syncthreads();
    // every child's accept test: the ratio (p0 / q0 - c_j)+ / S_j at its token after j rejected
    // siblings (p0 / q0 itself for j = 0, as p_j / q = (p0 - c_j q)+ / (S_j q)) against its
    // uniform.  A chain that stopped at its first accepted child was tested by the prep (the
    // verdict is in sj); with every ratio wanted, each child's is computed here, one thread per
    // node, in double precision from its parent's row statistics.
    // a prep CTA of this call whose wait ran out left its statistics unwritten: commit nothing
    const bool call_failed = *reinterpret_cast<volatile const int32_t *>(a.fail_tag) == a.gen;
    const bool ok = !s_bad && !call_failed;
    bool acc = false;
    if (tid < n) {
        float r = NAN;
        if (!a.greedy && ok && tid > 0 && !a.full_chain) {
            acc = (cs.sj >> kVerdictShift) == 2;
        } else if (!a.greedy && ok && tid > 0) {
            const NodeStat ps = a.stat[size_t(b) * n + p];
            const double x = a.target[(size_t(b) * n + p) * a.V + t];
            const double yv = a.draft[(size_t(b) * a.R + s_row[p]) * a.V + t];
            const double rr = exp(((x - double(ps.mp)) * a.inv_td - double(ps.lnsp)) -
                                  ((yv - double(ps.mq)) * a.inv_td - double(ps.lnsq)));
            const uint64_t sj = cs.sj & kSjMask;
            const double sjd = double(sj) * kFxInv;
            r = cs.cj == 0 ? float(rr) : (sjd > 0.0 ? float(fmax(rr - double(cs.cj) * kFxInv, 0.0) / sjd) : INFINITY);
            acc = accept_fx(u, cs.cj, sj, ratio_fx(rr));
        } else if (a.greedy && ok && tid > 0) {
            acc = t == s_fin[p];
        }
        if (a.out_ratio) a.out_ratio[size_t(b) * n + tid] = r;
    }
    // each parent's first accepted child (children in index order)
    if (acc) atomicMin(&s_next[p], tid);
    __syncthreads();
    if (tid != 0) return;
    int32_t *ot = a.out_tokens + size_t(b) * (D + 1);
    int32_t *op = a.out_path + size_t(b) * D;
    for (int j = 0; j <= D; ++j) ot[j] = -1;
    for (int j = 0; j < D; ++j) op[j] = -1;
    a.bonus[b] = -1;
    if (!ok) {
        set_status(a.status, call_failed ? EAGLE_ERR_TIMEOUT : EAGLE_ERR_DEVICE_INPUT);
        a.out_len[b] = 0;
        return;
    }
    int node = 0, len = 0;
    for (;;) {
        const int next = s_next[node];
        if (next >= n || len >= D) {
            if (next < n) set_status(a.status, EAGLE_ERR_DEVICE_INPUT);  // tree deeper than D
            if (!a.greedy && !s_kids[node] && a.full_chain) {
                // a leaf with every ratio wanted: its draw from the target distribution is made by
                // the bonus launch, which also writes the token into this slot (otherwise the prep
                // drew it: the leaf's parent accepted it, or it is the root without children)
                a.bonus[b] = node | (len << 8);
                ++len;
            } else {
                ot[len++] = s_fin[node];
            }
            break;
        }
        ot[len] = s_tok[next];
        op[len] = next;
        ++len;
        node = next;
    }
    a.out_len[b] = len;
}

}  // namespace

size_t tree_verify_workspace_bytes(const eagle_verify_cfg &c) {
    const int n = c.keep + 1;
    return kWsHeader + align_up(size_t(c.batch) * n * sizeof(NodeStat), 256) +
           align_up(size_t(c.batch) * n * sizeof(int32_t), 256) + align_up(size_t(c.batch) * sizeof(int32_t), 256);
}

namespace {
template <int CL>
cudaError_t launch_prep(const VerifyArgs &a, int clusters, int batch, cudaStream_t stream) {
    static std::atomic<uint64_t> ready{0};
    const cudaError_t e = once_per_device(ready, [] {
        cudaError_t r = cudaFuncSetAttribute(verify_prep_kernel<CL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             int(kPrepSmem));
        if (r == cudaSuccess && CL > 8)
            r = cudaFuncSetAttribute(verify_prep_kernel<CL>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        return r;
    });
    if (e != cudaSuccess) return e;
    return launch_pdl(verify_prep_kernel<CL>, dim3(CL, batch, clusters), dim3(kPrepThreads), kPrepSmem, stream,
                      unsigned(CL), a);
}
}  // namespace

eagle_status tree_verify_launch(const eagle_verify_cfg &c, const float *target, const float *draft,
                                const int32_t *tokens, const int32_t *parents, const int32_t *node_row,
                                const float *uniforms, int32_t *out_tokens, int32_t *out_len, int32_t *out_path,
                                float *out_ratio, void *ws, cudaStream_t stream) {
    unsigned char *w = static_cast<unsigned char *>(ws);
    const int n = c.keep + 1;
    VerifyArgs a;
    a.target = target;
    a.draft = draft;
    a.tokens = tokens;
    a.parents = parents;
    a.node_row = node_row;
    a.uniforms = uniforms;
    static std::atomic<uint32_t> call_gen{0};
    uint32_t gen = call_gen.fetch_add(1, std::memory_order_relaxed) + 1;
    if (gen == 0u) gen = call_gen.fetch_add(1, std::memory_order_relaxed) + 1;  // 0: a fresh workspace's tag
    a.status = reinterpret_cast<int32_t *>(w);
    a.fail_tag = reinterpret_cast<int32_t *>(w + 16);
    a.gen = int32_t(gen);
    a.stat = reinterpret_cast<NodeStat *>(w + kWsHeader);
    a.final_tok = reinterpret_cast<int32_t *>(w + kWsHeader + align_up(size_t(c.batch) * n * sizeof(NodeStat), 256));
    a.bonus = reinterpret_cast<int32_t *>(reinterpret_cast<unsigned char *>(a.final_tok) +
                                          align_up(size_t(c.batch) * n * sizeof(int32_t), 256));
    a.bonus_mode = 0;
    a.full_chain = out_ratio != nullptr;
    a.out_ratio = out_ratio;
    a.out_tokens = out_tokens;
    a.out_len = out_len;
    a.out_path = out_path;
    a.B = c.batch;
    a.n = n;
    a.V = c.vocab;
    a.R = 1 + (c.depth - 1) * c.topk;
    a.D = c.depth;
    a.greedy = c.temperature <= 0.f;
    a.inv_t = a.greedy ? 1.f : 1.f / c.temperature;
    a.inv_td = a.greedy ? 1.0 : 1.0 / double(c.temperature);
    a.c = kLog2e * a.inv_t;
    const int per_cta = kPrepThreads * kE;
    const int cl = c.vocab <= 8 * per_cta ? 8 : 16;
    int slice = (c.vocab + cl - 1) / cl;
    slice = (slice + 3) & ~3;
    a.slice = slice;
    // sampling: one per node at most (the working nodes take the first clusters, the rest exit);
    // grid (CL, B, clusters), so that every sequence's working clusters come before idle ones
    const int clusters = a.greedy ? (n + 1) / 2 : n;
    cudaError_t e = cl == 8 ? launch_prep<8>(a, clusters, c.batch, stream) : launch_prep<16>(a, clusters, c.batch, stream);
    if (e != cudaSuccess) return EAGLE_ERR_CUDA;
    note_launch();
    if (launch_pdl(verify_walk_kernel, dim3(c.batch), dim3(64), 0, stream, 1u, a) != cudaSuccess) return EAGLE_ERR_CUDA;
    note_launch();
    if (!a.greedy && a.full_chain) {  // the bonus token of a walk that ended at a leaf
        a.bonus_mode = 1;
        e = cl == 8 ? launch_prep<8>(a, 1, c.batch, stream) : launch_prep<16>(a, 1, c.batch, stream);
        if (e != cudaSuccess) return EAGLE_ERR_CUDA;
        note_launch();
    }
    return cudaPeekAtLastError() == cudaSuccess ? EAGLE_OK : EAGLE_ERR_CUDA;
}

size_t verify_max_vocab() { return size_t(16) * kPrepThreads * kE; }

}  // namespace eagle
