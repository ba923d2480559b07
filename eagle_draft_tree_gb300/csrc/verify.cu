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
//                       with children, or per pair of leaves.  Each thread holds 32 consecutive
//                       tokens of a row in registers: the node's target and draft rows, or the
//                       two leaves' target rows.  Log-sum-exp, the S_j passes and the inverse-CDF
//                       scan are register loops; each CTA reduces a pass to one record and pushes
//                       it to every peer (st.async completing on the receiver's mbarrier), so a
//                       pass costs one point-to-point exchange, not a cluster-wide barrier, and the
//                       final draw reuses the records of the last exchange.  Per-node statistics
//                       (row maxima, log normalisers, each child's c_j and S_j) go to the workspace.
//   verify_walk_kernel  one CTA per sequence: validates the tree, computes every child's accept
//                       ratio in double precision (one thread per node), and walks the tree.
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
constexpr int kE = 32;  // tokens per thread and row
constexpr int kMaxNodes = 64;

// Per-node statistics the prep kernel leaves for the walk.  Row statistics (mp, mq, lnsp, lnsq)
// belong to a node with children; (cj, sj) to a node as a child: its parent's rejection chain
// state when this child is tested.
struct NodeStat {
    double lnsp, lnsq;  // ln of the normaliser sum_t exp((x_t - max) / T), target and draft rows
    double cj, sj;      // c_j, S_j of the parent's chain at this child's sibling index
    float mp, mq;       // row maxima (logit units)
    int32_t pad[2];
};
static_assert(sizeof(NodeStat) == 48, "NodeStat layout");

struct VerifyArgs {
    const float *target;    // [B][n][V]
    const float *draft;     // [B][R][V]
    const int32_t *tokens;  // [B][n]
    const int32_t *parents;
    const int32_t *node_row;
    const float *uniforms;  // [B][n]
    NodeStat *stat;         // [B][n] workspace
    int32_t *final_tok;     // [B][n] workspace
    float *out_ratio;       // optional
    int32_t *out_tokens, *out_len, *out_path;
    int32_t *status;
    int B, n, V, R, D, slice;
    float inv_t;    // 1/T (T > 0)
    double inv_td;  // 1/T in double
    float c;        // log2(e)/T
    int greedy;
};

__device__ __forceinline__ void ms_merge(float &m, float &s, float mo, float so, float c) {
    const float M = fmaxf(m, mo);
    if (M == -INFINITY) return;
    const float x = (m == -INFINITY) ? 0.f : s * exp2f((m - M) * c);
    const float y = (mo == -INFINITY) ? 0.f : so * exp2f((mo - M) * c);
    m = M;
    s = x + y;
}

// Load this thread's kE consecutive values of a row slice into registers (-inf past the end).
__device__ __forceinline__ void load_run(float (&v)[kE], const float *src, int t0, int cnt, bool vec) {
    if (vec) {
#pragma unroll
        for (int j = 0; j < kE / 4; ++j) {
            const int idx = t0 + 4 * j;
            const float4 w = idx < cnt ? __ldg(reinterpret_cast<const float4 *>(src + idx))
                                       : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
            v[4 * j] = w.x;
            v[4 * j + 1] = w.y;
            v[4 * j + 2] = w.z;
            v[4 * j + 3] = w.w;
        }
    } else {
#pragma unroll
        for (int j = 0; j < kE; ++j) v[j] = t0 + j < cnt ? __ldg(src + t0 + j) : -INFINITY;
    }
}

// In place: v <- 2^((v - m) c) against the run's max m (0 past the end); returns the sum.
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
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }
__device__ __forceinline__ float4 shfl4(float4 v, int src) {
    return make_float4(__shfl_sync(0xffffffffu, v.x, src), __shfl_sync(0xffffffffu, v.y, src),
                       __shfl_sync(0xffffffffu, v.z, src), __shfl_sync(0xffffffffu, v.w, src));
}
// Warp-wide deterministic merges of (max, scaled sum) pairs held as (x, y) and (z, w).
__device__ __forceinline__ float4 warp_ms_merge(float4 v, float c) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        ms_merge(v.x, v.y, __shfl_xor_sync(0xffffffffu, v.x, off), __shfl_xor_sync(0xffffffffu, v.y, off), c);
        ms_merge(v.z, v.w, __shfl_xor_sync(0xffffffffu, v.z, off), __shfl_xor_sync(0xffffffffu, v.w, off), c);
    }
    return v;
}
__device__ __forceinline__ FF ff_from(float hi, float lo) {
    FF r;
    r.hi = hi;
    r.lo = lo;
    return r;
}

// Owner search of a final draw from the CL per-rank weight totals (float-float, in rank order):
// the owner rank holds the first CDF step above u * total (running sums over the ranks are
// monotone); if rounding leaves the target at or above the total, the draw clamps to the last rank
// with mass.  Writes owner (-1: no mass at all), clamp and the target relative to the owner's start.
template <int CL>
__device__ __forceinline__ void decide_owner(const FF (&tot)[CL], float u, int &owner, int &clamp, float &local) {
    FF total;
#pragma unroll
    for (int r = 0; r < CL; ++r) total = ff_add(total, tot[r]);
    // target = u * total in float-float (u * hi exactly as hi + lo via FMA)
    const float th = u * total.hi;
    FF target = ff_from(th, fmaf(u, total.hi, -th) + u * total.lo);
    FF base;
    int own = -1, last = -1;
    FF rbase;
#pragma unroll
    for (int r = 0; r < CL; ++r) {
        const FF next = ff_add(base, tot[r]);
        const FF gap = ff_add(next, ff_from(-target.hi, -target.lo));  // next - target
        if (own < 0 && (gap.hi > 0.f || (gap.hi == 0.f && gap.lo > 0.f))) {
            own = r;
            rbase = base;
        }
        base = next;
        if (tot[r].hi > 0.f) last = r;
    }
    clamp = own < 0 ? 1 : 0;
    owner = own < 0 ? last : own;
    const FF lt = ff_add(target, ff_from(-rbase.hi, -rbase.lo));
    local = lt.hi + lt.lo;
}

// Final draw at a node over this CTA's slice: w holds the weights (probabilities or residuals) of
// this thread's run; the owner CTA finds the token whose cumulative weight first exceeds `local`
// (ascending ids).  CTA-uniform call; uses s_wp, s_claim, s_last.
__device__ __forceinline__ int draw_in_slice(const float (&w)[kE], float local, bool clamp, float4 *s_wp,
                                             int *s_claim, int *s_last) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int t0 = tid * kE;
    float tsum = 0.f;
    int tlast = -1;
#pragma unroll
    for (int e = 0; e < kE; ++e) {
        tsum += w[e];
        if (w[e] > 0.f) tlast = t0 + e;
    }
    float incl = tsum;  // inclusive scan of the run sums within the warp
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
    }
    int wl = tlast;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) wl = max(wl, __shfl_xor_sync(0xffffffffu, wl, off));
    __syncthreads();  // s_wp free
    if (lane == 31) s_wp[warp].x = incl;
    if (tid == 0) {
        *s_claim = kPrepThreads;
        *s_last = -1;
    }
    __syncthreads();
    if (lane == 0) atomicMax(s_last, wl);
    float wbase = 0.f;
    for (int w2 = 0; w2 < warp; ++w2) wbase += s_wp[w2].x;  // this CTA's earlier warps
    const float excl = wbase + incl - tsum;
    // the first thread whose run ends above the local target owns the step
    if (!clamp && tsum > 0.f && excl + tsum > local) atomicMin(s_claim, tid);
    __syncthreads();
    int found = -1;
    if (!clamp && tid == *s_claim) {
        float acc = excl;
        found = tlast;
        bool done = false;
#pragma unroll
        for (int e = 0; e < kE; ++e) {
            acc += w[e];
            if (!done && w[e] > 0.f && acc > local) {
                found = t0 + e;
                done = true;
            }
        }
    } else if (tid == 0 && (clamp || *s_claim == kPrepThreads)) {
        found = max(*s_last, 0);
    }
    return found;  // >= 0 in exactly one thread of the CTA
}

template <int CL>
__global__ void __launch_bounds__(kPrepThreads, 1) verify_prep_kernel(VerifyArgs a) {
    __shared__ float4 s_wp[kWarpsPrep];  // per-warp partials of the current pass
    __shared__ float4 s_recv[2][CL];     // the cluster's records of an exchange, by parity
    __shared__ __align__(8) uint64_t s_rbar[2];
    __shared__ int s_kid[kMaxNodes];     // children of the node (sampling), ascending
    __shared__ int s_nk, s_claim, s_last, s_fail, s_second;
    __shared__ float s_bc[8];  // broadcasts: maxima, log2 normalisers, next c, c_J
    __shared__ int s_own[2], s_clamp[2];
    __shared__ float s_local[2];

    cg::cluster_group cluster = cg::this_cluster();
    const int rank = int(cluster.block_rank());
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n = a.n, V = a.V, b = blockIdx.z;
    const int lo = rank * a.slice;
    const int hi = min(V, lo + a.slice);
    const int cnt = hi > lo ? hi - lo : 0;
    const int t0 = tid * kE;  // this thread's run, relative to lo
    const int32_t *par = a.parents + size_t(b) * n;

    // ---- work of this cluster.  Greedy: nodes 2y and 2y + 1 (argmax of two target rows).
    // Sampling: node y when it has children; when y is a leaf, the cluster of an even-ranked leaf
    // (in ascending order among the leaves) takes y and the next leaf, an odd-ranked leaf's exits.
    const int y = blockIdx.y;
    const int nodeA = a.greedy ? 2 * y : y;
    const float *rowA = a.target + (size_t(b) * n + nodeA) * V;
    const bool vecA = ((V & 3) == 0) && ((lo & 3) == 0) && ((reinterpret_cast<uintptr_t>(rowA) & 15) == 0);
    float xp[kE], xq[kE];
    load_run(xp, rowA + lo, t0, cnt, vecA);  // node y's target row is needed in every case
    if (warp == 0) {
        // every node's "has children" bit, and the children of node y, from the <= 64 parents
        const int p0 = lane < n ? par[lane] : -1;
        const int p1 = lane + 32 < n ? par[lane + 32] : -1;
        uint64_t mine = 0;
        if (lane > 0 && p0 >= 0 && p0 < n) mine |= 1ull << p0;
        if (p1 >= 0 && p1 < n) mine |= 1ull << p1;
        const unsigned ml = __reduce_or_sync(0xffffffffu, uint32_t(mine));
        const unsigned mh = __reduce_or_sync(0xffffffffu, uint32_t(mine >> 32));
        const uint64_t internal = (uint64_t(mh) << 32) | ml;
        const uint64_t all = n >= 64 ? ~0ull : ((1ull << n) - 1ull);
        const uint64_t leaves = all & ~internal;
        const bool k0 = lane > 0 && p0 == y, k1 = p1 == y;
        const unsigned b0 = __ballot_sync(0xffffffffu, k0), b1 = __ballot_sync(0xffffffffu, k1);
        if (k0) s_kid[__popc(b0 & ((1u << lane) - 1u))] = lane;
        if (k1) s_kid[__popc(b0) + __popc(b1 & ((1u << lane) - 1u))] = lane + 32;
        if (lane == 0) {
            s_nk = __popc(b0) + __popc(b1);
            int second = -1;  // sampling: the leaf paired with leaf y (-2: this cluster has no work)
            if (!a.greedy && ((leaves >> y) & 1ull)) {
                const int lrank = __popcll(leaves & ((1ull << y) - 1ull));
                if (lrank & 1) {
                    second = -2;
                } else {
                    const uint64_t after = leaves & ~((2ull << y) - 1ull);
                    second = after ? __ffsll(static_cast<long long>(after)) - 1 : -1;
                }
            }
            if (a.greedy) second = 2 * y + 1 < n ? 2 * y + 1 : -1;
            s_second = second;
            s_fail = 0;
        }
    }
    __syncthreads();
    const int second = s_second;
    if (second == -2) return;  // uniform for the cluster: no barrier has been touched yet
    const int J = a.greedy ? 0 : s_nk;
    const bool pair = J == 0;  // a leaf pair (sampling) or a node pair (greedy)
    const int nodeB = pair ? second : -1;
    const int rowq = J > 0 ? a.node_row[size_t(b) * n + nodeA] : -1;
    const bool has_q = J > 0 && rowq >= 0 && rowq < a.R;
    if (tid == 0) {
        mbar_init(&s_rbar[0], 1);
        mbar_init(&s_rbar[1], 1);
        fence_barrier_init();
    }
    cluster_arrive();  // peers may push records only after these barriers exist (wait below)
    const float *rowB = nullptr;
    if (nodeB >= 0) rowB = a.target + (size_t(b) * n + nodeB) * V;
    else if (has_q) rowB = a.draft + (size_t(b) * a.R + rowq) * V;
    if (rowB) load_run(xq, rowB + lo, t0, cnt, vecA && (reinterpret_cast<uintptr_t>(rowB) & 15) == 0);
    // every final draw uses the sequence's first uniform (the root's, which no accept test uses)
    const float uA = __ldg(a.uniforms + size_t(b) * n), uB = uA;
    cluster_wait();

    // One exchange, executed by warp 0 (all lanes): rec (valid in lane 0) goes to every CTA; on
    // return lanes r < CL hold rank r's record.  A receive that times out marks the CTA failed
    // (its results are then not written).
    int xch = 0;
    auto exchange = [&](float4 rec, float4 neutral) -> float4 {
        const int slot = xch & 1;
        rec = shfl4(rec, 0);
        if (lane == 0) mbar_expect_tx(&s_rbar[slot], CL * 16);
        __syncwarp();
        if (lane < CL)
            st_async_v4(mapa_u32(static_cast<uint32_t>(__cvta_generic_to_shared(&s_recv[slot][rank])), lane), rec,
                        mapa_u32(static_cast<uint32_t>(__cvta_generic_to_shared(&s_rbar[slot])), lane));
        bool got = false;
        for (uint32_t it = 0; it < (1u << 22) && !got; ++it)
            got = __all_sync(0xffffffffu, mbar_try_wait(&s_rbar[slot], (xch >> 1) & 1));
        ++xch;
        if (!got) {
            if (lane == 0) {
                s_fail = 1;
                set_status(a.status, EAGLE_ERR_TIMEOUT);
            }
            return neutral;
        }
        return lane < CL ? s_recv[slot][lane] : neutral;
    };

    if (a.greedy) {
        // argmax of the two target rows (ties to the lower id): thread, warp, CTA, cluster
        uint64_t ba = 0, bb = 0;
#pragma unroll
        for (int j = 0; j < kE; ++j) {
            const uint32_t t = uint32_t(lo + t0 + j);
            const uint64_t ka = xp[j] == -INFINITY ? 0ull : topk_key(xp[j], t);
            ba = ka > ba ? ka : ba;
            if (nodeB >= 0) {
                const uint64_t kb = xq[j] == -INFINITY ? 0ull : topk_key(xq[j], t);
                bb = kb > bb ? kb : bb;
            }
        }
        ba = warp_max_u64(ba);
        bb = warp_max_u64(bb);
        if (lane == 0)
            s_wp[warp] = make_float4(__uint_as_float(uint32_t(ba)), __uint_as_float(uint32_t(ba >> 32)),
                                     __uint_as_float(uint32_t(bb)), __uint_as_float(uint32_t(bb >> 32)));
        __syncthreads();
        if (warp == 0) {
            uint64_t ga = 0, gb = 0;
            if (lane < kWarpsPrep) {
                const float4 v = s_wp[lane];
                ga = (uint64_t(__float_as_uint(v.y)) << 32) | __float_as_uint(v.x);
                gb = (uint64_t(__float_as_uint(v.w)) << 32) | __float_as_uint(v.z);
            }
            ga = warp_max_u64(ga);
            gb = warp_max_u64(gb);
            const float4 v = exchange(make_float4(__uint_as_float(uint32_t(ga)), __uint_as_float(uint32_t(ga >> 32)),
                                                  __uint_as_float(uint32_t(gb)), __uint_as_float(uint32_t(gb >> 32))),
                                      make_float4(0.f, 0.f, 0.f, 0.f));
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

    const float c = a.c;
    // ---- row statistics of both held rows.  Values become 2^((x - m) c) against the run's max
    // m, so the probabilities later cost one multiply each (no second exponential).
    float mA, mB = -INFINITY, sB = 0.f;
    const float sA = exp_run(xp, mA, c);
    if (rowB) sB = exp_run(xq, mB, c);
    {
        const float4 wv = warp_ms_merge(make_float4(mA, sA, mB, sB), c);
        if (lane == 0) s_wp[warp] = wv;
        __syncthreads();
        if (warp == 0) {
            const float4 neutral = make_float4(-INFINITY, 0.f, -INFINITY, 0.f);
            const float4 cta = warp_ms_merge(lane < kWarpsPrep ? s_wp[lane] : neutral, c);
            const float4 mine = exchange(cta, neutral);  // lane r < CL: rank r's record
            const float4 g = warp_ms_merge(mine, c);
            const float l2A = g.y > 0.f ? log2f(g.y) : 0.f;
            const float l2B = g.w > 0.f ? log2f(g.w) : 0.f;
            // per-rank probability totals of both rows (the final draws' weights, for leaves)
            const float trA = lane < CL && mine.x != -INFINITY ? mine.y * exp2f((mine.x - g.x) * c - l2A) : 0.f;
            const float trB = lane < CL && mine.z != -INFINITY ? mine.w * exp2f((mine.z - g.z) * c - l2B) : 0.f;
            FF tA[CL], tB[CL];
#pragma unroll
            for (int r = 0; r < CL; ++r) {
                tA[r] = ff_from(__shfl_sync(0xffffffffu, trA, r), 0.f);
                tB[r] = ff_from(__shfl_sync(0xffffffffu, trB, r), 0.f);
            }
            if (lane == 0) {
                s_bc[0] = g.x;
                s_bc[1] = l2A;
                s_bc[2] = g.z;
                s_bc[3] = l2B;
                s_bc[4] = 1.f;  // c_1 = c_0 + S_0
                s_bc[5] = 0.f;
                s_own[0] = s_own[1] = -1;
                s_clamp[0] = s_clamp[1] = 0;
                if (!has_q) decide_owner<CL>(tA, uA, s_own[0], s_clamp[0], s_local[0]);
                if (nodeB >= 0) decide_owner<CL>(tB, uB, s_own[1], s_clamp[1], s_local[1]);
                if (rank == 0 && J > 0 && !s_fail) {
                    NodeStat *st = a.stat + size_t(b) * n + nodeA;
                    st->mp = g.x;
                    st->mq = g.z;
                    st->lnsp = log_fast(double(g.y));
                    st->lnsq = has_q && g.w > 0.f ? log_fast(double(g.w)) : 0.0;
                }
            }
        }
        __syncthreads();
    }
    {
        // probabilities: p = 2^((x - m) c) * 2^((m - M) c - log2 S), one exponential per run
        const float fA = mA == -INFINITY ? 0.f : fast_exp2(fmaf(mA - s_bc[0], c, -s_bc[1]));
#pragma unroll
        for (int j = 0; j < kE; ++j) xp[j] *= fA;
        if (rowB) {
            const float fB = mB == -INFINITY ? 0.f : fast_exp2(fmaf(mB - s_bc[2], c, -s_bc[3]));
#pragma unroll
            for (int j = 0; j < kE; ++j) xq[j] *= fB;
        }
    }

    // ---- rejection chain of a node with children: c_0 = 0, S_0 = 1; after rejecting child j:
    // c_{j+1} = c_j + S_j and S_{j+1} = sum (p0 - c_{j+1} q)+ (a zero sum keeps the previous
    // distribution).  Lane 0 of warp 0 carries c_j, S_j in float-float; every thread sees c_{j+1}
    // rounded to float.  When the last pass moves c, its per-rank sums are exactly the final
    // draw's per-rank weights.
    FF cj = ff_from(0.f, 0.f), Sj = ff_from(1.f, 0.f);  // meaningful in lane 0 of warp 0
    bool decided = !has_q;
    for (int j = 0; j < J && has_q; ++j) {
        if (rank == 0 && warp == 0 && lane == 0 && !s_fail) {  // the child tested at step j
            NodeStat *st = a.stat + size_t(b) * n + s_kid[j];
            st->cj = double(cj.hi) + double(cj.lo);
            st->sj = double(Sj.hi) + double(Sj.lo);
        }
        const float cnf = s_bc[4];
        float part = 0.f;
#pragma unroll
        for (int e = 0; e < kE; ++e) part += fmaxf(fmaf(-cnf, xq[e], xp[e]), 0.f);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
        if (lane == 0) s_wp[warp].x = part;
        __syncthreads();
        if (warp == 0) {
            FF t = ff_from(lane < kWarpsPrep ? s_wp[lane].x : 0.f, 0.f);
            t = ff_warp_sum(t);
            const float4 mine = exchange(make_float4(t.hi, t.lo, 0.f, 0.f), make_float4(0.f, 0.f, 0.f, 0.f));
            const FF g = ff_warp_sum(ff_from(mine.x, mine.y));
            FF tot[CL];
#pragma unroll
            for (int r = 0; r < CL; ++r) tot[r] = ff_from(__shfl_sync(0xffffffffu, mine.x, r), __shfl_sync(0xffffffffu, mine.y, r));
            const bool moved = g.hi > 0.f;
            if (moved) {
                cj = ff_add(cj, Sj);
                Sj = g;
            }
            if (lane == 0) {
                const FF nx = ff_add(cj, Sj);
                s_bc[4] = nx.hi + nx.lo;
                s_bc[5] = cj.hi + cj.lo;
                if (j == J - 1 && moved) decide_owner<CL>(tot, uA, s_own[0], s_clamp[0], s_local[0]);
            }
            decided = j == J - 1 && moved;
        }
        __syncthreads();
    }
    const float cjf = s_bc[5];
    if (has_q) {
        decided = __shfl_sync(0xffffffffu, decided ? 1 : 0, 0) != 0;  // warp 0's verdict ...
        if (warp == 0 && lane == 0) s_nk = decided ? 1 : 0;             // ... for the whole CTA
        __syncthreads();
        decided = s_nk != 0;
    }
    // residual weights of a node with children: (p0 - c_J q)+
    if (has_q) {
#pragma unroll
        for (int e = 0; e < kE; ++e) xp[e] = fmaxf(fmaf(-cjf, xq[e], xp[e]), 0.f);
    }
    if (has_q && !decided) {
        // the last pass left c unchanged: one more exchange for the residual's per-rank weights
        float part = 0.f;
#pragma unroll
        for (int e = 0; e < kE; ++e) part += xp[e];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
        if (lane == 0) s_wp[warp].x = part;
        __syncthreads();
        if (warp == 0) {
            FF t = ff_from(lane < kWarpsPrep ? s_wp[lane].x : 0.f, 0.f);
            t = ff_warp_sum(t);
            const float4 mine = exchange(make_float4(t.hi, t.lo, 0.f, 0.f), make_float4(0.f, 0.f, 0.f, 0.f));
            FF tot[CL];
#pragma unroll
            for (int r = 0; r < CL; ++r) tot[r] = ff_from(__shfl_sync(0xffffffffu, mine.x, r), __shfl_sync(0xffffffffu, mine.y, r));
            if (lane == 0) decide_owner<CL>(tot, uA, s_own[0], s_clamp[0], s_local[0]);
        }
        __syncthreads();
    }
    // every record this CTA sends has been sent: the closing cluster barrier can start
    cluster_arrive();

    // ---- final draws: node A over xp (probabilities or residual), leaf B over xq
    for (int k = 0; k < (nodeB >= 0 ? 2 : 1); ++k) {
        const int owner = s_own[k];
        const int node = k ? nodeB : nodeA;
        if (owner < 0) {
            if (rank == 0 && tid == 0 && !s_fail) a.final_tok[size_t(b) * n + node] = 0;  // no positive mass
        } else if (rank == owner) {
            const int found = draw_in_slice(k ? xq : xp, s_local[k], s_clamp[k] != 0, s_wp, &s_claim, &s_last);
            if (found >= 0 && !s_fail) a.final_tok[size_t(b) * n + node] = lo + found;
        }
    }
    cluster_wait();  // no peer leaves while records it sent may still be landing here, or vice versa
}

__global__ void __launch_bounds__(64) verify_walk_kernel(VerifyArgs a) {
    __shared__ int s_tok[64], s_par[64], s_row[64], s_fin[64];
    __shared__ float s_u[64], s_ratio[64];
    __shared__ int s_bad;
    const int b = blockIdx.x, tid = threadIdx.x;
    const int n = a.n, D = a.D;
    if (tid == 0) s_bad = 0;
    __syncthreads();
    if (tid < n) {
        const size_t o = size_t(b) * n + tid;
        const int t = a.tokens[o], p = a.parents[o];
        s_tok[tid] = t;
        s_par[tid] = p;
        s_row[tid] = a.node_row[o];
        s_fin[tid] = a.final_tok[o];
        s_u[tid] = a.uniforms[o];
        bool bad = t < 0 || t >= a.V;
        bad |= tid == 0 ? p != -1 : (p < 0 || p >= tid);
        if (bad) s_bad = 1;
    }
    __syncthreads();
    if (!a.greedy && tid > 0 && tid < n && !s_bad) {
        const int p = s_par[tid];
        if (s_row[p] < 0 || s_row[p] >= a.R) s_bad = 1;
    }
    __syncthreads();
    // accept ratio of every child (one thread per node, double precision):
    //   p0 = exp((x - Mp)/T - ln Sp), q0 = exp((y - Mq)/T - ln Sq) at the child's token, then
    //   (p0 - c_j q0)+ / (S_j q0) for the child tested after j rejected siblings (p0 / q0 first)
    if (tid < n) {
        float r = NAN;
        if (!a.greedy && !s_bad && tid > 0) {
            const int p = s_par[tid], t = s_tok[tid];
            int sib = 0;
            for (int j = p + 1; j < tid; ++j) sib += s_par[j] == p;
            const NodeStat ps = a.stat[size_t(b) * n + p];
            const NodeStat cs = a.stat[size_t(b) * n + tid];
            const double x = a.target[(size_t(b) * n + p) * a.V + t];
            const double yv = a.draft[(size_t(b) * a.R + s_row[p]) * a.V + t];
            const double p0 = exp((x - double(ps.mp)) * a.inv_td - ps.lnsp);
            const double q0 = exp((yv - double(ps.mq)) * a.inv_td - ps.lnsq);
            const double num = sib == 0 ? p0 : fmax(p0 - cs.cj * q0, 0.0);
            const double den = cs.sj * q0;
            r = den > 0.0 ? float(num / den) : INFINITY;
        }
        s_ratio[tid] = r;
        if (a.out_ratio) a.out_ratio[size_t(b) * n + tid] = r;
    }
    __syncthreads();
    int32_t *ot = a.out_tokens + size_t(b) * (D + 1);
    int32_t *op = a.out_path + size_t(b) * D;
    if (tid != 0) return;
    for (int j = 0; j <= D; ++j) ot[j] = -1;
    for (int j = 0; j < D; ++j) op[j] = -1;
    if (s_bad) {
        set_status(a.status, EAGLE_ERR_DEVICE_INPUT);
        a.out_len[b] = 0;
        return;
    }
    int node = 0, len = 0;
    for (;;) {
        int next = -1;
        if (a.greedy) {
            const int g = s_fin[node];
            for (int j = node + 1; j < n; ++j)
                if (s_par[j] == node && s_tok[j] == g) {
                    next = j;
                    break;
                }
        } else {
            for (int j = node + 1; j < n; ++j)
                if (s_par[j] == node && s_u[j] < s_ratio[j]) {
                    next = j;
                    break;
                }
        }
        if (next < 0 || len >= D) {
            if (next >= 0) set_status(a.status, EAGLE_ERR_DEVICE_INPUT);  // tree deeper than D
            ot[len++] = s_fin[node];
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
           align_up(size_t(c.batch) * n * sizeof(int32_t), 256);
}

namespace {
template <int CL>
cudaError_t launch_prep(const VerifyArgs &a, int clusters, int batch, cudaStream_t stream) {
    static bool attr = false;
    if (!attr && CL > 8) {
        cudaError_t e = cudaFuncSetAttribute(verify_prep_kernel<CL>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
    attr = true;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(CL, clusters, batch);
    cfg.blockDim = dim3(kPrepThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = CL;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, verify_prep_kernel<CL>, a);
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
    a.status = reinterpret_cast<int32_t *>(w);
    a.stat = reinterpret_cast<NodeStat *>(w + kWsHeader);
    a.final_tok = reinterpret_cast<int32_t *>(w + kWsHeader + align_up(size_t(c.batch) * n * sizeof(NodeStat), 256));
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
    const int clusters = a.greedy ? (n + 1) / 2 : n;  // sampling: one per node, odd-ranked leaves idle
    const cudaError_t e = cl == 8 ? launch_prep<8>(a, clusters, c.batch, stream)
                                  : launch_prep<16>(a, clusters, c.batch, stream);
    if (e != cudaSuccess) return EAGLE_ERR_CUDA;
    note_launch();
    verify_walk_kernel<<<c.batch, 64, 0, stream>>>(a);
    note_launch();
    return cudaPeekAtLastError() == cudaSuccess ? EAGLE_OK : EAGLE_ERR_CUDA;
}

size_t verify_max_vocab() { return size_t(16) * kPrepThreads * kE; }

}  // namespace eagle
