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
//   verify_prep_kernel  one cluster of CL CTAs (8, or 16 for vocabularies above 131072) per
//                       (sequence, node).  Each thread holds 32 consecutive tokens of the node's
//                       target row (and of its draft row when the node has children) in
//                       registers; log-sum-exp, the S_j passes and the inverse-CDF scan are
//                       register loops whose partials are reduced across the cluster through
//                       distributed shared memory (one cluster barrier per pass).
//   verify_walk_kernel  one CTA per sequence: validates the tree and walks it.
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
constexpr int kMaxKids = 64;

struct VerifyArgs {
    const float *target;    // [B][n][V]
    const float *draft;     // [B][R][V]
    const int32_t *tokens;  // [B][n]
    const int32_t *parents;
    const int32_t *node_row;
    const float *uniforms;  // [B][n]
    float *ratio;           // [B][n] workspace
    int32_t *final_tok;     // [B][n] workspace
    float *out_ratio;       // optional
    int32_t *out_tokens, *out_len, *out_path;
    int32_t *status;
    int B, n, V, R, D, slice;
    float inv_t;    // 1/T (T > 0)
    double inv_td;  // 1/T in double (for the gathered per-child probabilities)
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

template <int CL>
__global__ void __launch_bounds__(kPrepThreads, 1) verify_prep_kernel(VerifyArgs a) {
    constexpr int kParts = CL * kWarpsPrep;
    // per-warp partials published to the cluster, double-buffered by pass parity
    __shared__ float4 s_part[2][kWarpsPrep];
    __shared__ double s_tot;
    __shared__ double s_rank[CL];  // final pass: per-rank totals
    __shared__ int s_rlast[CL];    // final pass: per-rank last positive index
    __shared__ int s_kids[kMaxKids];
    __shared__ float s_xk[kMaxKids], s_yk[kMaxKids];
    __shared__ double s_cj[kMaxKids + 1], s_Sj[kMaxKids + 1];
    __shared__ int s_nk, s_claim;
    __shared__ float s_M[2];
    __shared__ double s_lnS[2];

    cg::cluster_group cluster = cg::this_cluster();
    const int rank = int(cluster.block_rank());
    const int i = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n = a.n, V = a.V;
    const int lo = rank * a.slice;
    const int hi = min(V, lo + a.slice);
    const int cnt = hi > lo ? hi - lo : 0;
    const int t0 = tid * kE;  // this thread's run, relative to lo

    const int32_t *par = a.parents + size_t(b) * n;
    const int32_t *tok = a.tokens + size_t(b) * n;
    // children of node i, in ascending index (warp 0: ballots over the <= 64 nodes)
    if (warp == 0) {
        int nk = 0;
        for (int j0 = i + 1; j0 < n; j0 += 32) {
            const int j = j0 + lane;
            const bool kid = j < n && par[j] == i;
            const unsigned bal = __ballot_sync(0xffffffffu, kid);
            if (kid) s_kids[nk + __popc(bal & ((1u << lane) - 1u))] = j;
            nk += __popc(bal);
        }
        if (lane == 0) s_nk = nk;
    }
    __syncthreads();
    const int J = s_nk;
    const float *xrow = a.target + (size_t(b) * n + i) * V;
    const int row = J > 0 ? a.node_row[size_t(b) * n + i] : -1;
    const bool has_q = J > 0 && row >= 0 && row < a.R && !a.greedy;
    const float *yrow = has_q ? a.draft + (size_t(b) * a.R + row) * V : nullptr;
    const bool vec = ((V & 3) == 0) && ((lo & 3) == 0) && ((reinterpret_cast<uintptr_t>(xrow) & 15) == 0) &&
                     (!has_q || (reinterpret_cast<uintptr_t>(yrow) & 15) == 0);
    int pass = 0;

    // Publish each warp's float4 (from lane 0), make it visible to the cluster; warp 0 then
    // fetches all kParts partials (part = rank * kWarpsPrep + warp).
    auto publish = [&](float4 v) {
        const int slot = pass & 1;
        if (lane == 0) s_part[slot][warp] = v;
        cluster.sync();
        ++pass;
        return slot;
    };
    auto fetch = [&](int slot, int part) -> float4 {
        const float4 *remote = cluster.map_shared_rank(&s_part[slot][0], part / kWarpsPrep);
        return remote[part % kWarpsPrep];
    };

    float xp[kE], xq[kE];
    load_run(xp, xrow + lo, t0, cnt, vec);
    if (has_q) load_run(xq, yrow + lo, t0, cnt, vec);
    if (rank == 0 && tid < J) {  // the children's logits, for their accept ratios
        const int t = tok[s_kids[tid]];
        const bool ok = has_q && t >= 0 && t < V;
        s_xk[tid] = ok ? __ldg(xrow + t) : 0.f;
        s_yk[tid] = ok ? __ldg(yrow + t) : 0.f;
    }

    if (a.greedy) {
        // argmax of the target row (ties to the lower id): thread, warp, cluster
        uint64_t best = 0;
#pragma unroll
        for (int j = 0; j < kE; ++j) {
            const uint64_t key = xp[j] == -INFINITY ? 0ull : topk_key(xp[j], uint32_t(lo + t0 + j));
            best = key > best ? key : best;
        }
        best = warp_max_u64(best);
        const int slot = publish(make_float4(__uint_as_float(uint32_t(best)), __uint_as_float(uint32_t(best >> 32)),
                                             0.f, 0.f));
        if (warp == 0) {
            uint64_t g = 0;
#pragma unroll
            for (int h = 0; h < kParts / 32; ++h) {
                const float4 v = fetch(slot, lane + 32 * h);
                const uint64_t key = (uint64_t(__float_as_uint(v.y)) << 32) | __float_as_uint(v.x);
                g = key > g ? key : g;
            }
            g = warp_max_u64(g);
            if (rank == 0 && lane == 0) a.final_tok[size_t(b) * n + i] = int32_t(topk_key_token(g));
        }
        if (rank == 0) {
            for (int j = tid; j < J; j += kPrepThreads) {
                a.ratio[size_t(b) * n + s_kids[j]] = NAN;
                if (a.out_ratio) a.out_ratio[size_t(b) * n + s_kids[j]] = NAN;
            }
            if (i == 0 && tid == 0 && a.out_ratio) a.out_ratio[size_t(b) * n] = NAN;
        }
        cluster.sync();
        return;
    }

    const float c = a.c;
    // row statistics: max, then the scaled sum of exponentials, per thread / warp / cluster
    float mp = -INFINITY, mq = -INFINITY, spp = 0.f, sqq = 0.f;
#pragma unroll
    for (int j = 0; j < kE; ++j) mp = fmaxf(mp, xp[j]);
    if (mp != -INFINITY) {
        const float mc = mp * c;
#pragma unroll
        for (int j = 0; j < kE; ++j) spp += fast_exp2(fmaf(xp[j], c, -mc));
    }
    if (has_q) {
#pragma unroll
        for (int j = 0; j < kE; ++j) mq = fmaxf(mq, xq[j]);
        if (mq != -INFINITY) {
            const float mc = mq * c;
#pragma unroll
            for (int j = 0; j < kE; ++j) sqq += fast_exp2(fmaf(xq[j], c, -mc));
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        ms_merge(mp, spp, __shfl_xor_sync(0xffffffffu, mp, off), __shfl_xor_sync(0xffffffffu, spp, off), c);
        ms_merge(mq, sqq, __shfl_xor_sync(0xffffffffu, mq, off), __shfl_xor_sync(0xffffffffu, sqq, off), c);
    }
    {
        const int slot = publish(make_float4(mp, spp, mq, sqq));
        if (warp == 0) {
            // row-wide max, then the scaled sums in double; identical in every CTA (same partials,
            // same order)
            float4 v[kParts / 32];
            float Mp = -INFINITY, Mq = -INFINITY;
#pragma unroll
            for (int h = 0; h < kParts / 32; ++h) {
                v[h] = fetch(slot, lane + 32 * h);
                Mp = fmaxf(Mp, v[h].x);
                Mq = fmaxf(Mq, v[h].z);
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                Mp = fmaxf(Mp, __shfl_xor_sync(0xffffffffu, Mp, off));
                Mq = fmaxf(Mq, __shfl_xor_sync(0xffffffffu, Mq, off));
            }
            FF Sp, Sq;
#pragma unroll
            for (int h = 0; h < kParts / 32; ++h) {
                FF tp, tq;
                tp.hi = v[h].x != -INFINITY ? v[h].y * exp2f((v[h].x - Mp) * c) : 0.f;
                tq.hi = v[h].z != -INFINITY ? v[h].w * exp2f((v[h].z - Mq) * c) : 0.f;
                Sp = ff_add(Sp, tp);
                Sq = ff_add(Sq, tq);
            }
            Sp = ff_warp_sum(Sp);
            Sq = ff_warp_sum(Sq);
            if (lane == 0) {
                s_M[0] = Mp;
                s_M[1] = Mq;
                s_lnS[0] = log_fast(ff_to_double(Sp));
                s_lnS[1] = has_q ? log_fast(ff_to_double(Sq)) : 0.0;
            }
        }
        __syncthreads();
    }
    const float Mp = s_M[0], Mq = s_M[1];
    const double lnSp = s_lnS[0], lnSq = s_lnS[1];
    {
        // probabilities in place: p0 = 2^(((x - Mp)/T - ln Sp) log2 e), ln S carried as hi + lo
        const float lp_hi = float(lnSp), lp_lo = float(lnSp - double(lp_hi));
        const float lq_hi = float(lnSq), lq_lo = float(lnSq - double(lq_hi));
        const float inv_t = a.inv_t;
#pragma unroll
        for (int j = 0; j < kE; ++j)
            xp[j] = xp[j] == -INFINITY ? 0.f : fast_exp2((fmaf(xp[j] - Mp, inv_t, -lp_hi) - lp_lo) * kLog2e);
        if (has_q) {
#pragma unroll
            for (int j = 0; j < kE; ++j)
                xq[j] = xq[j] == -INFINITY ? 0.f : fast_exp2((fmaf(xq[j] - Mq, inv_t, -lq_hi) - lq_lo) * kLog2e);
        }
    }

    // rejection chain: c_0 = 0, S_0 = 1; after rejecting child j: c_{j+1} = c_j + S_j and
    // S_{j+1} = sum (p0 - c_{j+1} q)+ (a zero sum keeps the previous distribution)
    double cj = 0.0, Sj = 1.0;
    if (tid == 0) {
        s_cj[0] = 0.0;
        s_Sj[0] = 1.0;
    }
    for (int j = 0; j < J && has_q; ++j) {
        const double cn = cj + Sj;
        const float cnf = float(cn);
        float part = 0.f;
#pragma unroll
        for (int e = 0; e < kE; ++e) part += fmaxf(fmaf(-cnf, xq[e], xp[e]), 0.f);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
        const int slot = publish(make_float4(part, 0.f, 0.f, 0.f));
        if (warp == 0) {
            FF S;
#pragma unroll
            for (int h = 0; h < kParts / 32; ++h) {
                FF t;
                t.hi = fetch(slot, lane + 32 * h).x;
                S = ff_add(S, t);
            }
            S = ff_warp_sum(S);
            if (lane == 0) s_tot = ff_to_double(S);
        }
        __syncthreads();
        const double Sn = s_tot;
        if (Sn > 0.0) {
            cj = cn;
            Sj = Sn;
        }
        if (tid == 0) {
            s_cj[j + 1] = cj;
            s_Sj[j + 1] = Sj;
        }
    }
    __syncthreads();
    // accept ratios of the children, in double (p0 - c_j q cancels when the two are close)
    if (rank == 0 && tid < J) {
        float r = NAN;
        if (has_q) {
            const double p0 = exp((double(s_xk[tid]) - double(Mp)) * a.inv_td - lnSp);
            const double q0 = exp((double(s_yk[tid]) - double(Mq)) * a.inv_td - lnSq);
            const double num = tid == 0 ? p0 : fmax(p0 - s_cj[tid] * q0, 0.0);
            const double den = s_Sj[tid] * q0;
            r = den > 0.0 ? float(num / den) : INFINITY;
        }
        a.ratio[size_t(b) * n + s_kids[tid]] = r;
        if (a.out_ratio) a.out_ratio[size_t(b) * n + s_kids[tid]] = r;
    }
    if (i == 0 && rank == 0 && tid == 0 && a.out_ratio) a.out_ratio[size_t(b) * n] = NAN;

    // final draw at this node: residual r(t) = (p0 - c_J q)+ (p0 itself when J == 0), inverse CDF
    // with u[0] over ascending token ids; this thread's run is tokens lo + t0 ... lo + t0 + kE - 1
    const float cjf = float(cj);
    const bool use_res = J > 0 && has_q;
    float tsum = 0.f;
    int tlast = -1;
#pragma unroll
    for (int e = 0; e < kE; ++e) {
        const float r = use_res ? fmaxf(fmaf(-cjf, xq[e], xp[e]), 0.f) : xp[e];
        xp[e] = r;  // keep the residual for the scan below
        tsum += r;
        if (r > 0.f) tlast = t0 + e;
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
    const float wtot = __shfl_sync(0xffffffffu, incl, 31);
    const int slot = publish(make_float4(wtot, __int_as_float(wl), 0.f, 0.f));
    if (warp == 0 && lane < CL) {
        // rank `lane`: total and last positive index (its warps in order)
        double rt = 0.0;
        int rl = -1;
        for (int w = 0; w < kWarpsPrep; ++w) {
            const float4 v = fetch(slot, lane * kWarpsPrep + w);
            rt += double(v.x);
            rl = max(rl, __float_as_int(v.y));
        }
        s_rank[lane] = rt;
        s_rlast[lane] = rl;
    }
    if (tid == 0) s_claim = kPrepThreads;
    __syncthreads();
    double total = 0.0;
    for (int r = 0; r < CL; ++r) total += s_rank[r];
    const double target = double(a.uniforms[size_t(b) * n]) * total;
    // The owner CTA holds the first CDF step above the target (running double sums over the
    // ranks are monotone).  If rounding leaves the target at or above the total, the draw clamps
    // to the last token of positive mass.
    double base = 0.0, rbase = 0.0;
    int owner = -1, last_rank = -1;
    for (int r = 0; r < CL; ++r) {
        if (owner < 0 && target < base + s_rank[r]) {
            owner = r;
            rbase = base;
        }
        base += s_rank[r];
        if (s_rlast[r] >= 0) last_rank = r;
    }
    const bool clamp = owner < 0;
    if (clamp) owner = last_rank;
    float wbase = 0.f;
    if (rank == owner && !clamp)
        for (int w = 0; w < warp; ++w) wbase += s_part[slot][w].x;  // this CTA's earlier warps
    const float excl = wbase + incl - tsum;
    const float local = float(target - rbase);
    // the first thread whose run ends above the local target owns the step
    if (rank == owner && !clamp && tsum > 0.f && excl + tsum > local) atomicMin(&s_claim, tid);
    __syncthreads();
    if (rank == owner) {
        if (!clamp && tid == s_claim) {
            float acc = excl;
            int found = tlast;
            bool done = false;
#pragma unroll
            for (int e = 0; e < kE; ++e) {
                acc += xp[e];
                if (!done && xp[e] > 0.f && acc > local) {
                    found = t0 + e;
                    done = true;
                }
            }
            a.final_tok[size_t(b) * n + i] = lo + found;
        } else if (tid == 0 && (clamp || s_claim == kPrepThreads)) {
            a.final_tok[size_t(b) * n + i] = lo + s_rlast[owner];
        }
    }
    if (owner < 0 && rank == 0 && tid == 0) a.final_tok[size_t(b) * n + i] = 0;  // no positive mass at all
    cluster.sync();  // keep this CTA's shared memory alive until every peer has read it
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
        s_ratio[tid] = a.ratio[o];
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
    return kWsHeader + align_up(size_t(c.batch) * n * sizeof(float), 256) +
           align_up(size_t(c.batch) * n * sizeof(int32_t), 256);
}

namespace {
template <int CL>
cudaError_t launch_prep(const VerifyArgs &a, int n, int batch, cudaStream_t stream) {
    static bool attr = false;
    if (!attr && CL > 8) {
        cudaError_t e = cudaFuncSetAttribute(verify_prep_kernel<CL>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
    attr = true;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(CL, n, batch);
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
    a.ratio = reinterpret_cast<float *>(w + kWsHeader);
    a.final_tok = reinterpret_cast<int32_t *>(w + kWsHeader + align_up(size_t(c.batch) * n * sizeof(float), 256));
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
    const cudaError_t e = cl == 8 ? launch_prep<8>(a, n, c.batch, stream) : launch_prep<16>(a, n, c.batch, stream);
    if (e != cudaSuccess) return EAGLE_ERR_CUDA;
    note_launch();
    verify_walk_kernel<<<c.batch, 64, 0, stream>>>(a);
    note_launch();
    return cudaPeekAtLastError() == cudaSuccess ? EAGLE_OK : EAGLE_ERR_CUDA;
}

size_t verify_max_vocab() { return size_t(16) * kPrepThreads * kE; }

}  // namespace eagle
