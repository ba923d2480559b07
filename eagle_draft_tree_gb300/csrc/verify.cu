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
//   verify_prep_kernel  one 8-CTA cluster per (sequence, node): each CTA holds 1/8 of the
//                       node's target row (and of its draft row when it has children) in shared
//                       memory; log-sum-exp, the S_j passes and the inverse-CDF scan are reduced
//                       across the cluster through distributed shared memory.
//   verify_walk_kernel  one warp per sequence: validates the tree and walks it.
#include <cooperative_groups.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "common.cuh"

namespace cg = cooperative_groups;

namespace eagle {

namespace {

constexpr int kCl = 8;            // CTAs per cluster (one node's row split 8 ways)
constexpr int kPrepThreads = 256;
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

__device__ __forceinline__ float block_sum(float v, float *scratch) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    __syncthreads();
    if (lane == 0) scratch[warp] = v;
    __syncthreads();
    float r = 0.f;
#pragma unroll
    for (int w = 0; w < kPrepThreads / 32; ++w) r += scratch[w];
    return r;
}

__device__ __forceinline__ void ms_merge(float &m, float &s, float mo, float so, float c) {
    const float M = fmaxf(m, mo);
    if (M == -INFINITY) return;
    const float x = (m == -INFINITY) ? 0.f : s * exp2f((m - M) * c);
    const float y = (mo == -INFINITY) ? 0.f : so * exp2f((mo - M) * c);
    m = M;
    s = x + y;
}

// add one element x to a running (max m, scaled sum s)
__device__ __forceinline__ void ms_add(float &m, float &s, float x, float c) {
    if (x > m) {
        s = s * exp2f((m - x) * c) + 1.f;
        m = x;
    } else {
        s += exp2f((x - m) * c);
    }
}

__global__ void __cluster_dims__(kCl, 1, 1) __launch_bounds__(kPrepThreads)
    verify_prep_kernel(VerifyArgs a) {
    extern __shared__ __align__(16) float sm[];  // [slice] target, then [slice] draft
    __shared__ float s_scratch[kPrepThreads / 32];
    __shared__ unsigned long long s_xchg[2][4];  // per-pass partials exchanged across the cluster (bit patterns)
    __shared__ int s_kids[kMaxKids];
    __shared__ int s_nk;

    cg::cluster_group cluster = cg::this_cluster();
    const int rank = int(cluster.block_rank());
    const int i = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x;
    const int n = a.n, V = a.V;
    const int lo = rank * a.slice;
    const int hi = min(V, lo + a.slice);
    const int cnt = hi > lo ? hi - lo : 0;

    const int32_t *par = a.parents + size_t(b) * n;
    const int32_t *tok = a.tokens + size_t(b) * n;
    if (tid == 0) {
        int nk = 0;
        for (int j = i + 1; j < n; ++j)
            if (par[j] == i && nk < kMaxKids) s_kids[nk++] = j;
        s_nk = nk;
    }
    __syncthreads();
    const int J = s_nk;
    const float *xrow = a.target + (size_t(b) * n + i) * V;
    int row = J > 0 ? a.node_row[size_t(b) * n + i] : -1;
    const bool has_q = J > 0 && row >= 0 && row < a.R;
    const float *yrow = has_q ? a.draft + (size_t(b) * a.R + row) * V : nullptr;
    int pass = 0;

    // exchange: every CTA publishes `vals` (up to 4 doubles) and reads all ranks' in rank order
    __shared__ unsigned long long s_all[kCl][4];
    auto exchange = [&](const unsigned long long *vals, int nv) {
        const int slot = pass & 1;
        if (tid < nv) s_xchg[slot][tid] = vals[tid];
        cluster.sync();
        if (tid < kCl * nv) {
            const int r = tid / nv, v = tid % nv;
            unsigned long long *remote = cluster.map_shared_rank(&s_xchg[slot][0], r);
            s_all[r][v] = remote[v];
        }
        __syncthreads();
        ++pass;
    };
    auto dbl = [](double x) { return static_cast<unsigned long long>(__double_as_longlong(x)); };
    auto all = [&](int r, int v) { return __longlong_as_double(static_cast<long long>(s_all[r][v])); };

    if (a.greedy) {
        // argmax of the target row (ties to the lower id)
        uint64_t best = 0;
        for (int t = lo + tid; t < hi; t += kPrepThreads) {
            const uint64_t key = topk_key(__ldg(xrow + t), uint32_t(t));
            best = key > best ? key : best;
        }
        best = warp_max_u64(best);
        __shared__ uint64_t s_best[kPrepThreads / 32];
        if ((tid & 31) == 0) s_best[tid >> 5] = best;
        __syncthreads();
        if (tid < 32) {
            uint64_t v = tid < kPrepThreads / 32 ? s_best[tid] : 0;
            v = warp_max_u64(v);
            if (tid == 0) s_best[0] = v;
        }
        __syncthreads();
        const unsigned long long mine[1] = {s_best[0]};
        exchange(mine, 1);
        if (rank == 0 && tid == 0) {
            uint64_t g = 0;
            for (int r = 0; r < kCl; ++r) {
                const uint64_t v = s_all[r][0];
                g = v > g ? v : g;
            }
            a.final_tok[size_t(b) * n + i] = int32_t(topk_key_token(g));
            for (int j = 0; j < J; ++j) a.ratio[size_t(b) * n + s_kids[j]] = NAN;
            if (a.out_ratio) {
                for (int j = 0; j < J; ++j) a.out_ratio[size_t(b) * n + s_kids[j]] = NAN;
                if (i == 0) a.out_ratio[size_t(b) * n] = NAN;
            }
        }
        cluster.sync();
        return;
    }

    float *sp = sm;
    float *sq = sm + a.slice;
    const float c = a.c;

    // pass A: stage the row slices and their (max, scaled sum)
    float mp = -INFINITY, spp = 0.f, mq = -INFINITY, sqq = 0.f;
    const bool vec = ((V & 3) == 0) && ((lo & 3) == 0);
    if (vec) {
        const float4 *x4 = reinterpret_cast<const float4 *>(xrow + lo);
        const float4 *y4 = has_q ? reinterpret_cast<const float4 *>(yrow + lo) : nullptr;
        for (int t = tid; t < cnt / 4; t += kPrepThreads) {
            const float4 v = __ldg(x4 + t);
            reinterpret_cast<float4 *>(sp)[t] = v;
            const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) ms_add(mp, spp, vv[e], c);
            if (has_q) {
                const float4 w = __ldg(y4 + t);
                reinterpret_cast<float4 *>(sq)[t] = w;
                const float ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) ms_add(mq, sqq, ww[e], c);
            }
        }
    } else {
        for (int t = tid; t < cnt; t += kPrepThreads) {
            const float v = __ldg(xrow + lo + t);
            sp[t] = v;
            ms_add(mp, spp, v, c);
            if (has_q) {
                const float w = __ldg(yrow + lo + t);
                sq[t] = w;
                ms_add(mq, sqq, w, c);
            }
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        ms_merge(mp, spp, __shfl_xor_sync(0xffffffffu, mp, off), __shfl_xor_sync(0xffffffffu, spp, off), c);
        ms_merge(mq, sqq, __shfl_xor_sync(0xffffffffu, mq, off), __shfl_xor_sync(0xffffffffu, sqq, off), c);
    }
    __shared__ float4 s_ms[kPrepThreads / 32];
    if ((tid & 31) == 0) s_ms[tid >> 5] = make_float4(mp, spp, mq, sqq);
    __syncthreads();
    {
        float M0 = -INFINITY, S0 = 0.f, M1 = -INFINITY, S1 = 0.f;
        for (int w = 0; w < kPrepThreads / 32; ++w) {
            ms_merge(M0, S0, s_ms[w].x, s_ms[w].y, c);
            ms_merge(M1, S1, s_ms[w].z, s_ms[w].w, c);
        }
        const unsigned long long mine[4] = {dbl(M0), dbl(S0), dbl(M1), dbl(S1)};
        exchange(mine, 4);
    }
    // row-wide max and log of the scaled sum (one thread computes, every CTA of the cluster gets
    // the same values because it reduces the same partials in the same order)
    __shared__ float s_M[2];
    __shared__ double s_lnS[2];
    if (tid == 0) {
        float Mp = -INFINITY, Mq = -INFINITY;
        for (int r = 0; r < kCl; ++r) {
            Mp = fmaxf(Mp, float(all(r, 0)));
            Mq = fmaxf(Mq, float(all(r, 2)));
        }
        double Sp = 0.0, Sq = 0.0;
        for (int r = 0; r < kCl; ++r) {
            const float m0 = float(all(r, 0)), m1 = float(all(r, 2));
            if (m0 != -INFINITY) Sp += all(r, 1) * double(exp2f((m0 - Mp) * c));
            if (m1 != -INFINITY) Sq += all(r, 3) * double(exp2f((m1 - Mq) * c));
        }
        s_M[0] = Mp;
        s_M[1] = Mq;
        s_lnS[0] = log(Sp);
        s_lnS[1] = has_q ? log(Sq) : 0.0;
    }
    __syncthreads();
    const float Mp = s_M[0], Mq = s_M[1];
    const double lnSp = s_lnS[0], lnSq = s_lnS[1];
    const float lp_hi = float(lnSp), lp_lo = float(lnSp - double(lp_hi));
    const float lq_hi = float(lnSq), lq_lo = float(lnSq - double(lq_hi));
    const float inv_t = a.inv_t;
    // p0(t) = exp((x - Mp)/T - ln Sp), with ln Sp carried as hi + lo
    auto p_of = [&](float x) { return expf(fmaf(x - Mp, inv_t, -lp_hi) - lp_lo); };
    auto q_of = [&](float y) { return expf(fmaf(y - Mq, inv_t, -lq_hi) - lq_lo); };

    // pass B: convert the slices to probabilities in place
    for (int t = tid; t < cnt; t += kPrepThreads) {
        sp[t] = p_of(sp[t]);
        if (has_q) sq[t] = q_of(sq[t]);
    }
    __syncthreads();

    // rejection chain at this node: ratio_j for child j, then the residual of the final draw
    double cj = 0.0, Sj = 1.0;  // c_0, S_0
    for (int j = 0; j < J; ++j) {
        const int child = s_kids[j];
        if (tid == 0 && rank == 0) {
            // the accept ratio of child j in double: p0(t) - c_j q(t) cancels when the two are close
            const int t = tok[child];
            float r = NAN;
            if (has_q && t >= 0 && t < V) {
                const double p0 = exp((double(__ldg(xrow + t)) - double(Mp)) * a.inv_td - lnSp);
                const double q0 = exp((double(__ldg(yrow + t)) - double(Mq)) * a.inv_td - lnSq);
                const double num = j == 0 ? p0 : fmax(p0 - cj * q0, 0.0);
                const double den = Sj * q0;
                r = den > 0.0 ? float(num / den) : INFINITY;
            }
            a.ratio[size_t(b) * n + child] = r;
            if (a.out_ratio) a.out_ratio[size_t(b) * n + child] = r;
        }
        // reject child j: c_{j+1} = c_j + S_j, S_{j+1} = sum (p0 - c_{j+1} q)+
        const double cn = cj + Sj;
        const float cnf = float(cn);
        float part = 0.f;
        if (has_q)
            for (int t = tid; t < cnt; t += kPrepThreads) part += fmaxf(fmaf(-cnf, sq[t], sp[t]), 0.f);
        part = block_sum(part, s_scratch);
        const unsigned long long mine[1] = {dbl(double(part))};
        exchange(mine, 1);
        double Sn = 0.0;
        for (int r = 0; r < kCl; ++r) Sn += all(r, 0);  // few double adds, same order everywhere
        if (Sn > 0.0) {  // otherwise the adjusted distribution keeps p_j
            cj = cn;
            Sj = Sn;
        }
    }
    if (i == 0 && rank == 0 && tid == 0 && a.out_ratio) a.out_ratio[size_t(b) * n] = NAN;

    // final draw at this node: residual r(t) = (p0 - c_J q)+ (p0 itself when J == 0), inverse CDF
    // with u[0].  Each thread owns a contiguous run of the slice.
    const float cjf = float(cj);
    const bool use_res = J > 0 && has_q;
    const int run = (cnt + kPrepThreads - 1) / kPrepThreads;
    const int t0 = min(cnt, tid * run), t1 = min(cnt, t0 + run);
    float tsum = 0.f;
    int tlast = -1;
    for (int t = t0; t < t1; ++t) {
        const float r = use_res ? fmaxf(fmaf(-cjf, sq[t], sp[t]), 0.f) : sp[t];
        tsum += r;
        if (r > 0.f) tlast = t;
    }
    // exclusive scan of the run sums across the block
    const int lane = tid & 31, warp = tid >> 5;
    float incl = tsum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
    }
    __shared__ float s_wtot[kPrepThreads / 32];
    __shared__ int s_wlast[kPrepThreads / 32];
    int wl = tlast;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) wl = max(wl, __shfl_xor_sync(0xffffffffu, wl, off));
    if (lane == 31) s_wtot[warp] = incl;
    if (lane == 0) s_wlast[warp] = wl;
    __syncthreads();
    float wbase = 0.f, ctot = 0.f;
    int clast = -1;
    for (int w = 0; w < kPrepThreads / 32; ++w) {
        if (w < warp) wbase += s_wtot[w];
        ctot += s_wtot[w];
        clast = max(clast, s_wlast[w]);
    }
    const float excl = wbase + incl - tsum;
    {
        const unsigned long long mine[2] = {dbl(double(ctot)), dbl(double(clast))};
        exchange(mine, 2);
    }
    double total = 0.0;
    for (int r = 0; r < kCl; ++r) total += all(r, 0);
    const double target = double(a.uniforms[size_t(b) * n]) * total;
    // The owner CTA holds the first CDF step above the target (running double sums over the
    // ranks are monotone).  If rounding leaves the target at or above the total, the draw clamps
    // to the last token of positive mass.
    double base = 0.0;
    int owner = -1, last_rank = -1;
    for (int r = 0; r < kCl; ++r) {
        if (owner < 0 && target < base + all(r, 0)) owner = r;
        base += all(r, 0);
        if (all(r, 1) >= 0.0) last_rank = r;
    }
    const bool clamp = owner < 0;
    if (clamp) owner = last_rank;
    __shared__ int s_claim;
    if (tid == 0) s_claim = kPrepThreads;
    __syncthreads();
    float local = 0.f;
    if (rank == owner && !clamp) {
        double rbase = 0.0;
        for (int r = 0; r < rank; ++r) rbase += all(r, 0);
        local = float(target - rbase);
        // the first thread whose run ends above the local target owns the step
        if (tsum > 0.f && excl + tsum > local) atomicMin(&s_claim, tid);
    }
    __syncthreads();
    if (rank == owner) {
        if (!clamp && tid == s_claim) {
            float acc = excl;
            int found = tlast;
            for (int t = t0; t < t1; ++t) {
                const float r = use_res ? fmaxf(fmaf(-cjf, sq[t], sp[t]), 0.f) : sp[t];
                acc += r;
                if (r > 0.f && acc > local) {
                    found = t;
                    break;
                }
            }
            a.final_tok[size_t(b) * n + i] = lo + found;
        } else if (tid == 0 && (clamp || s_claim == kPrepThreads)) {
            a.final_tok[size_t(b) * n + i] = lo + clast;
        }
    }
    if (owner < 0 && rank == 0 && tid == 0) a.final_tok[size_t(b) * n + i] = 0;  // no positive mass at all
    cluster.sync();  // keep this CTA's shared memory alive until every peer has read it
}

__global__ void verify_walk_kernel(VerifyArgs a) {
    const int b = blockIdx.x;
    if (threadIdx.x != 0) return;
    const int n = a.n, D = a.D;
    const int32_t *tok = a.tokens + size_t(b) * n;
    const int32_t *par = a.parents + size_t(b) * n;
    const int32_t *row = a.node_row + size_t(b) * n;
    const float *u = a.uniforms + size_t(b) * n;
    const float *ratio = a.ratio + size_t(b) * n;
    const int32_t *fin = a.final_tok + size_t(b) * n;
    int32_t *ot = a.out_tokens + size_t(b) * (D + 1);
    int32_t *op = a.out_path + size_t(b) * D;
    for (int j = 0; j <= D; ++j) ot[j] = -1;
    for (int j = 0; j < D; ++j) op[j] = -1;

    bool bad = par[0] != -1;
    for (int j = 0; j < n; ++j) {
        if (tok[j] < 0 || tok[j] >= a.V) bad = true;
        if (j > 0 && (par[j] < 0 || par[j] >= j)) bad = true;
    }
    if (!bad && !a.greedy) {
        for (int j = 1; j < n; ++j) {
            const int p = par[j];
            if (row[p] < 0 || row[p] >= a.R) bad = true;
        }
    }
    if (bad) {
        set_status(a.status, EAGLE_ERR_DEVICE_INPUT);
        a.out_len[b] = 0;
        return;
    }
    int node = 0, len = 0;
    for (;;) {
        int next = -1;
        if (a.greedy) {
            const int g = fin[node];
            for (int j = node + 1; j < n; ++j)
                if (par[j] == node && tok[j] == g) {
                    next = j;
                    break;
                }
        } else {
            for (int j = node + 1; j < n; ++j)
                if (par[j] == node && u[j] < ratio[j]) {
                    next = j;
                    break;
                }
        }
        if (next < 0 || len >= D) {
            if (next >= 0) set_status(a.status, EAGLE_ERR_DEVICE_INPUT);  // tree deeper than D
            ot[len++] = fin[node];
            break;
        }
        ot[len] = tok[next];
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
    int slice = (c.vocab + kCl - 1) / kCl;
    slice = (slice + 3) & ~3;
    a.slice = slice;
    a.greedy = c.temperature <= 0.f;
    a.inv_t = a.greedy ? 1.f : 1.f / c.temperature;
    a.inv_td = a.greedy ? 1.0 : 1.0 / double(c.temperature);
    a.c = kLog2e * a.inv_t;
    const size_t smem = a.greedy ? 0 : size_t(2) * slice * sizeof(float);
    static size_t attr = 0;
    if (smem > attr) {
        if (cudaFuncSetAttribute(verify_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) !=
            cudaSuccess)
            return EAGLE_ERR_CUDA;
        attr = smem;
    }
    dim3 grid(kCl, n, c.batch);
    verify_prep_kernel<<<grid, kPrepThreads, smem, stream>>>(a);
    note_launch();
    verify_walk_kernel<<<c.batch, 32, 0, stream>>>(a);
    note_launch();
    return cudaPeekAtLastError() == cudaSuccess ? EAGLE_OK : EAGLE_ERR_CUDA;
}

size_t verify_max_vocab() {
    // two fp32 slices of V/8 entries must fit the opt-in shared memory of one CTA (227 KB)
    return size_t(227 * 1024 - 4096) / (2 * sizeof(float)) * kCl;
}

}  // namespace eagle
