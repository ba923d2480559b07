// build_tree.cu -- EAGLE-2 dynamic draft-tree build on sm_103a.
//
// Page: "(EAGLE 2) EAGLE-2: Faster Inference of Language Models with Dynamic Draft Trees",
// sections "Expanding the Draft Tree" (V_i = product of draft confidences on the root->i path;
// only the k most valuable nodes of a depth are expanded), "Rerank draft tokens" (top-m by V over
// every candidate, shallower first on equal V, so the kept set is still a connected tree) and
// "Tree Attention Mask" (flattened sequence, ancestors-only visibility).
//
// Kernels:
//   row_topk_kernel    one HBM pass over every draft row.  A row is cut into `splits` slices
//                      handled by the CTAs of one thread-block cluster; each CTA keeps an online
//                      log-sum-exp of x/T and a top-16 list (per-warp sorted lists that only see
//                      values above a block-shared threshold), pushes both into rank 0's shared
//                      memory, and rank 0 merges them after one cluster barrier and writes the
//                      row's k children (token, fp64 log-confidence).  With sampled children the rows go
//                      to row_sample_kernel (sample_children.cu) instead, same outputs.
//   tree_select_kernel one CTA per sequence: per-depth frontier selection (rank of a 64-bit
//                      composite key within its depth by counting, a group of threads per
//                      candidate), the frontier's expansion, the global rerank (a key's rank
//                      within its depth plus binary searches in the other depths' sorted lists),
//                      flatten, masks.  A stepwise build runs it once, to finalize, replaying the frontiers
//                      tree_step_kernel chose one depth at a time.
//   static_tree_kernel the static (EAGLE-1) tree or chain of a caller's template over the rows'
//                      children (see the section below).
#include <cooperative_groups.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "common.cuh"

namespace cg = cooperative_groups;

namespace eagle {

int splits_for_rows(long rows, int vocab);
eagle_status row_sample_launch(const float *draft, const float *u, int B, int R, int V, int k, float tree_temp,
                               int32_t *row_tok, double *row_lc, int out_R, int out_r0, int32_t *status,
                               cudaStream_t stream);

namespace {

constexpr int kRowThreads = 512;
constexpr int kRowWarps = kRowThreads / 32;
constexpr int kRowVals = 16;  // values per thread per batch (4 float4 in registers)
constexpr int kSelThreads = 512;
constexpr int kMaxPool = 1024;
constexpr int kMaxSelDepth = 65;  // depths 1 .. 64
constexpr int kMaxSplits = 8;  // portable cluster size

// Merge (m_a, s_a) and (m_b, s_b) where s = sum 2^((x - m) c).
__device__ __forceinline__ void ms_merge(float &m, float &s, float mo, float so, float c) {
    float M = fmaxf(m, mo);
    if (M == -INFINITY) return;
    float a = (m == -INFINITY) ? 0.f : s * exp2f((m - M) * c);
    float b = (mo == -INFINITY) ? 0.f : so * exp2f((mo - M) * c);
    m = M;
    s = a + b;
}

struct RowArgs {
    const float *x;     // [B][R][V]
    int32_t *row_tok;   // [B][out_R][k]  children tokens (rows out_r0 ..)
    double *row_lc;     // [B][out_R][k]  children log-confidences (rows out_r0 ..)
    int V, R, k, chunk, out_R, out_r0;
    float c;            // log2(e) / tree_temp
    double inv_t;       // 1 / tree_temp
};

// The warp's 32 lane keys sorted descending across the lanes (bitonic network).
__device__ __forceinline__ uint64_t warp_sort_desc(uint64_t v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            const uint64_t o = shfl_xor_u64(v, stride);
            const bool up = (lane & size) == 0;       // this pair sorts descending when up
            const bool lower = (lane & stride) == 0;  // this lane holds the earlier position
            v = (up == lower) ? (o > v ? o : v) : (o < v ? o : v);
        }
    }
    return v;
}

// Fold `count` descending 16-key lists (zero padded) stored in buf[0][0..count) into buf[?][0]
// with a tree of warp bitonic merges; returns the buffer index holding the result.  Called by the
// whole CTA (block barriers inside).
__device__ __forceinline__ int tree_merge16(uint64_t (*buf)[kRowWarps][16], int count) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int cur = 0;
    while (count > 1) {
        const int pairs = count >> 1;
        if (warp < pairs) {
            const uint64_t v = lane < 16 ? buf[cur][2 * warp][lane] : buf[cur][2 * warp + 1][31 - lane];
            const uint64_t w = warp_bitonic_merge32(v);
            if (lane < 16) buf[cur ^ 1][warp][lane] = w;
        } else if (warp == pairs && (count & 1)) {
            if (lane < 16) buf[cur ^ 1][warp][lane] = buf[cur][2 * warp][lane];  // odd list carried over
        }
        __syncthreads();
        count = pairs + (count & 1);
        cur ^= 1;
    }
    return cur;
}

__global__ void __launch_bounds__(kRowThreads) row_topk_kernel(RowArgs a) {
    pdl_wait();
    pdl_launch_next();
    __shared__ uint64_t s_lists[2][kRowWarps][16];
    __shared__ unsigned long long s_bound;  // CTA-wide lower bound of the slice's 16th key
    __shared__ float2 s_ms[kRowWarps];
    __shared__ uint64_t s_recv[kMaxSplits][16];  // rank 0: every slice's list, pushed by its CTA
    __shared__ float2 s_recvms[kMaxSplits];      // rank 0: every slice's (max, scaled sum)

    cg::cluster_group cluster = cg::this_cluster();
    const int split = int(cluster.block_rank());
    const int splits = int(cluster.num_blocks());
    const int r = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float *row = a.x + (size_t(b) * a.R + r) * size_t(a.V);
    const int lo = split * a.chunk;
    const int hi = min(a.V, lo + a.chunk);
    const float c = a.c;
    const bool vec = ((a.V & 3) == 0) && ((reinterpret_cast<uintptr_t>(row) & 15) == 0) && ((lo & 3) == 0);

    float m = -INFINITY, s = 0.f;
    WarpTopK<16> top;
    uint64_t seed = 0;  // CTA-wide lower bound of the slice's top-16, from the first batch
    bool seeded = false;

    // One batch: kRowVals values per thread.  Statistics in registers, then the top-16 offer: a
    // value can only be in the slice's top-16 if its key reaches the bound, the larger of the
    // seed (the 16th largest of the CTA's 512 thread maxima of the first batch, found by sorting
    // each warp's lane maxima and merging the sixteen top halves) and the largest of the warps'
    // current 16th keys, which the warps publish with atomicMax: 16 distinct keys at or above
    // either are known.  A lane offers values only when its batch maximum reaches the bound (one
    // vote per batch).  The first batch is CTA-uniform (block barriers inside the seed).
    auto batch = [&](const float (&x)[kRowVals], const int (&tk)[kRowVals]) {
        float mx = x[0];
#pragma unroll
        for (int j = 1; j < kRowVals; ++j) mx = fmaxf(mx, x[j]);
        if (mx > m) {
            s = (m == -INFINITY) ? 0.f : s * fast_exp2((m - mx) * c);
            m = mx;
        }
        if (m != -INFINITY) {
            const float mc = m * c;
#pragma unroll
            for (int j = 0; j < kRowVals; ++j) s += fast_exp2(fmaf(x[j], c, -mc));
        }
        if (!seeded) {
            int tmx = -1;  // the lane maximum's token (lowest id among equal values)
#pragma unroll
            for (int j = kRowVals - 1; j >= 0; --j)
                if (x[j] == mx) tmx = tk[j];
            const uint64_t srt = warp_sort_desc(mx == -INFINITY ? 0ull : topk_key(mx, uint32_t(tmx)));
            if (lane < 16) s_lists[0][warp][lane] = srt;
            __syncthreads();
            const int cur = tree_merge16(s_lists, kRowWarps);
            seed = s_lists[cur][0][15];
            seeded = true;
            __syncthreads();  // s_lists is reused by the final merge
        }
        const uint64_t shared_bound = *reinterpret_cast<volatile unsigned long long *>(&s_bound);
        uint64_t bound = seed > top.thr ? seed : top.thr;
        bound = shared_bound > bound ? shared_bound : bound;
        const float bval = bound == 0 ? -INFINITY : topk_key_value(bound);
        if (!__any_sync(0xffffffffu, mx >= bval && mx != -INFINITY)) return;
#pragma unroll
        for (int j = 0; j < kRowVals; ++j) {
            const bool cand = x[j] >= bval && x[j] != -INFINITY;
            if (__any_sync(0xffffffffu, cand)) {
                const uint64_t key = cand ? topk_key(x[j], uint32_t(tk[j])) : 0ull;
                top.insert(key >= bound ? key : 0ull);
            }
        }
        if (lane == 0 && top.thr > bound) atomicMax(&s_bound, static_cast<unsigned long long>(top.thr));
    };

    constexpr int kBatch = kRowThreads * kRowVals;
    const int nb = (hi - lo + kBatch - 1) / kBatch;  // same for every thread of the CTA
    if (tid == 0) s_bound = 0;
    __syncthreads();
    if (vec) {
        const float4 *row4 = reinterpret_cast<const float4 *>(row);
        float4 nxt[kRowVals / 4];
        auto load = [&](int bi, float4 (&dst)[kRowVals / 4]) {
#pragma unroll
            for (int j = 0; j < kRowVals / 4; ++j) {
                const int i4 = ((lo + bi * kBatch) >> 2) + tid + j * kRowThreads;
                dst[j] = 4 * i4 < hi ? __ldg(row4 + i4) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
            }
        };
        if (nb > 0) load(0, nxt);
        for (int bi = 0; bi < nb; ++bi) {
            float x[kRowVals];
            int tk[kRowVals];
#pragma unroll
            for (int j = 0; j < kRowVals / 4; ++j) {
                const int i4 = ((lo + bi * kBatch) >> 2) + tid + j * kRowThreads;
                x[4 * j] = nxt[j].x;
                x[4 * j + 1] = nxt[j].y;
                x[4 * j + 2] = nxt[j].z;
                x[4 * j + 3] = nxt[j].w;
#pragma unroll
                for (int e = 0; e < 4; ++e) tk[4 * j + e] = 4 * i4 + e;
            }
            if (bi + 1 < nb) load(bi + 1, nxt);  // next batch in flight while this one is consumed
            batch(x, tk);
        }
    } else {
        for (int bi = 0; bi < nb; ++bi) {
            float x[kRowVals];
            int tk[kRowVals];
#pragma unroll
            for (int j = 0; j < kRowVals; ++j) {
                const int t = lo + bi * kBatch + tid + j * kRowThreads;
                x[j] = t < hi ? __ldg(row + t) : -INFINITY;
                tk[j] = t;
            }
            batch(x, tk);
        }
    }

    // block: (max, sum) and the merged list
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        float mo = __shfl_xor_sync(0xffffffffu, m, off);
        float so = __shfl_xor_sync(0xffffffffu, s, off);
        ms_merge(m, s, mo, so, c);
    }
    if (lane == 0) s_ms[warp] = make_float2(m, s);
    if (lane < 16) s_lists[0][warp][lane] = top.key;
    __syncthreads();
    const int cur = tree_merge16(s_lists, kRowWarps);
    // this CTA's list and (max, sum) go to rank 0's receive slots (rank 0's own by local stores);
    // the cluster barrier (release / acquire) then makes them visible there.  Nothing of a
    // slice's own shared memory is read by another CTA, so the slices leave after the barrier.
    if (warp == 0) {
        float mm = lane < kRowWarps ? s_ms[lane].x : -INFINITY;
        float ss = lane < kRowWarps ? s_ms[lane].y : 0.f;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            float mo = __shfl_xor_sync(0xffffffffu, mm, off);
            float so = __shfl_xor_sync(0xffffffffu, ss, off);
            ms_merge(mm, ss, mo, so, c);
        }
        if (lane < 16) cluster.map_shared_rank(&s_recv[split][0], 0)[lane] = s_lists[cur][0][lane];
        if (lane == 0) *cluster.map_shared_rank(&s_recvms[split], 0) = make_float2(mm, ss);
    }
    cluster.sync();
    if (split != 0 || warp != 0) return;

    // cluster rank 0, one warp: merge the slices' lists (lanes 0..15 carry the running top 16,
    // lanes 16..31 the next slice's list reversed: a bitonic sequence for the merge network) and
    // sums, write the row's children
    uint64_t run = lane < 16 ? s_recv[0][lane] : 0ull;
    for (int j = 1; j < splits; ++j) run = warp_bitonic_merge32(lane < 16 ? run : s_recv[j][31 - lane]);
    const float2 ms = lane < splits ? s_recvms[lane] : make_float2(-INFINITY, 0.f);
    float M = ms.x;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    double S = ms.x == -INFINITY ? 0.0 : double(ms.y) * double(exp2f((ms.x - M) * c));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) S += __shfl_xor_sync(0xffffffffu, S, off);
    double lse = 0.0;
    if (lane == 0) lse = double(M) * a.inv_t + ln_pos(S);  // S >= 1: the maximum's own term
    lse = __shfl_sync(0xffffffffu, lse, 0);
    if (lane < a.k) {
        const size_t o = (size_t(b) * a.out_R + a.out_r0 + r) * a.k + lane;
        a.row_tok[o] = int32_t(topk_key_token(run));
        a.row_lc[o] = double(topk_key_value(run)) * a.inv_t - lse;
    }
}

// Composite selection key: larger = better.  High 54 bits: orderable log V (the low 10 bits of
// the double dropped); low 10 bits: 1023 - creation index (earlier creation wins a tie).
__device__ __forceinline__ uint64_t pool_key(double logv, int creation) {
    return (double_order_key(logv) & ~uint64_t(1023)) | uint64_t(1023 - creation);
}

struct SelectArgs {
    const int32_t *row_tok;
    const double *row_lc;
    const int32_t *root_token;
    int32_t *tokens, *parents, *depths, *node_row;
    uint64_t *mask;
    float *node_logv;
    int32_t *status;
    int V, D, k, m, R;
    // The finalize stage of a stepwise build: the frontier of every depth comes from `slots`
    // (pool index of slot s of depth f at [b][f][s], as the step kernel stored it) instead of
    // being ranked again.  nullptr in the one-call build.
    const int32_t *slots;
};

// Pool layout: depth 1 holds the root's k children (entries 0 .. k - 1, in child-rank order);
// depth f >= 2 holds the k^2 children of the depth f - 1 frontier from k + (f - 2)k^2 on, slot by
// slot (slot s's k children at s k .. s k + k - 1 of the depth).  The pool index is the creation
// index.
__device__ __forceinline__ int depth_base(int f, int k) { return f == 1 ? 0 : k + (f - 2) * k * k; }
__device__ __forceinline__ int depth_count(int f, int k) { return f == 1 ? k : k * k; }
__device__ __forceinline__ int depth_of(int e, int k) { return e < k ? 1 : 2 + (e - k) / (k * k); }
// Start of depth f's list of its min(count, m) best keys (descending) in the rerank's table.
__device__ __forceinline__ int list_base(int f, int k, int m) {
    return f == 1 ? 0 : min(k, m) + (f - 2) * min(k * k, m);
}

struct SelSmem {
    union {
        double lc[kMaxPool];        // [R*k] the rows' child log-confidences (R*k = P <= 1024)
        uint64_t sorted[kMaxPool];  // after the depth loop: each depth's best keys, descending
    } u;
    struct {
        int ctok[kMaxPool];  // [R*k] the rows' child tokens
    } v;
    double logv[kMaxPool];    // pool: log V
    uint64_t key[kMaxPool];   // pool: composite key
    int par[kMaxPool];        // pool: parent pool index (-1: the root)
    int row[kMaxPool];        // pool: draft row that expanded it, or -1
    int flat[kMaxPool];       // pool: rank within its depth; for a kept entry, then its flattened index
    int ptok[kMaxPool];       // pool: token
    int lent[kMaxPool];       // the rerank table: pool index of each sorted-list entry
    int fslot[kMaxSelDepth][16];  // frontier of each depth: pool index of slot s
    unsigned kbits[kMaxPool / 32];  // kept entries, one bit each
    int klist[64];                  // kept entries (m <= 63), in no particular order
    int nkept;
};

// Ranks of a depth's candidates within the depth (cnt <= 256 unique keys; rank = the number of
// keys above).  Each thread holds four consecutive candidates in registers and compares them with
// a strided slice of the keys, so every key read from shared memory serves four comparisons (the
// rank is bound by the bytes shared memory delivers, not by the comparisons).  The NS threads of
// a group cover the keys between them and sum their counts by shuffles, two counts packed in one
// word (each < 2^16).  Warps past the last group skip the count.  `done(i, rank)` runs in one
// thread per candidate.
template <int NS, typename F>
__device__ __forceinline__ void rank_blocked(const uint64_t *keys, int cnt, F &&done) {
    const int tid = threadIdx.x;
    const int groups = (cnt + 3) >> 2;
    if ((tid & ~31) >= groups * NS) return;  // warp-uniform
    const int g = tid / NS, sl = tid % NS;
    const int c0 = 4 * g;
    const uint64_t v0 = c0 < cnt ? keys[c0] : ~0ull, v1 = c0 + 1 < cnt ? keys[c0 + 1] : ~0ull;
    const uint64_t v2 = c0 + 2 < cnt ? keys[c0 + 2] : ~0ull, v3 = c0 + 3 < cnt ? keys[c0 + 3] : ~0ull;
    uint32_t n01 = 0, n23 = 0;  // counts of candidates 0, 1 (low, high half) and 2, 3
    for (int o = sl; o < cnt; o += NS) {
        const uint64_t kv = keys[o];
        n01 += (kv > v0 ? 1u : 0u) + (kv > v1 ? 0x10000u : 0u);
        n23 += (kv > v2 ? 1u : 0u) + (kv > v3 ? 0x10000u : 0u);
    }
#pragma unroll
    for (int x = 1; x < NS; x <<= 1) {
        n01 += __shfl_xor_sync(0xffffffffu, n01, x);
        n23 += __shfl_xor_sync(0xffffffffu, n23, x);
    }
    if (sl == 0 && g < groups) {
        if (c0 < cnt) done(c0, int(n01 & 0xffffu));
        if (c0 + 1 < cnt) done(c0 + 1, int(n01 >> 16));
        if (c0 + 2 < cnt) done(c0 + 2, int(n23 & 0xffffu));
        if (c0 + 3 < cnt) done(c0 + 3, int(n23 >> 16));
    }
}
template <typename F>
__device__ __forceinline__ void rank_depth(const uint64_t *keys, int cnt, F &&done) {
    const int groups = (cnt + 3) >> 2;
    if (groups * 32 <= kSelThreads) rank_blocked<32>(keys, cnt, done);
    else if (groups * 16 <= kSelThreads) rank_blocked<16>(keys, cnt, done);
    else rank_blocked<8>(keys, cnt, done);
}

// One CTA per sequence.  Depth by depth: every candidate's rank within its depth (counting, a
// group of threads per candidate), then the expansion of the k best (the frontier), each phase
// closed by a block barrier.  The rerank keeps the m largest keys of the pool: a key's rank in the
// pool is its rank within its depth plus, for every other depth, the number of that depth's keys
// above it, found by binary search in that depth's sorted list of its m best keys; only the
// entries of those lists can be kept.  Then the flatten (creation order) and the outputs.
__global__ void __launch_bounds__(kSelThreads) tree_select_kernel(SelectArgs a) {
    pdl_wait();
    pdl_launch_next();
    extern __shared__ __align__(16) unsigned char sel_smem_raw[];
    SelSmem &S = *reinterpret_cast<SelSmem *>(sel_smem_raw);

    const int b = blockIdx.x;
    const int tid = threadIdx.x;
    const int k = a.k, R = a.R, D = a.D, m = a.m;
    const int np = k + (D - 1) * k * k;  // pool size
    const int32_t rt = tid == 0 ? a.root_token[b] : 0;  // loaded now: only the outputs use it

    // the rows' children (written by the row kernel): every load in flight before the first store
    const int nload = R * k;
    {
        constexpr int kPer = kMaxPool / kSelThreads;
        double lcv[kPer];
        int tkv[kPer];
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
            const int i = tid + u * kSelThreads;
            if (i < nload) {
                lcv[u] = a.row_lc[size_t(b) * R * k + i];
                tkv[u] = a.row_tok[size_t(b) * R * k + i];
            }
        }
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
            const int i = tid + u * kSelThreads;
            if (i < nload) {
                S.u.lc[i] = lcv[u];
                S.v.ctok[i] = tkv[u];
            }
            if (i < np) S.row[i] = -1;
        }
    }
    if (tid < kMaxPool / 32) S.kbits[tid] = 0u;
    if (tid == 0) S.nkept = 0;
    __syncthreads();
    // depth 1: the root's children (row 0)
    for (int i = tid; i < k; i += kSelThreads) {
        S.logv[i] = S.u.lc[i];
        S.key[i] = pool_key(S.u.lc[i], i);
        S.ptok[i] = S.v.ctok[i];
        S.par[i] = -1;
    }
    __syncthreads();

    for (int f = 1; f <= D; ++f) {
        const int lb = depth_base(f, k), cnt = depth_count(f, k);
        // rank within the depth; a candidate of rank r < k is frontier slot r
        rank_depth(S.key + lb, cnt, [&](int i, int rank) {
            const int e = lb + i;
            S.flat[e] = rank;
            if (f < D && !a.slots && rank < k) {
                S.fslot[f][rank] = e;
                S.row[e] = 1 + (f - 1) * k + rank;
            }
        });
        __syncthreads();
        if (f == D) break;
        // expansion: child c of frontier slot s (expanded with draft row 1 + (f - 1)k + s) becomes
        // entry s k + c of depth f + 1
        const int nb = lb + cnt;
        const int32_t *slots_f = a.slots ? a.slots + (size_t(b) * D + f) * k : nullptr;
        for (int t = tid; t < k * k; t += kSelThreads) {
            const int s = t / k, c = t - s * k;
            const int rr = 1 + (f - 1) * k + s;
            int e;
            if (slots_f) {
                // the frontier chosen by an earlier call (stepwise build); an index outside this
                // depth's candidates (a stale or foreign state) is flagged and replaced by the
                // slot's own position
                e = slots_f[s];
                if (e < lb || e >= lb + cnt) {
                    if (c == 0) set_status(a.status, EAGLE_ERR_DEVICE_INPUT);
                    e = lb + s;
                }
                if (c == 0) S.row[e] = rr;
            } else {
                e = S.fslot[f][s];
            }
            const int ne = nb + t;
            const double lv = S.logv[e] + S.u.lc[rr * k + c];
            S.logv[ne] = lv;
            S.key[ne] = pool_key(lv, ne);
            S.ptok[ne] = S.v.ctok[rr * k + c];
            S.par[ne] = e;
        }
        __syncthreads();
    }

    // rerank table: each depth's min(count, m) best keys in descending order with their pool
    // indices; every entry of the table gets its rank in the pool, and those below m are kept
    const int k1 = min(k, m), kk = min(k * k, m);
    const int nlist = k1 + (D - 1) * kk;
    for (int e = tid; e < np; e += kSelThreads) {
        const int r = S.flat[e];
        if (r < m) {
            const int idx = list_base(depth_of(e, k), k, m) + r;
            S.u.sorted[idx] = S.key[e];
            S.lent[idx] = e;
        }
    }
    __syncthreads();
    for (int t = tid; t < nlist; t += kSelThreads) {
        const int d = t < k1 ? 1 : 2 + (t - k1) / kk;
        const uint64_t v = S.u.sorted[t];
        int g = t - list_base(d, k, m);
        // four depths' searches at a time, with unconditional loads from clamped indices so that
        // their shared-memory loads overlap (a depth past D, or the key's own depth, contributes
        // an empty list)
        for (int d2 = 1; d2 <= D && g < m; d2 += 4) {
            int len[4], pos[4] = {0, 0, 0, 0};
            const uint64_t *lst[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int dd = d2 + u;
                len[u] = (dd > D || dd == d) ? 0 : (dd == 1 ? k1 : kk);
                lst[u] = S.u.sorted + (dd <= D ? list_base(dd, k, m) : 0);
            }
#pragma unroll
            for (int step = 32; step > 0; step >>= 1)  // lists are descending, m <= 63
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const uint64_t kv = lst[u][max(min(pos[u] + step, len[u]) - 1, 0)];
                    pos[u] += (pos[u] + step <= len[u] && kv > v) ? step : 0;
                }
            g += (pos[0] + pos[1]) + (pos[2] + pos[3]);
        }
        if (g < m) {
            const int e = S.lent[t];
            atomicOr(&S.kbits[e >> 5], 1u << (e & 31));
            const int slot = atomicAdd(&S.nkept, 1);
            if (slot < 64) S.klist[slot] = e;
        }
    }
    __syncthreads();

    // flatten: flat index = 1 + number of kept entries created earlier (popcounts of the kept bits)
    const int nk = min(S.nkept, 64);
    auto kept_bit = [&](int e) { return (S.kbits[e >> 5] >> (e & 31)) & 1u; };
    for (int q = tid; q < nk; q += kSelThreads) {
        const int e = S.klist[q];
        int before = __popc(S.kbits[e >> 5] & ((1u << (e & 31)) - 1u));
        for (int w = 0; w < (e >> 5); ++w) before += __popc(S.kbits[w]);
        S.flat[e] = 1 + before;
    }
    __syncthreads();

    // outputs
    const int n = m + 1;
    int32_t *tokens = a.tokens + size_t(b) * n;
    int32_t *parents = a.parents + size_t(b) * n;
    int32_t *depths = a.depths + size_t(b) * n;
    int32_t *node_row = a.node_row + size_t(b) * n;
    uint64_t *mask = a.mask + size_t(b) * n;
    if (tid == 0) {
        if (rt < 0 || rt >= a.V) set_status(a.status, EAGLE_ERR_DEVICE_INPUT);
        tokens[0] = rt;
        parents[0] = -1;
        depths[0] = 0;
        node_row[0] = 0;
        mask[0] = 1ull;
        if (a.node_logv) a.node_logv[size_t(b) * n] = 0.f;
    }
    if (tid == 0 && S.nkept != m) set_status(a.status, EAGLE_ERR_DEVICE_INPUT);  // cannot happen: m distinct keys
    for (int q = tid; q < nk; q += kSelThreads) {
        const int e = S.klist[q];
        const int i = S.flat[e];
        const int pe = S.par[e];
        int pi = 0;
        if (pe >= 0) {
            pi = kept_bit(pe) ? S.flat[pe] : -1;
            if (pi < 0) {  // cannot happen for a consistent pool: the kept set is ancestor-closed
                set_status(a.status, EAGLE_ERR_DEVICE_INPUT);
                pi = 0;
            }
        }
        uint64_t bits = 1ull | (1ull << i);
        for (int anc = pe; anc >= 0; anc = S.par[anc])
            if (kept_bit(anc)) bits |= 1ull << S.flat[anc];
        tokens[i] = S.ptok[e];
        parents[i] = pi;
        depths[i] = depth_of(e, k);
        node_row[i] = S.row[e];
        mask[i] = bits;
        if (a.node_logv) a.node_logv[size_t(b) * n + i] = float(S.logv[e]);
    }
}

// ---- stepwise build: one depth's frontier --------------------------------------------------
// The candidates of depth hi are the root's children (hi = 1: row 0) or the children of the
// depth hi - 1 frontier that the previous step stored (its pool indices and log V in the
// workspace; slot s read row 1 + (hi - 2)k + s).  Their keys are the select kernel's: log V =
// the parent's log V + the child's log-confidence, creation index = the depth's pool offset
// (0 at depth 1, k + (d - 2)k^2 at depth d >= 2) + slot * k + child.  The k best are ranked by
// counting, stored (pool index, log V) for the next step and for the finalize replay, and
// returned (token, parent slot).
constexpr int kStepThreads = 256;
constexpr int kStepMax = 256;  // k^2 candidates, k <= 16

struct StepArgs {
    const int32_t *row_tok;  // [B][R][k]
    const double *row_lc;    // [B][R][k]
    int32_t *slots;          // [B][D][k] pool index of each frontier slot
    double *flogv;           // [B][D][k] log V of each frontier slot
    int32_t *front_tok, *front_par;  // [B][k]
    int D, k, R, hi;
};

__global__ void __launch_bounds__(kStepThreads) tree_step_kernel(StepArgs a) {
    pdl_wait();
    pdl_launch_next();
    __shared__ uint64_t s_key[kStepMax];
    __shared__ double s_lv[kStepMax];
    __shared__ int s_tok[kStepMax];
    const int b = blockIdx.x, tid = threadIdx.x, k = a.k, hi = a.hi, D = a.D;
    const int cnt = hi == 1 ? k : k * k;
    const int lb = hi == 1 ? 0 : k + (hi - 2) * k * k;
    const int r0 = hi == 1 ? 0 : 1 + (hi - 2) * k;
    for (int i = tid; i < cnt; i += kStepThreads) {
        const int sl = hi == 1 ? 0 : i / k, ch = hi == 1 ? i : i % k;
        const size_t o = (size_t(b) * a.R + r0 + sl) * k + ch;
        const double lc = a.row_lc[o];
        const double lv = hi == 1 ? lc : a.flogv[(size_t(b) * D + hi - 1) * k + sl] + lc;
        s_lv[i] = lv;
        s_key[i] = pool_key(lv, lb + i);
        s_tok[i] = a.row_tok[o];
    }
    __syncthreads();
    // rank by counting: two adjacent threads per candidate, each over one half
    for (int base = 0, half = (cnt + 1) >> 1; base < cnt; base += kStepThreads / 2) {
        const int i = base + (tid >> 1);
        const bool act = i < cnt;
        const uint64_t v = act ? s_key[i] : ~0ull;
        const int o0 = (tid & 1) * half, o1 = min(o0 + half, cnt);
        int r0c = 0, r1c = 0, r2c = 0, r3c = 0;
        int o = o0;
        for (; o + 4 <= o1; o += 4) {
            r0c += s_key[o] > v;
            r1c += s_key[o + 1] > v;
            r2c += s_key[o + 2] > v;
            r3c += s_key[o + 3] > v;
        }
        for (; o < o1; ++o) r0c += s_key[o] > v;
        const int part = (r0c + r1c) + (r2c + r3c);
        const int rank = part + __shfl_xor_sync(0xffffffffu, part, 1);
        if (act && !(tid & 1) && rank < k) {
            const size_t so = (size_t(b) * D + hi) * k + rank;
            a.slots[so] = lb + i;
            a.flogv[so] = s_lv[i];
            a.front_tok[size_t(b) * k + rank] = s_tok[i];
            a.front_par[size_t(b) * k + rank] = hi == 1 ? -1 : i / k;
        }
    }
}

// ---- static tree (EAGLE-1) and chain: a template of parent indices shared by the batch -------
// Page: "EAGLE: Speculative Sampling Requires Rethinking Feature Uncertainty", appendix A.1 (a
// fixed draft tree; greedy: a node's children are the top tokens of the draft distribution at
// it) and section 4.3.1 (the chain).  The template node p with children reads draft row
// row(p) = the number of such nodes before it; its children, in ascending index, take that row's
// tokens of rank 0, 1, ... (value desc, ties to the lower id).  log V = the sum of the
// log-confidences along the path.
struct StaticArgs {
    const int32_t *row_tok;  // [B][R][k]
    const double *row_lc;    // [B][R][k]
    const int32_t *root_token;
    int32_t *tokens, *parents, *depths, *node_row;
    uint64_t *mask;
    float *node_logv;
    int32_t *status;
    int n, k, R, V;
    int8_t tmpl[64];  // parents[i]; tmpl[0] = -1
};

__global__ void __launch_bounds__(64) static_tree_kernel(StaticArgs a) {
    pdl_wait();
    pdl_launch_next();
    __shared__ int s_internal[64], s_row[64], s_tok[64];
    __shared__ double s_lc[64];
    const int b = blockIdx.x, i = threadIdx.x, n = a.n;
    const int p = i < n ? a.tmpl[i] : -1;
    bool internal = false;
    for (int j = i + 1; j < n; ++j) internal |= a.tmpl[j] == i;
    s_internal[i] = internal;
    __syncthreads();
    int row = -1;
    if (internal) {
        row = 0;
        for (int j = 0; j < i; ++j) row += s_internal[j];
    }
    s_row[i] = row;
    __syncthreads();
    if (i == 0) {
        const int32_t rt = a.root_token[b];
        if (rt < 0 || rt >= a.V) set_status(a.status, EAGLE_ERR_DEVICE_INPUT);
        s_tok[0] = rt;
        s_lc[0] = 0.0;
    } else if (i < n) {
        int rank = 0;  // this node among its parent's children, in ascending index
        for (int j = p + 1; j < i; ++j) rank += a.tmpl[j] == p;
        const size_t o = (size_t(b) * a.R + s_row[p]) * a.k + rank;
        s_tok[i] = a.row_tok[o];
        s_lc[i] = a.row_lc[o];
    }
    __syncthreads();
    if (i >= n) return;
    double logv = 0.0;
    uint64_t bits = 1ull;
    int depth = 0;
    for (int q = i; q > 0; q = a.tmpl[q]) {
        logv += s_lc[q];
        bits |= 1ull << q;
        ++depth;
    }
    const size_t o = size_t(b) * n + i;
    a.tokens[o] = s_tok[i];
    a.parents[o] = p;
    a.depths[o] = depth;
    a.node_row[o] = s_row[i];
    a.mask[o] = bits;
    if (a.node_logv) a.node_logv[o] = float(logv);
}

// a1 over R rows of B sequences: each row's k children (token, fp64 log-confidence at tree_temp)
// into row_tok / row_lc [B][out_R][k] at rows out_r0 .. out_r0 + R - 1.  A row's slices are
// planned for `plan_rows` rows in all: the log normaliser's float sums depend on the slicing,
// so a stepwise build plans its partial calls like the one-call build to get the same bits.
eagle_status row_topk_launch(const float *draft, int B, int R, int V, int k, float tree_temp, int32_t *row_tok,
                             double *row_lc, int out_R, int out_r0, long plan_rows, cudaStream_t stream) {
    const int splits = splits_for_rows(plan_rows, V);
    int chunk = (V + splits - 1) / splits;
    chunk = (chunk + 3) & ~3;
    RowArgs ra;
    ra.x = draft;
    ra.row_tok = row_tok;
    ra.row_lc = row_lc;
    ra.V = V;
    ra.R = R;
    ra.k = k;
    ra.chunk = chunk;
    ra.out_R = out_R;
    ra.out_r0 = out_r0;
    ra.c = kLog2e / tree_temp;
    ra.inv_t = 1.0 / double(tree_temp);
    if (launch_pdl(row_topk_kernel, dim3(splits, R, B), dim3(kRowThreads), 0, stream, unsigned(splits), ra) !=
        cudaSuccess)
        return EAGLE_ERR_CUDA;
    note_launch();
    return EAGLE_OK;
}

// A row's k children: its top k (u == nullptr) or k draws with the uniforms u [B][R][k].  The
// draws are exact fixed-point decisions whatever the slicing, so only the top-k kernel takes the
// one-call plan (B * out_R rows).
eagle_status row_children_launch(const float *draft, const float *u, int B, int R, int V, int k, float tree_temp,
                                 int32_t *row_tok, double *row_lc, int out_R, int out_r0, int32_t *status,
                                 cudaStream_t stream) {
    if (u) return row_sample_launch(draft, u, B, R, V, k, tree_temp, row_tok, row_lc, out_R, out_r0, status, stream);
    return row_topk_launch(draft, B, R, V, k, tree_temp, row_tok, row_lc, out_R, out_r0, long(B) * out_R, stream);
}

// The build's workspace: status header | row_tok [B][R][k] | row_lc [B][R][k] | slots [B][D][k]
// (the frontier of every depth, kept between the calls of a stepwise build).
struct BuildWs {
    int32_t *status, *row_tok, *slots;
    double *row_lc, *flogv;
};
BuildWs build_ws(const eagle_tree_cfg &c, void *ws) {
    unsigned char *w = static_cast<unsigned char *>(ws);
    const size_t ent = size_t(c.batch) * (1 + (c.depth - 1) * c.topk) * c.topk;
    BuildWs r;
    r.status = reinterpret_cast<int32_t *>(w);
    r.row_tok = reinterpret_cast<int32_t *>(w + kWsHeader);
    r.row_lc = reinterpret_cast<double *>(w + kWsHeader + align_up(ent * 4, 256));
    const size_t sl = size_t(c.batch) * c.depth * c.topk;
    r.slots = reinterpret_cast<int32_t *>(w + kWsHeader + align_up(ent * 4, 256) + align_up(ent * 8, 256));
    r.flogv = reinterpret_cast<double *>(reinterpret_cast<unsigned char *>(r.slots) + align_up(sl * 4, 256));
    return r;
}

// The select kernel over the rows' children in the workspace; with `replay`, the frontiers the
// step kernel stored.
eagle_status select_launch(const eagle_tree_cfg &c, const BuildWs &w, const int32_t *root, int32_t *tokens,
                           int32_t *parents, int32_t *depths, int32_t *node_row, uint64_t *mask, float *node_logv,
                           bool replay, cudaStream_t stream) {
    SelectArgs sa;
    sa.row_tok = w.row_tok;
    sa.row_lc = w.row_lc;
    sa.root_token = root;
    sa.tokens = tokens;
    sa.parents = parents;
    sa.depths = depths;
    sa.node_row = node_row;
    sa.mask = mask;
    sa.node_logv = node_logv;
    sa.status = w.status;
    sa.V = c.vocab;
    sa.D = c.depth;
    sa.k = c.topk;
    sa.m = c.keep;
    sa.R = 1 + (c.depth - 1) * c.topk;
    sa.slots = replay ? w.slots : nullptr;
    static std::atomic<uint64_t> ready{0};
    if (once_per_device(ready, [] {
            return cudaFuncSetAttribute(tree_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        int(sizeof(SelSmem)));
        }) != cudaSuccess)
        return EAGLE_ERR_CUDA;
    if (launch_pdl(tree_select_kernel, dim3(c.batch), dim3(kSelThreads), sizeof(SelSmem), stream, 1u, sa) !=
        cudaSuccess)
        return EAGLE_ERR_CUDA;
    note_launch();
    return cudaPeekAtLastError() == cudaSuccess ? EAGLE_OK : EAGLE_ERR_CUDA;
}

}  // namespace

// One wave of CTAs: rows are split over a cluster only while the grid stays within the SM count
// (each CTA streams its slice with loads of the next batch in flight).
int splits_for_rows(long rows, int vocab) {
    long sp = device_sm_count() / rows;
    const long per = long(kRowThreads) * kRowVals;
    const long useful = (vocab + per - 1) / per;  // no empty CTAs
    if (sp > useful) sp = useful;
    if (sp > kMaxSplits) sp = kMaxSplits;
    return sp < 1 ? 1 : int(sp);
}

size_t static_tree_workspace_bytes(const eagle_static_tree_cfg &c, int R, int k) {
    const size_t ent = size_t(c.batch) * (R > 0 ? R : 1) * (k > 0 ? k : 1);
    return kWsHeader + align_up(ent * 4, 256) + align_up(ent * 8, 256);
}

eagle_status build_static_tree_launch(const eagle_static_tree_cfg &c, int R, int k, const float *draft,
                                      const float *child_u, const int32_t *root, int32_t *tokens, int32_t *parents,
                                      int32_t *depths, int32_t *node_row, uint64_t *mask, float *node_logv, void *ws,
                                      cudaStream_t stream) {
    unsigned char *w = static_cast<unsigned char *>(ws);
    const size_t ent = size_t(c.batch) * (R > 0 ? R : 1) * (k > 0 ? k : 1);
    StaticArgs a;
    a.row_tok = reinterpret_cast<int32_t *>(w + kWsHeader);
    a.row_lc = reinterpret_cast<double *>(w + kWsHeader + align_up(ent * 4, 256));
    if (R > 0) {
        if (eagle_status e = row_children_launch(draft, child_u, c.batch, R, c.vocab, k, c.tree_temp,
                                                 const_cast<int32_t *>(a.row_tok), const_cast<double *>(a.row_lc), R,
                                                 0, reinterpret_cast<int32_t *>(w), stream))
            return e;
    }
    a.root_token = root;
    a.tokens = tokens;
    a.parents = parents;
    a.depths = depths;
    a.node_row = node_row;
    a.mask = mask;
    a.node_logv = node_logv;
    a.status = reinterpret_cast<int32_t *>(w);
    a.n = c.nodes;
    a.k = k > 0 ? k : 1;
    a.R = R > 0 ? R : 1;
    a.V = c.vocab;
    for (int i = 0; i < 64; ++i) a.tmpl[i] = i < c.nodes ? c.parents[i] : int8_t(-1);
    if (launch_pdl(static_tree_kernel, dim3(c.batch), dim3(64), 0, stream, 1u, a) != cudaSuccess) return EAGLE_ERR_CUDA;
    note_launch();
    return cudaPeekAtLastError() == cudaSuccess ? EAGLE_OK : EAGLE_ERR_CUDA;
}

size_t build_tree_workspace_bytes(const eagle_tree_cfg &c) {
    const size_t ent = size_t(c.batch) * (1 + (c.depth - 1) * c.topk) * c.topk;
    const size_t sl = size_t(c.batch) * c.depth * c.topk;
    return kWsHeader + align_up(ent * 4, 256) + align_up(ent * 8, 256) + align_up(sl * 4, 256) +
           align_up(sl * 8, 256);
}

// The whole build in one call: every row's children (top k, or draws when child_u is set), then
// the select kernel over all depths.
eagle_status build_tree_launch(const eagle_tree_cfg &c, const float *draft, const float *child_u, const int32_t *root,
                               int32_t *tokens, int32_t *parents, int32_t *depths, int32_t *node_row, uint64_t *mask,
                               float *node_logv, void *ws, cudaStream_t stream) {
    const BuildWs w = build_ws(c, ws);
    const int R = 1 + (c.depth - 1) * c.topk;
    if (eagle_status e = row_children_launch(draft, child_u, c.batch, R, c.vocab, c.topk, c.tree_temp, w.row_tok,
                                             w.row_lc, R, 0, w.status, stream))
        return e;
    return select_launch(c, w, root, tokens, parents, depths, node_row, mask, node_logv, false, stream);
}

// Stepwise build, stage f (0 = begin: the root's row; f >= 1: the rows of the depth-f frontier).
// The rows' children go to rows 1 + (f-1)k .. of the workspace (row 0 for the root); then, while
// a deeper frontier is still to be expanded (f + 1 <= D - 1), the step kernel ranks depth f + 1
// from the stored depth-f frontier and writes the new frontier.
eagle_status build_step_launch(const eagle_tree_cfg &c, int f, const float *rows, const float *child_u,
                               int32_t *front_tok, int32_t *front_par, void *ws, cudaStream_t stream) {
    const BuildWs w = build_ws(c, ws);
    const int R = 1 + (c.depth - 1) * c.topk;
    const int nrows = f == 0 ? 1 : c.topk;
    const int r0 = f == 0 ? 0 : 1 + (f - 1) * c.topk;
    if (eagle_status e = row_children_launch(rows, child_u, c.batch, nrows, c.vocab, c.topk, c.tree_temp, w.row_tok,
                                             w.row_lc, R, r0, w.status, stream))
        return e;
    if (f + 1 > c.depth - 1) return cudaPeekAtLastError() == cudaSuccess ? EAGLE_OK : EAGLE_ERR_CUDA;
    StepArgs sa;
    sa.row_tok = w.row_tok;
    sa.row_lc = w.row_lc;
    sa.slots = w.slots;
    sa.flogv = w.flogv;
    sa.front_tok = front_tok;
    sa.front_par = front_par;
    sa.D = c.depth;
    sa.k = c.topk;
    sa.R = R;
    sa.hi = f + 1;
    if (launch_pdl(tree_step_kernel, dim3(c.batch), dim3(kStepThreads), 0, stream, 1u, sa) != cudaSuccess)
        return EAGLE_ERR_CUDA;
    note_launch();
    return cudaPeekAtLastError() == cudaSuccess ? EAGLE_OK : EAGLE_ERR_CUDA;
}

// Stepwise build, last stage: the select kernel over the stored rows and frontiers.
eagle_status build_finalize_launch(const eagle_tree_cfg &c, const int32_t *root, int32_t *tokens, int32_t *parents,
                                   int32_t *depths, int32_t *node_row, uint64_t *mask, float *node_logv, void *ws,
                                   cudaStream_t stream) {
    const BuildWs w = build_ws(c, ws);
    return select_launch(c, w, root, tokens, parents, depths, node_row, mask, node_logv, true, stream);
}

}  // namespace eagle
