// build_tree.cu -- EAGLE-2 dynamic draft-tree build on sm_103a.
//
// Page: "(EAGLE 2) EAGLE-2: Faster Inference of Language Models with Dynamic Draft Trees",
// sections "Expanding the Draft Tree" (V_i = product of draft confidences on the root->i path;
// only the k most valuable nodes of a depth are expanded), "Rerank draft tokens" (top-m by V over
// every candidate, shallower first on equal V, so the kept set is still a connected tree) and
// "Tree Attention Mask" (flattened sequence, ancestors-only visibility).
//
// Two kernels:
//   row_topk_kernel   one HBM pass over every draft row: online log-sum-exp of x/T and the row's
//                     top-k logits (value desc, token asc).  A row is split across several CTAs
//                     so that the grid covers the GPU even at batch 1; each CTA leaves a partial
//                     (max, scaled sum, its top-KMAX keys) in the workspace.
//   tree_select_kernel one CTA per sequence: merges the partials, computes the log-confidences
//                     in fp64, runs the per-depth frontier selection, the global rerank (bitonic
//                     sort of the <= 1024-entry pool) and writes the flattened tree.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "common.cuh"

namespace eagle {

namespace {

constexpr int kRowThreads = 256;
constexpr int kSelThreads = 512;
constexpr int kMaxPool = 1024;

template <int KMAX>
__device__ __forceinline__ void list_insert(uint64_t (&list)[KMAX], uint64_t key) {
    if (key <= list[KMAX - 1]) return;
    list[KMAX - 1] = key;
#pragma unroll
    for (int j = KMAX - 1; j > 0; --j) {
        if (list[j] > list[j - 1]) {
            uint64_t t = list[j];
            list[j] = list[j - 1];
            list[j - 1] = t;
        }
    }
}

// Merge (m_a, s_a) and (m_b, s_b) where s = sum 2^((x - m) c).
__device__ __forceinline__ void ms_merge(float &m, float &s, float mo, float so, float c) {
    float M = fmaxf(m, mo);
    if (M == -INFINITY) return;
    float a = (m == -INFINITY) ? 0.f : s * exp2f((m - M) * c);
    float b = (mo == -INFINITY) ? 0.f : so * exp2f((mo - M) * c);
    m = M;
    s = a + b;
}

template <int KMAX>
__global__ void __launch_bounds__(kRowThreads) row_topk_kernel(const float *__restrict__ x, int V, int R, int splits,
                                                                 int chunk, float c, uint64_t *__restrict__ part_keys,
                                                                 float2 *__restrict__ part_ms) {
    __shared__ uint64_t s_lists[kRowThreads][KMAX + 1];  // +1 breaks bank alignment
    __shared__ uint64_t s_warp[kRowThreads / 32][KMAX];
    __shared__ float2 s_ms[kRowThreads / 32];

    const int split = blockIdx.x, r = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x;
    const float *row = x + (size_t(b) * R + r) * size_t(V);
    const int lo = split * chunk;
    const int hi = min(V, lo + chunk);

    float m = -INFINITY, s = 0.f;
    uint64_t list[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; ++j) list[j] = 0;

    auto consume = [&](float v, int t) {
        if (v > m) {
            s = s * exp2f((m - v) * c) + 1.f;
            m = v;
        } else {
            s += exp2f((v - m) * c);
        }
        list_insert<KMAX>(list, topk_key(v, uint32_t(t)));
    };

    const bool vec = ((V & 3) == 0) && ((reinterpret_cast<uintptr_t>(row) & 15) == 0);
    if (vec) {
        const float4 *row4 = reinterpret_cast<const float4 *>(row);
        const int lo4 = lo >> 2, hi4 = hi >> 2;
        int i = lo4 + tid;
        for (; i + 3 * kRowThreads < hi4; i += 4 * kRowThreads) {
            float4 a0 = __ldg(row4 + i);
            float4 a1 = __ldg(row4 + i + kRowThreads);
            float4 a2 = __ldg(row4 + i + 2 * kRowThreads);
            float4 a3 = __ldg(row4 + i + 3 * kRowThreads);
            const float4 av[4] = {a0, a1, a2, a3};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                int t = 4 * (i + u * kRowThreads);
                consume(av[u].x, t);
                consume(av[u].y, t + 1);
                consume(av[u].z, t + 2);
                consume(av[u].w, t + 3);
            }
        }
        for (; i < hi4; i += kRowThreads) {
            float4 a = __ldg(row4 + i);
            int t = 4 * i;
            consume(a.x, t);
            consume(a.y, t + 1);
            consume(a.z, t + 2);
            consume(a.w, t + 3);
        }
    } else {
        for (int t = lo + tid; t < hi; t += kRowThreads) consume(__ldg(row + t), t);
    }

    // (max, sum) across the block
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        float mo = __shfl_xor_sync(0xffffffffu, m, off);
        float so = __shfl_xor_sync(0xffffffffu, s, off);
        ms_merge(m, s, mo, so, c);
    }
    const int warp = tid >> 5, lane = tid & 31;
    if (lane == 0) s_ms[warp] = make_float2(m, s);

    // top-KMAX across the block: lanes -> warp lists -> block list
#pragma unroll
    for (int j = 0; j < KMAX; ++j) s_lists[tid][j] = list[j];
    __syncwarp();
    {
        int ptr = 0;
        for (int j = 0; j < KMAX; ++j) {
            uint64_t mine = ptr < KMAX ? s_lists[tid][ptr] : 0;
            uint64_t best = warp_max_u64(mine);
            if (best != 0 && mine == best) ++ptr;
            if (lane == 0) s_warp[warp][j] = best;
        }
    }
    __syncthreads();
    if (warp == 0) {
        float mm = lane < kRowThreads / 32 ? s_ms[lane].x : -INFINITY;
        float ss = lane < kRowThreads / 32 ? s_ms[lane].y : 0.f;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            float mo = __shfl_xor_sync(0xffffffffu, mm, off);
            float so = __shfl_xor_sync(0xffffffffu, ss, off);
            ms_merge(mm, ss, mo, so, c);
        }
        const size_t slot = (size_t(b) * R + r) * splits + split;
        int ptr = 0;
        for (int j = 0; j < KMAX; ++j) {
            uint64_t mine = (lane < kRowThreads / 32 && ptr < KMAX) ? s_warp[lane][ptr] : 0;
            uint64_t best = warp_max_u64(mine);
            if (best != 0 && mine == best) ++ptr;
            if (lane == 0) part_keys[slot * KMAX + j] = best;
        }
        if (lane == 0) part_ms[slot] = make_float2(mm, ss);
    }
}

struct PoolEntry {
    double logv;
    int idx;  // creation index (pool position)
    int pad;
};

// a comes strictly before b in (logv desc, creation asc)
__device__ __forceinline__ bool entry_before(const PoolEntry &a, const PoolEntry &b) {
    return a.logv > b.logv || (a.logv == b.logv && a.idx < b.idx);
}

struct SelectArgs {
    const uint64_t *part_keys;
    const float2 *part_ms;
    const int32_t *root_token;
    int32_t *tokens, *parents, *depths, *node_row;
    uint64_t *mask;
    float *node_logv;
    int32_t *status;
    int V, D, k, m, R, splits;
    float c;        // log2(e) / tree_temp
    double inv_t;   // 1 / tree_temp
};

template <int KMAX>
__global__ void __launch_bounds__(kSelThreads) tree_select_kernel(SelectArgs a) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const int b = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int k = a.k, R = a.R, D = a.D, m = a.m;
    const int P = k + (D - 1) * k * k;
    int NP = 1;
    while (NP < P) NP <<= 1;

    // shared layout
    double *s_lc = reinterpret_cast<double *>(smem_raw);                 // [R*k] child log-confidence
    PoolEntry *s_sort = reinterpret_cast<PoolEntry *>(s_lc + kMaxPool);  // [NP <= kMaxPool]
    double *s_logv = reinterpret_cast<double *>(s_sort + kMaxPool);      // [P]
    int *s_tok = reinterpret_cast<int *>(s_logv + kMaxPool);             // [R*k] child token
    int *s_ptok = s_tok + kMaxPool;                                      // [P] token
    int *s_par = s_ptok + kMaxPool;                                      // [P] parent pool idx
    int *s_row = s_par + kMaxPool;                                       // [P] expanding row or -1
    int *s_dep = s_row + kMaxPool;                                       // [P] depth
    int *s_flat = s_dep + kMaxPool;                                      // [P] flattened index or -1
    int *s_slot = s_flat + kMaxPool;                                     // [k] frontier slot -> pool idx
    int *s_wsum = s_slot + 16;                                           // [32] scan scratch

    // 1. merge the row partials: lse in fp64 and the top-k children
    for (int r = warp; r < R; r += kSelThreads / 32) {
        const size_t base = (size_t(b) * R + r) * a.splits;
        float M = -INFINITY;
        for (int s = lane; s < a.splits; s += 32) M = fmaxf(M, a.part_ms[base + s].x);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
        double S = 0.0;
        for (int s = lane; s < a.splits; s += 32) {
            float2 ms = a.part_ms[base + s];
            if (ms.x != -INFINITY) S += double(ms.y) * double(exp2f((ms.x - M) * a.c));
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) S += __shfl_xor_sync(0xffffffffu, S, off);
        double lse = 0.0;
        if (lane == 0) lse = double(M) * a.inv_t + log(S);
        lse = __shfl_sync(0xffffffffu, lse, 0);
        // top-k of the union of the split lists: pass j takes the largest key below pass j-1's
        const int ncand = a.splits * KMAX;
        const uint64_t *cand = a.part_keys + base * KMAX;
        uint64_t prev = ~uint64_t(0);
        for (int j = 0; j < k; ++j) {
            uint64_t best = 0;
            for (int i = lane; i < ncand; i += 32) {
                uint64_t key = cand[i];
                if (key < prev && key > best) best = key;
            }
            best = warp_max_u64(best);
            prev = best;
            if (lane == 0) {
                s_tok[r * k + j] = int(topk_key_token(best));
                s_lc[r * k + j] = double(topk_key_value(best)) * a.inv_t - lse;
            }
        }
    }
    __syncthreads();

    // 2. depth 1: the root's children (row 0)
    for (int i = tid; i < k; i += kSelThreads) {
        s_logv[i] = s_lc[i];
        s_ptok[i] = s_tok[i];
        s_par[i] = -1;
        s_row[i] = -1;
        s_dep[i] = 1;
    }
    __syncthreads();

    // 3. depths 2..D: expand the top-k frontier of the previous depth
    int lb = 0, cnt = k, np = k;
    for (int f = 1; f <= D - 1; ++f) {
        for (int e = lb + tid; e < lb + cnt; e += kSelThreads) {
            const double v = s_logv[e];
            int rank = 0;
            for (int o = lb; o < lb + cnt; ++o) {
                const double w = s_logv[o];
                rank += (w > v) || (w == v && o < e);
            }
            if (rank < k) {
                s_slot[rank] = e;
                s_row[e] = 1 + (f - 1) * k + rank;
            }
        }
        __syncthreads();
        const int nf = cnt < k ? cnt : k;
        for (int i = tid; i < nf * k; i += kSelThreads) {
            const int s = i / k, r = i % k;
            const int par = s_slot[s];
            const int rr = 1 + (f - 1) * k + s;
            const int e = np + i;
            s_logv[e] = s_logv[par] + s_lc[rr * k + r];
            s_ptok[e] = s_tok[rr * k + r];
            s_par[e] = par;
            s_row[e] = -1;
            s_dep[e] = f + 1;
        }
        __syncthreads();
        lb = np;
        cnt = nf * k;
        np += nf * k;
    }

    // 4. rerank: bitonic sort of the pool by (logv desc, creation asc)
    for (int i = tid; i < NP; i += kSelThreads) {
        PoolEntry pe;
        pe.logv = i < np ? s_logv[i] : -INFINITY;
        pe.idx = i;
        pe.pad = 0;
        s_sort[i] = pe;
        s_flat[i] = -1;
    }
    __syncthreads();
    for (int kk = 2; kk <= NP; kk <<= 1) {
        for (int j = kk >> 1; j > 0; j >>= 1) {
            for (int i = tid; i < NP; i += kSelThreads) {
                const int ixj = i ^ j;
                if (ixj > i) {
                    PoolEntry x0 = s_sort[i], x1 = s_sort[ixj];
                    const bool first_half = (i & kk) == 0;
                    // first_half: ascending position = better first
                    const bool swap = first_half ? entry_before(x1, x0) : entry_before(x0, x1);
                    if (swap) {
                        s_sort[i] = x1;
                        s_sort[ixj] = x0;
                    }
                }
            }
            __syncthreads();
        }
    }
    // kept flags live in s_flat (1 = kept) until the scan below
    for (int i = tid; i < m; i += kSelThreads) s_flat[s_sort[i].idx] = 1;
    __syncthreads();

    // 5. flatten: flat index = 1 + number of kept entries created earlier
    {
        const int nchunks = (np + 31) / 32;
        for (int ch = warp; ch < nchunks; ch += kSelThreads / 32) {
            const int e = ch * 32 + lane;
            const bool kept = e < np && s_flat[e] == 1;
            const unsigned bal = __ballot_sync(0xffffffffu, kept);
            if (lane == 0) s_wsum[ch] = __popc(bal);
        }
        __syncthreads();
        if (warp == 0) {
            int v = lane < nchunks ? s_wsum[lane] : 0;
            int incl = v;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                int o = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += o;
            }
            if (lane < nchunks) s_wsum[lane] = incl - v;  // exclusive
        }
        __syncthreads();
        for (int ch = warp; ch < nchunks; ch += kSelThreads / 32) {
            const int e = ch * 32 + lane;
            const bool kept = e < np && s_flat[e] == 1;
            const unsigned bal = __ballot_sync(0xffffffffu, kept);
            const int before = __popc(bal & ((1u << lane) - 1u));
            if (e < np) s_flat[e] = kept ? 1 + s_wsum[ch] + before : -1;
        }
        __syncthreads();
    }

    // 6. outputs
    const int n = m + 1;
    int32_t *tokens = a.tokens + size_t(b) * n;
    int32_t *parents = a.parents + size_t(b) * n;
    int32_t *depths = a.depths + size_t(b) * n;
    int32_t *node_row = a.node_row + size_t(b) * n;
    uint64_t *mask = a.mask + size_t(b) * n;
    if (tid == 0) {
        int32_t rt = a.root_token[b];
        if (rt < 0 || rt >= a.V) set_status(a.status, EAGLE_ERR_DEVICE_INPUT);
        tokens[0] = rt;
        parents[0] = -1;
        depths[0] = 0;
        node_row[0] = 0;
        mask[0] = 1ull;
        if (a.node_logv) a.node_logv[size_t(b) * n] = 0.f;
    }
    for (int e = tid; e < np; e += kSelThreads) {
        const int i = s_flat[e];
        if (i < 0) continue;
        const int pe = s_par[e];
        int pi = 0;
        if (pe >= 0) {
            pi = s_flat[pe];
            if (pi < 0) {  // cannot happen for a consistent pool: the kept set is ancestor-closed
                set_status(a.status, EAGLE_ERR_DEVICE_INPUT);
                pi = 0;
            }
        }
        uint64_t bits = 1ull | (1ull << i);
        for (int anc = pe; anc >= 0; anc = s_par[anc]) {
            const int fi = s_flat[anc];
            if (fi > 0) bits |= 1ull << fi;
        }
        tokens[i] = s_ptok[e];
        parents[i] = pi;
        depths[i] = s_dep[e];
        node_row[i] = s_row[e];
        mask[i] = bits;
        if (a.node_logv) a.node_logv[size_t(b) * n + i] = float(s_logv[e]);
    }
}

constexpr size_t select_smem_bytes() {
    return size_t(kMaxPool) * sizeof(double)       // s_lc
           + size_t(kMaxPool) * sizeof(PoolEntry)  // s_sort
           + size_t(kMaxPool) * sizeof(double)     // s_logv
           + size_t(kMaxPool) * sizeof(int) * 6    // s_tok .. s_flat
           + 16 * sizeof(int) + 32 * sizeof(int);
}

int kmax_for(int k) { return k <= 4 ? 4 : (k <= 8 ? 8 : 16); }

int splits_for(const eagle_tree_cfg &c) {
    const int R = 1 + (c.depth - 1) * c.topk;
    const long rows = long(c.batch) * R;
    const int want = int((4L * 152 + rows - 1) / rows);
    const int cap = c.vocab / 2048 > 1 ? c.vocab / 2048 : 1;
    int s = want < cap ? want : cap;
    if (s > 32) s = 32;
    return s < 1 ? 1 : s;
}

template <int KMAX>
cudaError_t launch_select_attr() {
    static bool done = false;  // set once per process; the attribute is per function
    if (done) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(tree_select_kernel<KMAX>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(select_smem_bytes()));
    if (e == cudaSuccess) done = true;
    return e;
}

template <int KMAX>
eagle_status launch_build(const eagle_tree_cfg &c, const float *draft, const int32_t *root, int32_t *tokens,
                          int32_t *parents, int32_t *depths, int32_t *node_row, uint64_t *mask, float *node_logv,
                          unsigned char *ws, cudaStream_t stream) {
    const int R = 1 + (c.depth - 1) * c.topk;
    const int splits = splits_for(c);
    int chunk = (c.vocab + splits - 1) / splits;
    chunk = (chunk + 3) & ~3;
    int32_t *status = reinterpret_cast<int32_t *>(ws);
    uint64_t *part_keys = reinterpret_cast<uint64_t *>(ws + kWsHeader);
    const size_t nslots = size_t(c.batch) * R * splits;
    float2 *part_ms = reinterpret_cast<float2 *>(ws + kWsHeader + align_up(nslots * KMAX * sizeof(uint64_t), 256));
    const float cexp = kLog2e / c.tree_temp;

    if (launch_select_attr<KMAX>() != cudaSuccess) return EAGLE_ERR_CUDA;
    dim3 g1(splits, R, c.batch);
    row_topk_kernel<KMAX><<<g1, kRowThreads, 0, stream>>>(draft, c.vocab, R, splits, chunk, cexp, part_keys, part_ms);
    note_launch();
    SelectArgs a;
    a.part_keys = part_keys;
    a.part_ms = part_ms;
    a.root_token = root;
    a.tokens = tokens;
    a.parents = parents;
    a.depths = depths;
    a.node_row = node_row;
    a.mask = mask;
    a.node_logv = node_logv;
    a.status = status;
    a.V = c.vocab;
    a.D = c.depth;
    a.k = c.topk;
    a.m = c.keep;
    a.R = R;
    a.splits = splits;
    a.c = cexp;
    a.inv_t = 1.0 / double(c.tree_temp);
    tree_select_kernel<KMAX><<<c.batch, kSelThreads, select_smem_bytes(), stream>>>(a);
    note_launch();
    return cudaPeekAtLastError() == cudaSuccess ? EAGLE_OK : EAGLE_ERR_CUDA;
}

}  // namespace

size_t build_tree_workspace_bytes(const eagle_tree_cfg &c) {
    const int R = 1 + (c.depth - 1) * c.topk;
    const int splits = splits_for(c);
    const size_t nslots = size_t(c.batch) * R * splits;
    const int kmax = kmax_for(c.topk);
    return kWsHeader + align_up(nslots * kmax * sizeof(uint64_t), 256) + align_up(nslots * sizeof(float2), 256);
}

eagle_status build_tree_launch(const eagle_tree_cfg &c, const float *draft, const int32_t *root, int32_t *tokens,
                               int32_t *parents, int32_t *depths, int32_t *node_row, uint64_t *mask,
                               float *node_logv, void *ws, cudaStream_t stream) {
    unsigned char *w = static_cast<unsigned char *>(ws);
    switch (kmax_for(c.topk)) {
        case 4: return launch_build<4>(c, draft, root, tokens, parents, depths, node_row, mask, node_logv, w, stream);
        case 8: return launch_build<8>(c, draft, root, tokens, parents, depths, node_row, mask, node_logv, w, stream);
        default:
            return launch_build<16>(c, draft, root, tokens, parents, depths, node_row, mask, node_logv, w, stream);
    }
}

}  // namespace eagle
