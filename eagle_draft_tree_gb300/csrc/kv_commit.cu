// kv_commit.cu -- append each sequence's committed tree nodes to its KV cache (sm_103a).
//
// Pages: "LLM speculative decoding explained" (hubwiz.com) section 1 (a round commits the accepted
// draft tokens and one more token) and section 5 (the flattened tree is scored in one target pass,
// node i at position ctx + depth(i), so that pass computed every node's keys and values); "EAGLE:
// Speculative Sampling Requires Rethinking Feature Uncertainty" section 3.3 (the accepted path runs
// from the root along accepted children).
//
// The cache of sequence b gains the root (node 0, at position ctx_b) and then the accepted nodes
// in path order (path entry i at ctx_b + 1 + i): out_len[b] rows in all.  The last committed token
// has no keys or values yet; it is the next round's root.  New length: ctx_b + out_len[b].
//
// One CTA per (layer, sequence): thread 0 validates the sequence's path and publishes the source
// rows; every thread then moves 16-byte words of the K and V rows.  The work is a few KB per CTA,
// so the kernel is bound by latency, not by HBM.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace eagle {

namespace {

constexpr int kCommitThreads = 256;
constexpr int kMaxRows = 64;  // n <= 64, so at most 64 committed rows

struct KvCommitArgs {
    const unsigned char *k_tree, *v_tree;  // [L][B][n][Hkv][d]
    const int32_t *out_path;               // [B][D]
    const int32_t *out_len, *ctx_len;      // [B]
    unsigned char *k_cache, *v_cache;      // [L][B][S_max][Hkv][d]
    int32_t *new_ctx_len;                  // [B]
    int32_t *status;
    int L, B, n, S_max, D;
    int row_words;  // 16-byte words per row: Hkv * d * element size / 16
};

__global__ void __launch_bounds__(kCommitThreads) kv_commit_kernel(KvCommitArgs a) {
    pdl_wait();
    pdl_launch_next();
    __shared__ int s_node[kMaxRows];
    __shared__ int s_len, s_ctx;
    const int l = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
    if (tid == 0) {
        const int len = a.out_len[b], ctx = a.ctx_len[b];
        bool ok = len >= 1 && len <= a.D + 1 && len <= kMaxRows && ctx >= 0 && ctx <= a.S_max - len;
        s_node[0] = 0;
        for (int i = 1; ok && i < len; ++i) {
            const int node = a.out_path[size_t(b) * a.D + i - 1];
            ok = node >= 1 && node < a.n;
            s_node[i] = node;
        }
        s_len = ok ? len : 0;
        s_ctx = ctx;
        if (l == 0) {
            a.new_ctx_len[b] = ok ? ctx + len : ctx;
            if (!ok && len != 0) set_status(a.status, EAGLE_ERR_DEVICE_INPUT);
        }
    }
    __syncthreads();
    const int len = s_len, ctx = s_ctx, W = a.row_words;
    const size_t rowb = size_t(W) * 16;
    const unsigned char *kt = a.k_tree + (size_t(l) * a.B + b) * a.n * rowb;
    const unsigned char *vt = a.v_tree + (size_t(l) * a.B + b) * a.n * rowb;
    unsigned char *kc = a.k_cache + ((size_t(l) * a.B + b) * a.S_max + ctx) * rowb;
    unsigned char *vc = a.v_cache + ((size_t(l) * a.B + b) * a.S_max + ctx) * rowb;
    // words of row i: [i * W, (i + 1) * W); K words first, then V words
    for (int w = tid; w < 2 * len * W; w += kCommitThreads) {
        const bool isv = w >= len * W;
        const int ww = isv ? w - len * W : w;
        const int i = ww / W, c = ww % W;
        const uint4 *src = reinterpret_cast<const uint4 *>((isv ? vt : kt) + size_t(s_node[i]) * rowb) + c;
        uint4 *dst = reinterpret_cast<uint4 *>((isv ? vc : kc) + size_t(i) * rowb) + c;
        *dst = __ldg(src);
    }
}

}  // namespace

eagle_status kv_commit_launch(const eagle_attn_cfg &c, int depth, const void *k_tree, const void *v_tree,
                              const int32_t *out_path, const int32_t *out_len, const int32_t *ctx_len,
                              void *k_cache, void *v_cache, int32_t *new_ctx_len, void *ws, cudaStream_t stream) {
    KvCommitArgs a;
    a.k_tree = static_cast<const unsigned char *>(k_tree);
    a.v_tree = static_cast<const unsigned char *>(v_tree);
    a.out_path = out_path;
    a.out_len = out_len;
    a.ctx_len = ctx_len;
    a.k_cache = static_cast<unsigned char *>(k_cache);
    a.v_cache = static_cast<unsigned char *>(v_cache);
    a.new_ctx_len = new_ctx_len;
    a.status = static_cast<int32_t *>(ws);
    a.L = c.layers;
    a.B = c.batch;
    a.n = c.nodes;
    a.S_max = c.max_seq;
    a.D = depth;
    const int es = c.dtype == EAGLE_DTYPE_BF16 ? 2 : 4;
    a.row_words = c.heads_kv * c.head_dim * es / 16;
    if (launch_pdl(kv_commit_kernel, dim3(c.layers, c.batch), dim3(kCommitThreads), 0, stream, 1u, a) != cudaSuccess)
        return EAGLE_ERR_CUDA;
    note_launch();
    return cudaPeekAtLastError() == cudaSuccess ? EAGLE_OK : EAGLE_ERR_CUDA;
}

}  // namespace eagle
