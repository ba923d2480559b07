// capi.cu -- the extern "C" entry points of libeagle: argument validation on the host, then the
// kernel launches of build_tree.cu, tree_attention.cu and verify.cu.  No entry point allocates
// memory or synchronises the stream (except eagle_get_device_status, which exists to read back).
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace eagle {

size_t build_tree_workspace_bytes(const eagle_tree_cfg &c);
eagle_status build_tree_launch(const eagle_tree_cfg &c, const float *draft, const float *child_u, const int32_t *root,
                               int32_t *tokens, int32_t *parents, int32_t *depths, int32_t *node_row, uint64_t *mask,
                               float *node_logv, void *ws, cudaStream_t stream);
eagle_status build_step_launch(const eagle_tree_cfg &c, int f, const float *rows, const float *child_u,
                               int32_t *front_tok, int32_t *front_par, void *ws, cudaStream_t stream);
eagle_status build_finalize_launch(const eagle_tree_cfg &c, const int32_t *root, int32_t *tokens, int32_t *parents,
                                   int32_t *depths, int32_t *node_row, uint64_t *mask, float *node_logv, void *ws,
                                   cudaStream_t stream);
size_t row_sample_max_vocab();
eagle_status exp2_error_launch(float *out, cudaStream_t stream);
size_t tree_attention_workspace_bytes(const eagle_attn_cfg &c);
eagle_status tree_attention_launch(const eagle_attn_cfg &c, const void *q, const void *k_cache, const void *v_cache,
                                   const int32_t *ctx_len, const void *k_tree, const void *v_tree,
                                   const uint64_t *mask, void *out, void *ws, cudaStream_t stream);
size_t tree_verify_workspace_bytes(const eagle_verify_cfg &c);
eagle_status tree_verify_launch(const eagle_verify_cfg &c, const float *target, const float *draft,
                                const int32_t *tokens, const int32_t *parents, const int32_t *node_row,
                                const float *uniforms, int32_t *out_tokens, int32_t *out_len, int32_t *out_path,
                                float *out_ratio, void *ws, cudaStream_t stream);
size_t verify_max_vocab();
size_t static_tree_workspace_bytes(const eagle_static_tree_cfg &c, int R, int k);
eagle_status build_static_tree_launch(const eagle_static_tree_cfg &c, int R, int k, const float *draft,
                                      const float *child_u, const int32_t *root, int32_t *tokens, int32_t *parents,
                                      int32_t *depths, int32_t *node_row, uint64_t *mask, float *node_logv, void *ws,
                                      cudaStream_t stream);
eagle_status kv_commit_launch(const eagle_attn_cfg &c, int depth, const void *k_tree, const void *v_tree,
                              const int32_t *out_path, const int32_t *out_len, const int32_t *ctx_len,
                              void *k_cache, void *v_cache, int32_t *new_ctx_len, void *ws, cudaStream_t stream);

static thread_local int32_t t_launches = 0;
void note_launch() { ++t_launches; }
void reset_launches() { t_launches = 0; }

int device_sm_count() {
    constexpr int kDefault = 152;
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
        cudaGetLastError();  // a host without a device: clear the error, use the default
        return kDefault;
    }
    if (dev < 64) {
        const int c = cache[dev].load(std::memory_order_relaxed);
        if (c > 0) return c;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) {
        cudaGetLastError();
        return kDefault;
    }
    if (dev < 64) cache[dev].store(n, std::memory_order_relaxed);
    return n;
}

namespace {

bool aligned256(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 255u) == 0; }

// 0 = ok, else an eagle status
int check_tree(const eagle_tree_cfg *c) {
    if (!c) return EAGLE_ERR_INVALID_ARG;
    if (c->batch < 1 || c->vocab < 1 || c->depth < 1 || c->topk < 1 || c->keep < 1) return EAGLE_ERR_INVALID_ARG;
    if (!(c->tree_temp > 0.f)) return EAGLE_ERR_INVALID_ARG;
    if (c->topk > c->vocab) return EAGLE_ERR_INVALID_ARG;
    if (c->topk > 16) return EAGLE_ERR_UNSUPPORTED;
    if (c->depth > 64) return EAGLE_ERR_UNSUPPORTED;
    const long P = long(c->topk) + long(c->depth - 1) * c->topk * c->topk;
    if (c->keep > P) return EAGLE_ERR_INVALID_ARG;
    if (P > 1024) return EAGLE_ERR_UNSUPPORTED;
    if (c->keep + 1 > 64) return EAGLE_ERR_UNSUPPORTED;
    return 0;
}

int check_attn(const eagle_attn_cfg *c) {
    if (!c) return EAGLE_ERR_INVALID_ARG;
    if (c->batch < 1 || c->layers < 1 || c->nodes < 1 || c->heads_q < 1 || c->heads_kv < 1 || c->head_dim < 1 ||
        c->max_seq < 0)
        return EAGLE_ERR_INVALID_ARG;
    if (c->dtype != EAGLE_DTYPE_BF16 && c->dtype != EAGLE_DTYPE_F32) return EAGLE_ERR_INVALID_ARG;
    if (!(c->scale >= 0.f)) return EAGLE_ERR_INVALID_ARG;
    if (c->heads_q % c->heads_kv) return EAGLE_ERR_UNSUPPORTED;
    if (c->head_dim != 64 && c->head_dim != 128) return EAGLE_ERR_UNSUPPORTED;
    if (c->nodes > 64) return EAGLE_ERR_UNSUPPORTED;
    const long rows = long(c->heads_q / c->heads_kv) * c->nodes;
    const long grid = long(c->layers) * c->batch * c->heads_kv * ((rows + 63) / 64);
    if (grid > 0x7fffffffL) return EAGLE_ERR_UNSUPPORTED;
    return 0;
}

// 0 = ok, else an eagle status; R = template nodes with children, k = most children of one node
int check_static(const eagle_static_tree_cfg *c, int *R, int *k) {
    if (!c) return EAGLE_ERR_INVALID_ARG;
    if (c->batch < 1 || c->vocab < 1 || c->nodes < 1 || !(c->tree_temp > 0.f)) return EAGLE_ERR_INVALID_ARG;
    if (c->nodes > 64) return EAGLE_ERR_UNSUPPORTED;
    if (c->batch > 65535) return EAGLE_ERR_UNSUPPORTED;
    if (c->parents[0] != -1) return EAGLE_ERR_INVALID_ARG;
    int kids[64] = {0};
    for (int i = 1; i < c->nodes; ++i) {
        if (c->parents[i] < 0 || c->parents[i] >= i) return EAGLE_ERR_INVALID_ARG;
        ++kids[c->parents[i]];
    }
    int r = 0, km = 0;
    for (int i = 0; i < c->nodes; ++i) {
        r += kids[i] > 0;
        km = kids[i] > km ? kids[i] : km;
    }
    if (km > 16 || km > c->vocab) return EAGLE_ERR_UNSUPPORTED;
    *R = r;
    *k = km;
    return 0;
}

int check_verify(const eagle_verify_cfg *c) {
    if (!c) return EAGLE_ERR_INVALID_ARG;
    if (c->batch < 1 || c->vocab < 1 || c->depth < 1 || c->topk < 1 || c->keep < 1) return EAGLE_ERR_INVALID_ARG;
    if (!(c->temperature >= 0.f)) return EAGLE_ERR_INVALID_ARG;
    if (c->keep + 1 > 64) return EAGLE_ERR_UNSUPPORTED;
    if (c->batch > 65535) return EAGLE_ERR_UNSUPPORTED;
    if (size_t(c->vocab) > verify_max_vocab()) return EAGLE_ERR_UNSUPPORTED;
    return 0;
}

}  // namespace
}  // namespace eagle

using namespace eagle;

// The bounded waits put to the test: warp 0 polls as a warp, lane 0 of warp 1 polls alone, both
// on an mbarrier that nothing ever completes.  Each gives up at the deadline, records
// EAGLE_ERR_TIMEOUT and stores how long it waited.
static __global__ void wait_selftest_kernel(int32_t *status, uint64_t *elapsed_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
    }
    __syncthreads();
    const uint64_t t0 = global_ns();
    bool got = true;
    if (threadIdx.x < 32)
        got = mbar_warp_wait_bounded(&bar, 0);
    else if (threadIdx.x == 32)
        got = mbar_wait_bounded(&bar, 0);
    if (!got) set_status(status, EAGLE_ERR_TIMEOUT);
    if ((threadIdx.x & 31) == 0) elapsed_ns[threadIdx.x >> 5] = global_ns() - t0;
}

extern "C" {

size_t eagle_build_tree_workspace_size(const eagle_tree_cfg *cfg) {
    if (check_tree(cfg)) return 0;
    return build_tree_workspace_bytes(*cfg);
}

eagle_status eagle_build_tree(const eagle_tree_cfg *cfg, const float *draft_logits, const int32_t *root_token,
                              int32_t *tokens, int32_t *parents, int32_t *depths, int32_t *node_row,
                              uint64_t *mask, float *node_logv, void *ws, size_t ws_bytes, cudaStream_t stream) {
    reset_launches();
    if (int e = check_tree(cfg)) return e;
    if (!draft_logits || !root_token || !tokens || !parents || !depths || !node_row || !mask || !ws)
        return EAGLE_ERR_INVALID_ARG;
    if (!aligned256(ws) || ws_bytes < build_tree_workspace_bytes(*cfg)) return EAGLE_ERR_INVALID_ARG;
    return build_tree_launch(*cfg, draft_logits, nullptr, root_token, tokens, parents, depths, node_row, mask,
                             node_logv, ws, stream);
}

eagle_status eagle_build_tree_sampled(const eagle_tree_cfg *cfg, const float *draft_logits, const float *child_u,
                                      const int32_t *root_token, int32_t *tokens, int32_t *parents, int32_t *depths,
                                      int32_t *node_row, uint64_t *mask, float *node_logv, void *ws, size_t ws_bytes,
                                      cudaStream_t stream) {
    reset_launches();
    if (int e = check_tree(cfg)) return e;
    if (size_t(cfg->vocab) > row_sample_max_vocab()) return EAGLE_ERR_UNSUPPORTED;
    if (!draft_logits || !child_u || !root_token || !tokens || !parents || !depths || !node_row || !mask || !ws)
        return EAGLE_ERR_INVALID_ARG;
    if (!aligned256(ws) || ws_bytes < build_tree_workspace_bytes(*cfg)) return EAGLE_ERR_INVALID_ARG;
    return build_tree_launch(*cfg, draft_logits, child_u, root_token, tokens, parents, depths, node_row, mask,
                             node_logv, ws, stream);
}

eagle_status eagle_build_begin(const eagle_tree_cfg *cfg, const float *root_logits, const float *child_u, void *ws,
                               size_t ws_bytes, int32_t *frontier_tok, int32_t *frontier_parent,
                               cudaStream_t stream) {
    reset_launches();
    if (int e = check_tree(cfg)) return e;
    if (child_u && size_t(cfg->vocab) > row_sample_max_vocab()) return EAGLE_ERR_UNSUPPORTED;
    if (!root_logits || !ws) return EAGLE_ERR_INVALID_ARG;
    if (cfg->depth >= 2 && (!frontier_tok || !frontier_parent)) return EAGLE_ERR_INVALID_ARG;
    if (!aligned256(ws) || ws_bytes < build_tree_workspace_bytes(*cfg)) return EAGLE_ERR_INVALID_ARG;
    return build_step_launch(*cfg, 0, root_logits, child_u, frontier_tok, frontier_parent, ws, stream);
}

eagle_status eagle_build_expand(const eagle_tree_cfg *cfg, int32_t depth, const float *frontier_logits,
                                const float *child_u, void *ws, size_t ws_bytes, int32_t *frontier_tok,
                                int32_t *frontier_parent, cudaStream_t stream) {
    reset_launches();
    if (int e = check_tree(cfg)) return e;
    if (child_u && size_t(cfg->vocab) > row_sample_max_vocab()) return EAGLE_ERR_UNSUPPORTED;
    if (depth < 1 || depth > cfg->depth - 1 || !frontier_logits || !ws) return EAGLE_ERR_INVALID_ARG;
    if (depth + 1 <= cfg->depth - 1 && (!frontier_tok || !frontier_parent)) return EAGLE_ERR_INVALID_ARG;
    if (!aligned256(ws) || ws_bytes < build_tree_workspace_bytes(*cfg)) return EAGLE_ERR_INVALID_ARG;
    return build_step_launch(*cfg, depth, frontier_logits, child_u, frontier_tok, frontier_parent, ws, stream);
}

eagle_status eagle_build_finalize(const eagle_tree_cfg *cfg, const int32_t *root_token, void *ws, size_t ws_bytes,
                                  int32_t *tokens, int32_t *parents, int32_t *depths, int32_t *node_row,
                                  uint64_t *mask, float *node_logv, cudaStream_t stream) {
    reset_launches();
    if (int e = check_tree(cfg)) return e;
    if (!root_token || !tokens || !parents || !depths || !node_row || !mask || !ws) return EAGLE_ERR_INVALID_ARG;
    if (!aligned256(ws) || ws_bytes < build_tree_workspace_bytes(*cfg)) return EAGLE_ERR_INVALID_ARG;
    return build_finalize_launch(*cfg, root_token, tokens, parents, depths, node_row, mask, node_logv, ws, stream);
}

size_t eagle_tree_attention_workspace_size(const eagle_attn_cfg *cfg) {
    if (check_attn(cfg)) return 0;
    return tree_attention_workspace_bytes(*cfg);
}

eagle_status eagle_tree_attention(const eagle_attn_cfg *cfg, const void *q, const void *k_cache,
                                  const void *v_cache, const int32_t *ctx_len, const void *k_tree,
                                  const void *v_tree, const uint64_t *mask, void *out, void *ws, size_t ws_bytes,
                                  cudaStream_t stream) {
    reset_launches();
    if (int e = check_attn(cfg)) return e;
    if (!q || !k_cache || !v_cache || !ctx_len || !k_tree || !v_tree || !mask || !out || !ws)
        return EAGLE_ERR_INVALID_ARG;
    if (!aligned256(ws) || ws_bytes < tree_attention_workspace_bytes(*cfg)) return EAGLE_ERR_INVALID_ARG;
    // 16-byte alignment of every K/V/Q/O row start (d elements of 2 or 4 bytes)
    const uintptr_t any = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k_cache) |
                          reinterpret_cast<uintptr_t>(v_cache) | reinterpret_cast<uintptr_t>(k_tree) |
                          reinterpret_cast<uintptr_t>(v_tree) | reinterpret_cast<uintptr_t>(out);
    if (any & 15u) return EAGLE_ERR_INVALID_ARG;
    return tree_attention_launch(*cfg, q, k_cache, v_cache, ctx_len, k_tree, v_tree, mask, out, ws, stream);
}

size_t eagle_tree_verify_workspace_size(const eagle_verify_cfg *cfg) {
    if (check_verify(cfg)) return 0;
    return tree_verify_workspace_bytes(*cfg);
}

eagle_status eagle_tree_verify(const eagle_verify_cfg *cfg, const float *target_logits, const float *draft_logits,
                               const int32_t *tokens, const int32_t *parents, const int32_t *node_row,
                               const float *uniforms, int32_t *out_tokens, int32_t *out_len, int32_t *out_path,
                               float *out_ratio, void *ws, size_t ws_bytes, cudaStream_t stream) {
    reset_launches();
    if (int e = check_verify(cfg)) return e;
    if (!target_logits || !draft_logits || !tokens || !parents || !node_row || !uniforms || !out_tokens ||
        !out_len || !out_path || !ws)
        return EAGLE_ERR_INVALID_ARG;
    if (!aligned256(ws) || ws_bytes < tree_verify_workspace_bytes(*cfg)) return EAGLE_ERR_INVALID_ARG;
    return tree_verify_launch(*cfg, target_logits, draft_logits, tokens, parents, node_row, uniforms, out_tokens,
                              out_len, out_path, out_ratio, ws, stream);
}

size_t eagle_build_static_tree_workspace_size(const eagle_static_tree_cfg *cfg) {
    int R = 0, k = 0;
    if (check_static(cfg, &R, &k)) return 0;
    return static_tree_workspace_bytes(*cfg, R, k);
}

eagle_status eagle_build_static_tree(const eagle_static_tree_cfg *cfg, const float *draft_logits,
                                     const int32_t *root_token, int32_t *tokens, int32_t *parents, int32_t *depths,
                                     int32_t *node_row, uint64_t *mask, float *node_logv, void *ws, size_t ws_bytes,
                                     cudaStream_t stream) {
    reset_launches();
    int R = 0, k = 0;
    if (int e = check_static(cfg, &R, &k)) return e;
    if ((R > 0 && !draft_logits) || !root_token || !tokens || !parents || !depths || !node_row || !mask || !ws)
        return EAGLE_ERR_INVALID_ARG;
    if (!aligned256(ws) || ws_bytes < static_tree_workspace_bytes(*cfg, R, k)) return EAGLE_ERR_INVALID_ARG;
    return build_static_tree_launch(*cfg, R, k, draft_logits, nullptr, root_token, tokens, parents, depths, node_row,
                                    mask, node_logv, ws, stream);
}

eagle_status eagle_build_static_tree_sampled(const eagle_static_tree_cfg *cfg, const float *draft_logits,
                                             const float *child_u, const int32_t *root_token, int32_t *tokens,
                                             int32_t *parents, int32_t *depths, int32_t *node_row, uint64_t *mask,
                                             float *node_logv, void *ws, size_t ws_bytes, cudaStream_t stream) {
    reset_launches();
    int R = 0, k = 0;
    if (int e = check_static(cfg, &R, &k)) return e;
    if (size_t(cfg->vocab) > row_sample_max_vocab()) return EAGLE_ERR_UNSUPPORTED;
    if ((R > 0 && (!draft_logits || !child_u)) || !root_token || !tokens || !parents || !depths || !node_row ||
        !mask || !ws)
        return EAGLE_ERR_INVALID_ARG;
    if (!aligned256(ws) || ws_bytes < static_tree_workspace_bytes(*cfg, R, k)) return EAGLE_ERR_INVALID_ARG;
    return build_static_tree_launch(*cfg, R, k, draft_logits, child_u, root_token, tokens, parents, depths, node_row,
                                    mask, node_logv, ws, stream);
}

size_t eagle_kv_commit_workspace_size(const eagle_attn_cfg *cfg) {
    if (check_attn(cfg)) return 0;
    return kWsHeader;
}

eagle_status eagle_kv_commit(const eagle_attn_cfg *cfg, int32_t depth, const void *k_tree, const void *v_tree,
                             const int32_t *out_path, const int32_t *out_len, const int32_t *ctx_len, void *k_cache,
                             void *v_cache, int32_t *new_ctx_len, void *ws, size_t ws_bytes, cudaStream_t stream) {
    reset_launches();
    if (int e = check_attn(cfg)) return e;
    if (depth < 0 || depth > 63) return EAGLE_ERR_INVALID_ARG;
    if (cfg->layers > 65535 || cfg->batch > 65535) return EAGLE_ERR_UNSUPPORTED;
    if (!k_tree || !v_tree || !out_path || !out_len || !ctx_len || !k_cache || !v_cache || !new_ctx_len || !ws)
        return EAGLE_ERR_INVALID_ARG;
    if (new_ctx_len == ctx_len) return EAGLE_ERR_INVALID_ARG;  // every CTA of a sequence reads ctx_len
    if (!aligned256(ws) || ws_bytes < kWsHeader) return EAGLE_ERR_INVALID_ARG;
    const uintptr_t any = reinterpret_cast<uintptr_t>(k_tree) | reinterpret_cast<uintptr_t>(v_tree) |
                          reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache);
    if (any & 15u) return EAGLE_ERR_INVALID_ARG;
    return kv_commit_launch(*cfg, depth, k_tree, v_tree, out_path, out_len, ctx_len, k_cache, v_cache, new_ctx_len,
                            ws, stream);
}

eagle_status eagle_workspace_init(void *ws, size_t bytes, cudaStream_t stream) {
    if (!ws || bytes < kWsHeader) return EAGLE_ERR_INVALID_ARG;
    return cudaMemsetAsync(ws, 0, bytes, stream) == cudaSuccess ? EAGLE_OK : EAGLE_ERR_CUDA;
}

eagle_status eagle_get_device_status(void *ws, cudaStream_t stream, int32_t *out) {
    if (!ws || !out) return EAGLE_ERR_INVALID_ARG;
    int32_t v = 0;
    if (cudaMemcpyAsync(&v, ws, sizeof v, cudaMemcpyDeviceToHost, stream) != cudaSuccess) return EAGLE_ERR_CUDA;
    if (cudaMemsetAsync(ws, 0, sizeof v, stream) != cudaSuccess) return EAGLE_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return EAGLE_ERR_CUDA;
    *out = v;
    return EAGLE_OK;
}

const char *eagle_status_string(eagle_status s) {
    switch (s) {
        case EAGLE_OK: return "ok";
        case EAGLE_ERR_INVALID_ARG: return "invalid argument";
        case EAGLE_ERR_UNSUPPORTED: return "unsupported size";
        case EAGLE_ERR_CUDA: return "CUDA launch error";
        case EAGLE_ERR_TIMEOUT: return "device wait timed out";
        case EAGLE_ERR_DEVICE_INPUT: return "bad device-side input";
        default: return "unknown status";
    }
}

int32_t eagle_last_launch_count(void) { return t_launches; }

eagle_status eagle_selftest_wait_timeout(void *ws, uint64_t *elapsed_ns, cudaStream_t stream) {
    if (!aligned256(ws) || !elapsed_ns) return EAGLE_ERR_INVALID_ARG;
    reset_launches();
    wait_selftest_kernel<<<1, 64, 0, stream>>>(static_cast<int32_t *>(ws), elapsed_ns);
    if (cudaPeekAtLastError() != cudaSuccess) return EAGLE_ERR_CUDA;
    note_launch();
    return EAGLE_OK;
}

eagle_status eagle_selftest_exp2_error(float *max_rel_err, cudaStream_t stream) {
    if (!max_rel_err) return EAGLE_ERR_INVALID_ARG;
    reset_launches();
    return exp2_error_launch(max_rel_err, stream);
}

}  // extern "C"
