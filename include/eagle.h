/*
 * eagle.h -- C ABI of the GB300 (sm_103a) EAGLE draft-tree verify round.
 *
 * One verify round of EAGLE-style speculative decoding, in three calls:
 *
 *   eagle_build_tree      draft logits -> EAGLE-2 dynamic draft tree (tokens, parents, depths,
 *                         expanding draft row per node, ancestor bit masks).
 *                         Defined by: "(EAGLE 2) EAGLE-2: Faster Inference of Language Models
 *                         with Dynamic Draft Trees" (tom-jerr.github.io), sections "Expanding the
 *                         Draft Tree" (value V_i = product of draft confidences along the path;
 *                         the k most valuable nodes of a depth are expanded), "Rerank draft
 *                         tokens" (global top-m by value, shallower first on ties; the kept set
 *                         stays a connected tree) and "Tree Attention Mask" (flatten to one
 *                         sequence; a token sees only its ancestors).
 *   eagle_build_static_tree  a static draft tree (EAGLE-1) or a chain from a caller's template:
 *                         the same outputs as eagle_build_tree (see the entry point below).
 *   *_sampled, eagle_build_begin/expand/finalize  the same builds with sampled children (the
 *                         non-greedy setting) and the dynamic build one depth at a time, so
 *                         that a draft model can run between the depths (see below).
 *   eagle_tree_attention  tree-masked grouped-query attention of the flattened tree against the
 *                         cached context, for every layer.  Defined by: "LLM speculative decoding
 *                         explained" (hubwiz.com), section 5 (the flattened tree is scored in one
 *                         pass; each candidate sees only its ancestors and the context), and the
 *                         EAGLE-2 notes' "Tree Attention Mask".
 *   eagle_tree_verify     recursive tree speculative sampling over target and draft logits ->
 *                         committed tokens.  Defined by: "EAGLE: Speculative Sampling Requires
 *                         Rethinking Feature Uncertainty" (papercache.org), section A3 (accept
 *                         with probability min(1, p/q); on rejection resample from
 *                         norm(max(0, p - q))), section 3.3 and appendix A.2 (multi-round: after
 *                         a rejection, test the next candidate against the adjusted distribution;
 *                         sample only after every candidate was rejected), and the hubwiz
 *                         article's sections 1-2 (p = target, q = draft; a bonus token when every
 *                         draft token on the path is accepted; temperature applied to both).
 *   eagle_kv_commit       appends the committed nodes' keys and values to each KV cache, which
 *                         sets up the next round (the same pages; see the entry point below).
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers; tensors are dense row-major with the shapes given
 *     per argument.  The caller owns all memory: inputs, outputs and the workspace.  The library
 *     never allocates device or host memory on these calls.
 *   - Calls are asynchronous on `stream` and make no host synchronisation, so a round can be
 *     captured in a CUDA graph (make one un-captured call of each entry point first: it sets the
 *     kernels' shared-memory attributes).
 *   - Workspace: `ws` must be at least eagle_*_workspace_size(cfg) bytes, 256-byte aligned, and
 *     zeroed once before its first use (eagle_workspace_init).  Its first 256 bytes hold a device
 *     status word that kernels set when they detect bad device-side input; it is sticky until read
 *     with eagle_get_device_status.  A workspace must not be used by two calls that may run
 *     concurrently.
 *   - Return value: EAGLE_OK, or an error detected on the host BEFORE any launch (nothing has
 *     been written then), or EAGLE_ERR_CUDA when a launch failed.
 *   - n = keep + 1 tree nodes per sequence; node 0 is the root (the last committed token).
 *     R = 1 + (depth-1)*topk draft rows per sequence: row 0 expands the root, row
 *     1 + (f-1)*topk + s expands the s-th most valuable node of depth f.
 *   - Supported sizes: 1 <= topk <= 16, n <= 64 (one 64-bit mask word per node),
 *     topk + (depth-1)*topk^2 <= 1024, head_dim in {64, 128}, heads_q % heads_kv == 0.
 *     Other sizes return EAGLE_ERR_UNSUPPORTED.
 */
#ifndef EAGLE_H
#define EAGLE_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t eagle_status;

#define EAGLE_OK 0
#define EAGLE_ERR_INVALID_ARG 1   /* null pointer, negative size, workspace too small ...     */
#define EAGLE_ERR_UNSUPPORTED 2   /* valid but outside the supported sizes listed above      */
#define EAGLE_ERR_CUDA 3          /* a kernel launch failed                                   */
#define EAGLE_ERR_TIMEOUT 4       /* device status only: a bounded device wait gave up        */
#define EAGLE_ERR_DEVICE_INPUT 5  /* device status only: bad token id, parent or context len  */

#define EAGLE_DTYPE_F32 0
#define EAGLE_DTYPE_BF16 1

/* Draft-tree build configuration. */
typedef struct {
    int32_t batch;   /* B: sequences                                              */
    int32_t vocab;   /* V                                                         */
    int32_t depth;   /* D: draft-token depths below the root                      */
    int32_t topk;    /* k: children per expanded node and nodes expanded per depth */
    int32_t keep;    /* m: kept draft tokens after the rerank (the root is extra)  */
    float tree_temp; /* temperature of the draft confidences (1.0 in EAGLE-2)    */
} eagle_tree_cfg;

/* Tree-attention configuration. */
typedef struct {
    int32_t batch;    /* B                                                   */
    int32_t layers;   /* L: layers processed by one call                     */
    int32_t nodes;    /* n = m + 1 tree nodes per sequence                   */
    int32_t heads_q;  /* Hq                                                  */
    int32_t heads_kv; /* Hkv (Hq / Hkv query heads share one KV head)        */
    int32_t head_dim; /* d: 64 or 128                                        */
    int32_t max_seq;  /* S_max: allocated context positions per sequence     */
    int32_t dtype;    /* EAGLE_DTYPE_BF16 or EAGLE_DTYPE_F32 (q, K, V, out)  */
    float scale;      /* softmax scale; 0 means 1/sqrt(d)                    */
} eagle_attn_cfg;

/* Verification configuration. */
typedef struct {
    int32_t batch;     /* B                                                     */
    int32_t vocab;     /* V                                                     */
    int32_t depth;     /* D (commits at most D + 1 tokens)                      */
    int32_t topk;      /* k (sets R = 1 + (D-1)k, the draft-logit rows)         */
    int32_t keep;      /* m (n = m + 1 nodes)                                   */
    float temperature; /* T > 0: speculative sampling at T;  T == 0: greedy     */
} eagle_verify_cfg;

/* A static draft tree (EAGLE-1) or chain: one template of parent indices for every sequence. */
typedef struct {
    int32_t batch;      /* B                                                         */
    int32_t vocab;      /* V                                                         */
    int32_t nodes;      /* n <= 64 template nodes; node 0 is the root                */
    float tree_temp;    /* temperature of the draft confidences (log V), > 0         */
    int8_t parents[64]; /* parents[0] = -1, parents[i] in [0, i) for 1 <= i < n      */
} eagle_static_tree_cfg;

/* ---------------------------------------------------------------------------------------- */

/* Workspace bytes needed by eagle_build_tree for this configuration (0 if the config is
 * invalid or unsupported). */
size_t eagle_build_tree_workspace_size(const eagle_tree_cfg *cfg);

/*
 * Build the EAGLE-2 dynamic draft tree of every sequence.
 *   draft_logits  f32 [B][R][V]  draft logits; row roles as in the conventions above.
 *   root_token    i32 [B]        token of node 0.
 * Outputs (n = keep + 1):
 *   tokens        i32 [B][n]     node tokens (node 0 = root_token).
 *   parents       i32 [B][n]     parent node index, -1 for the root; parents precede children.
 *   depths        i32 [B][n]     0 for the root, 1..D otherwise.
 *   node_row      i32 [B][n]     draft row that expanded the node (0 for the root), -1 if the
 *                                node was never expanded.
 *   mask          u64 [B][n]     bit j set iff node j is node i itself or one of its ancestors.
 *   node_logv     f32 [B][n]     optional (may be NULL): log V_i, the log of the product of
 *                                draft confidences along the path (0 for the root).
 * Node order: the root, then the kept nodes by creation order (depth, then the parent's rank
 * among the expanded nodes of its depth, then the child's rank in its row).  Ties in value are
 * broken shallower first, then by creation order; ties in logit by the lower token id.
 * Device-side check: a root token outside [0, V) sets EAGLE_ERR_DEVICE_INPUT.
 */
eagle_status eagle_build_tree(const eagle_tree_cfg *cfg, const float *draft_logits, const int32_t *root_token,
                              int32_t *tokens, int32_t *parents, int32_t *depths, int32_t *node_row,
                              uint64_t *mask, float *node_logv, void *ws, size_t ws_bytes, cudaStream_t stream);

/*
 * eagle_build_tree with sampled children: the non-greedy drafting of "EAGLE: Speculative Sampling
 * Requires Rethinking Feature Uncertainty" (papercache.org), appendix A.1 (a node's k children
 * are sampled from the draft distribution rather than taken as its top k).
 *   child_u  f32 [B][R][k]  uniforms in [0, 1) (others are clamped into it; NaN counts as 0).
 * Row r's children are k independent draws from q_r = softmax(x_r / tree_temp), with
 * replacement (a token may be drawn twice), draw j by inverse CDF over ascending token id with
 * child_u[b][r][j]; the children keep draw order, so creation order, frontier slots, the rerank
 * and every output are then as in eagle_build_tree.  Draft confidences (node_logv) are q at the
 * drawn tokens.  The draw is decided on exact fixed-point sums of the row's weights against its
 * maximum (units of 2^-S of the maximum's weight, S = 62 - ceil(log2 vocab)), each weight's
 * exponent formed without rounding error; the fp64 definition can differ only where a uniform
 * lies within about 1e-7 of a CDF step (eagle_selftest_exp2_error bounds the one approximate
 * factor).
 * Losslessness: with tree_temp equal to the verify temperature, verification of a tree whose
 * every expanded node keeps all k children (keep = topk + (depth-1) topk^2, or a static tree)
 * commits exactly the target distribution.  A rerank that keeps fewer nodes drops children by
 * their drawn values, which biases the kept candidates.
 * Workspace: eagle_build_tree_workspace_size.  Extra checks: vocab <= 2^21 (else
 * EAGLE_ERR_UNSUPPORTED).  Device-side: a row with no finite logit sets EAGLE_ERR_DEVICE_INPUT
 * and its children are token 0.
 */
eagle_status eagle_build_tree_sampled(const eagle_tree_cfg *cfg, const float *draft_logits, const float *child_u,
                                      const int32_t *root_token, int32_t *tokens, int32_t *parents, int32_t *depths,
                                      int32_t *node_row, uint64_t *mask, float *node_logv, void *ws, size_t ws_bytes,
                                      cudaStream_t stream);

/*
 * Stepwise build: the same tree as eagle_build_tree (or _sampled), one depth at a time, so that a
 * draft model can produce each depth's rows from the frontier chosen by the previous step (the
 * EAGLE-2 notes, "Expanding the Draft Tree": only the k most valuable nodes of a depth are fed to
 * the draft model for the next depth).  The calls, in this order, on one workspace (size
 * eagle_build_tree_workspace_size; it carries the state between them):
 *   eagle_build_begin(root_logits f32 [B][V])              row 0;
 *   eagle_build_expand(depth = f, frontier_logits [B][k][V])  rows 1 + (f-1)k + s, s < k: the
 *                                                          draft logits at frontier slot s of
 *                                                          depth f, for f = 1 .. D-1;
 *   eagle_build_finalize                                   the rerank, flatten and outputs.
 * child_u: NULL for top-k children, else the step's uniforms, f32 [B][1][k] for begin and
 * [B][k][k] for expand (the rows' slices of eagle_build_tree_sampled's child_u).
 * begin and expand(f) with f + 1 <= D - 1 write the frontier of the next depth (1 for begin,
 * f + 1 for expand), the nodes the draft model expands next:
 *   frontier_tok     i32 [B][k]  token of slot s;
 *   frontier_parent  i32 [B][k]  slot, within the previous depth's frontier, of its parent
 *                                (-1 at depth 1: the parent is the root).
 * Otherwise the frontier pointers are not used (they may be NULL).  Fed the rows that
 * eagle_build_tree would read, the steps produce bit-identical outputs.  Calls out of order read
 * stale state: the result is unspecified, and frontier slots outside their depth set
 * EAGLE_ERR_DEVICE_INPUT.
 */
eagle_status eagle_build_begin(const eagle_tree_cfg *cfg, const float *root_logits, const float *child_u, void *ws,
                               size_t ws_bytes, int32_t *frontier_tok, int32_t *frontier_parent,
                               cudaStream_t stream);
eagle_status eagle_build_expand(const eagle_tree_cfg *cfg, int32_t depth, const float *frontier_logits,
                                const float *child_u, void *ws, size_t ws_bytes, int32_t *frontier_tok,
                                int32_t *frontier_parent, cudaStream_t stream);
/* Outputs as eagle_build_tree. */
eagle_status eagle_build_finalize(const eagle_tree_cfg *cfg, const int32_t *root_token, void *ws, size_t ws_bytes,
                                  int32_t *tokens, int32_t *parents, int32_t *depths, int32_t *node_row,
                                  uint64_t *mask, float *node_logv, cudaStream_t stream);

/* Workspace bytes needed by eagle_build_static_tree (0 for an invalid or unsupported cfg). */
size_t eagle_build_static_tree_workspace_size(const eagle_static_tree_cfg *cfg);

/*
 * A static draft tree or a chain, as EAGLE-1 drafts them.  Defined by: "EAGLE: Speculative
 * Sampling Requires Rethinking Feature Uncertainty" (papercache.org), appendix A.1 (a fixed tree;
 * in the greedy setting a node's children are the top tokens of the draft distribution at it)
 * and section 4.3.1 (the chain: one child per node).  The pages draw the tree only as a figure,
 * so its shape is the caller's template (cfg->parents).
 *   draft_logits f32 [B][R][V]  R = the number of template nodes with children; row r of a
 *                               sequence belongs to the r-th such node in ascending index.
 *   root_token   i32 [B]
 * Outputs as eagle_build_tree (n = cfg->nodes): a node's children, in ascending index, take its
 * row's tokens of rank 0, 1, ... (value desc, ties to the lower token id); node_row[i] is node
 * i's own row or -1; node_logv[i] is the sum of log-confidences x/T - logsumexp(x/T) along the
 * path; masks are ancestor-or-self bits.  A chain of depth D is the template
 * parents = {-1, 0, 1, ..., D - 1}.
 * Host-side checks: the template (parents[0] = -1, parents[i] in [0, i)), n <= 64, at most 16
 * children per node and at most V.  Device-side: a root token outside [0, V) sets
 * EAGLE_ERR_DEVICE_INPUT.
 */
eagle_status eagle_build_static_tree(const eagle_static_tree_cfg *cfg, const float *draft_logits,
                                     const int32_t *root_token, int32_t *tokens, int32_t *parents, int32_t *depths,
                                     int32_t *node_row, uint64_t *mask, float *node_logv, void *ws, size_t ws_bytes,
                                     cudaStream_t stream);

/*
 * eagle_build_static_tree with sampled children (appendix A.1 of the EAGLE-1 page: the
 * non-greedy setting samples a node's children).  child_u f32 [B][R][kmax], kmax = the most
 * children of one template node: node p's children, in ascending index, are draws 0, 1, ... of
 * its row, as eagle_build_tree_sampled draws them.  A static template keeps every drawn child,
 * so build -> verify at tree_temp = the verify temperature is exactly lossless.
 * Workspace: eagle_build_static_tree_workspace_size.  Extra checks: vocab <= 2^21.
 */
eagle_status eagle_build_static_tree_sampled(const eagle_static_tree_cfg *cfg, const float *draft_logits,
                                             const float *child_u, const int32_t *root_token, int32_t *tokens,
                                             int32_t *parents, int32_t *depths, int32_t *node_row, uint64_t *mask,
                                             float *node_logv, void *ws, size_t ws_bytes, cudaStream_t stream);

/* Workspace bytes needed by eagle_tree_attention. */
size_t eagle_tree_attention_workspace_size(const eagle_attn_cfg *cfg);

/*
 * Tree-masked GQA attention for every layer, sequence and query head.
 *   q        [L][B][n][Hq][d]       queries of the tree nodes (position embedding applied by
 *                                   the caller: node i sits at position ctx_len[b] + depth_i).
 *   k_cache  [L][B][S_max][Hkv][d]  cached context keys; positions >= ctx_len[b] are not read.
 *   v_cache  [L][B][S_max][Hkv][d]  cached context values.
 *   ctx_len  i32 [B]                context length per sequence, 0 <= ctx_len[b] <= S_max.
 *   k_tree   [L][B][n][Hkv][d]      keys of the tree nodes.
 *   v_tree   [L][B][n][Hkv][d]      values of the tree nodes.
 *   mask     u64 [B][n]             ancestor-or-self bit masks (as eagle_build_tree writes).
 *   out      [L][B][n][Hq][d]       softmax(scale * q.k over the context and the masked tree)
 *                                   times v; query head h reads KV head h / (Hq/Hkv).
 * Element type of q, K, V and out is cfg->dtype (bf16 with fp32 accumulation and softmax, or
 * fp32 throughout).  Device-side check: a context length outside [0, S_max] sets
 * EAGLE_ERR_DEVICE_INPUT and that sequence's rows are left unwritten.
 */
eagle_status eagle_tree_attention(const eagle_attn_cfg *cfg, const void *q, const void *k_cache,
                                  const void *v_cache, const int32_t *ctx_len, const void *k_tree,
                                  const void *v_tree, const uint64_t *mask, void *out, void *ws, size_t ws_bytes,
                                  cudaStream_t stream);

/* Workspace bytes needed by eagle_kv_commit (the status header only; 0 for an invalid cfg). */
size_t eagle_kv_commit_workspace_size(const eagle_attn_cfg *cfg);

/*
 * Append each sequence's committed tree nodes to its KV cache, for every layer.  Defined by:
 * "LLM speculative decoding explained" (hubwiz.com) sections 1 and 5 (a round commits the accepted
 * draft tokens and one more; the tree pass computed every node's keys and values at position
 * ctx + depth) and the EAGLE notes' section 3.3 (the accepted path).
 *   cfg          the attention configuration of the round (B, L, n, Hkv, d, S_max, dtype).
 *   depth        D: the width of out_path.
 *   k_tree, v_tree  [L][B][n][Hkv][d]  the round's tree keys and values (as given to
 *                   eagle_tree_attention).
 *   out_path     i32 [B][D], out_len i32 [B]: as eagle_tree_verify writes them.
 *   ctx_len      i32 [B]  context lengths of the round.
 *   k_cache, v_cache  [L][B][S_max][Hkv][d]: sequence b gains the root (node 0) at position
 *                   ctx_len[b], then path entries 0 .. out_len[b] - 2 at ctx_len[b] + 1 ...:
 *                   out_len[b] rows.  The last committed token has no keys or values yet (it is
 *                   the next round's root).  Other positions are not touched.
 *   new_ctx_len  i32 [B]  ctx_len[b] + out_len[b] (must not alias ctx_len).
 * Element type: cfg->dtype.  Device-side check: a sequence whose out_len exceeds D + 1, whose path
 * holds an id outside [1, n), or whose new length exceeds S_max sets EAGLE_ERR_DEVICE_INPUT and
 * keeps its cache and length; out_len 0 (a refused tree) is a no-op.  The K/V pointers must be
 * 16-byte aligned.
 */
eagle_status eagle_kv_commit(const eagle_attn_cfg *cfg, int32_t depth, const void *k_tree, const void *v_tree,
                             const int32_t *out_path, const int32_t *out_len, const int32_t *ctx_len, void *k_cache,
                             void *v_cache, int32_t *new_ctx_len, void *ws, size_t ws_bytes, cudaStream_t stream);

/* Workspace bytes needed by eagle_tree_verify. */
size_t eagle_tree_verify_workspace_size(const eagle_verify_cfg *cfg);

/*
 * Recursive tree speculative sampling (T > 0) or greedy verification (T == 0).
 *   target_logits f32 [B][n][V]  target logits after each node (row i = next-token logits of
 *                                the path ending at node i).
 *   draft_logits  f32 [B][R][V]  the draft logits the tree was built from.
 *   tokens, parents, node_row    i32 [B][n] as eagle_build_tree writes them.
 *   uniforms      f32 [B][n]     caller-drawn U(0,1): uniforms[b][i] (i >= 1) is node i's
 *                                accept test, uniforms[b][0] draws the final token.
 * At node a (starting at the root) with p = softmax(target[a]/T), q = softmax(draft[row(a)]/T):
 * each kept child c, in ascending node index, is accepted iff u[c] < p(tok_c)/q(tok_c); a
 * rejection replaces p by max(0, p - q) renormalised (kept if that has no mass).  An accepted
 * child becomes the new a.  When every child is rejected, or a has none, the final token is the
 * smallest t with sum_{s<=t} p(s) > u[0] and the walk stops.  At T == 0 the walk follows the
 * child holding argmax target[a] (ties to the lower id) and otherwise commits that argmax.
 * Outputs:
 *   out_tokens i32 [B][D+1]  committed tokens, -1 padded.
 *   out_len    i32 [B]       committed count (accepted nodes + 1).
 *   out_path   i32 [B][D]    accepted node indices in order, -1 padded.
 *   out_ratio  f32 [B][n]    optional (may be NULL): for every non-root node, the ratio p/q it
 *                            is (or would be) tested with once all its earlier siblings were
 *                            rejected; NaN for the root and at T == 0.
 * Device-side check: a malformed tree (parent not before child, token outside [0, V), missing
 * draft row under a node with children) sets EAGLE_ERR_DEVICE_INPUT and that sequence's
 * out_len to 0.  A device wait that runs out (EAGLE_ERR_TIMEOUT) sets out_len to 0 for every
 * sequence of the call.
 */
eagle_status eagle_tree_verify(const eagle_verify_cfg *cfg, const float *target_logits, const float *draft_logits,
                               const int32_t *tokens, const int32_t *parents, const int32_t *node_row,
                               const float *uniforms, int32_t *out_tokens, int32_t *out_len, int32_t *out_path,
                               float *out_ratio, void *ws, size_t ws_bytes, cudaStream_t stream);

/*
 * eagle_tree_verify without a caller workspace: the same computation and outputs (the same
 * kernels run), with the scratch in the library's own static device storage of 256 KB: about
 * 36 bytes per tree node and 4 per sequence (eagle_tree_verify_workspace_size), e.g. 113
 * sequences of 64 nodes; a configuration needing more returns EAGLE_ERR_UNSUPPORTED before
 * anything runs.  It exists for callers that cannot hand the library a device workspace:
 * a serving process that reserves all device memory for weights and the KV cache at start-up and
 * grants no further buffers, or a host framework whose plugin interface passes tensors but no
 * scratch.  The pages describe no such entry point; it is an interface convenience only.
 *   - Allocates nothing.  The first call on each device looks up the scratch's address
 *     (cudaGetSymbolAddress) and caches it; make that first call before any stream capture.
 *     `stream` must belong to the current device (EAGLE_ERR_INVALID_ARG otherwise): the scratch
 *     used is the current device's.
 *   - The scratch starts zeroed (static storage) and needs no initialisation; no state carries
 *     from one call to the next except the device status word, which this entry point never
 *     reads: device-side errors show only through out_len, which is 0 for a malformed tree and
 *     for every sequence of a call in which a device wait ran out (each call tags its own
 *     failures, so an earlier call's scratch contents never reach the outputs).  Callers that
 *     need the status word use eagle_tree_verify with their own workspace.
 *   - There is one scratch per device: two calls that may overlap on the device (different
 *     streams, or different host threads) race on it and must be serialised by the caller.
 */
eagle_status eagle_tree_verify_static(const eagle_verify_cfg *cfg, const float *target_logits,
                                      const float *draft_logits, const int32_t *tokens, const int32_t *parents,
                                      const int32_t *node_row, const float *uniforms, int32_t *out_tokens,
                                      int32_t *out_len, int32_t *out_path, float *out_ratio, cudaStream_t stream);

/* Zero `bytes` of a workspace on `stream` (needed once before a workspace's first use). */
eagle_status eagle_workspace_init(void *ws, size_t bytes, cudaStream_t stream);

/* Read (and clear) the device status word of a workspace: synchronises `stream`, then stores
 * EAGLE_OK or the largest error code any kernel recorded since the last read into *out. */
eagle_status eagle_get_device_status(void *ws, cudaStream_t stream, int32_t *out);

/* Static description of a status code. */
const char *eagle_status_string(eagle_status status);

/* Number of kernel launches the most recent call of each entry point issued on this thread
 * (for launch accounting in benchmarks). */
int32_t eagle_last_launch_count(void);

/* Self-test of the device-side wait bound: one launch in which a warp and a single thread each
 * wait on a barrier that nothing completes.  Both give up after the library's wait limit (one
 * second), set EAGLE_ERR_TIMEOUT in the status word of `ws` (256-byte aligned, read it with
 * eagle_get_device_status) and store the nanoseconds they waited into elapsed_ns[0] (the warp)
 * and elapsed_ns[1] (the thread), a DEVICE buffer of two uint64.  The context stays usable. */
eagle_status eagle_selftest_wait_timeout(void *ws, uint64_t *elapsed_ns, cudaStream_t stream);

/* Self-test of the exponential behind the sampled children (eagle_build_tree_sampled and the
 * sampled static tree): the largest relative error of the SFU's 2^f over every float f with
 * |f| <= 1/2, against the double-precision exp2, stored into max_rel_err[0] (a DEVICE float).
 * The draws' CDF steps are off by at most half the weights' relative error plus V 2^-S (S =
 * 62 - ceil(log2 V)); a test bounds the former with this.  One launch, tens of milliseconds. */
eagle_status eagle_selftest_exp2_error(float *max_rel_err, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* EAGLE_H */
