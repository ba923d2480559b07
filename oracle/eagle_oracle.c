/*
 * eagle_oracle.c -- plain fp64 CPU restatement of the EAGLE draft-tree verify round.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the checker, not the product: only the test suite,
 * the smoke check and the benchmark's CPU-baseline leg load it.  It shares no code, header or
 * constant with the CUDA library and never calls it.  It favours being checkable by eye over
 * being fast: every step is the plain definition, in double precision, one element at a time.
 *
 * Sources (web pages on EAGLE; the method is defined there in prose):
 *   [EAGLE-2 notes]  "(EAGLE 2) EAGLE-2: Faster Inference of Language Models with Dynamic Draft
 *                    Trees", sections "Expanding the Draft Tree" (path value V_i = product of
 *                    confidences; top-k frontier), "Rerank draft tokens" (global top-m, shallower
 *                    first on equal value, result stays a connected tree), "Tree Attention Mask"
 *                    (flatten; each token sees only its ancestors).
 *   [EAGLE-1 notes]  "EAGLE: Speculative Sampling Requires Rethinking Feature Uncertainty",
 *                    section A3 "speculative sampling" (accept with min(1, p/q), resample from
 *                    norm(max(0, p - q))), section 3.3 (tree verification, recursive), appendix
 *                    A.1 (top-k children when greedy), appendix A.2 (multi-round speculative
 *                    sampling: after a rejection call the accept step again on the adjusted
 *                    distribution; sample from it only when every candidate was rejected).
 *   [EAGLE-3 blog]   "LLM speculative decoding explained" (hubwiz), section 1 (p = target,
 *                    q = draft; bonus token when all are accepted; 1 <= committed <= accepted+1),
 *                    section 2 (temperature is applied to both distributions before the test),
 *                    section 5 (flattened tree scored in one pass; ancestors-only mask).
 *
 * Readings where the pages are silent (the same list is kept in the design notes):
 *   - V_i is compared in log space: log V_i = sum of log-confidences (equal to the product).
 *   - Confidence = the draft row's softmax at the tree temperature (1 by default).
 *   - Children of a row = its k largest logits, ties to the lower token id (greedy).  When
 *     sampling ([EAGLE-1 notes] appendix A.1, non-greedy): k independent inverse-CDF draws from
 *     the row's q = softmax(x/T), with replacement, one caller uniform per draw, in draw order.
 *   - Frontier at depth f (1..D-1) = the k depth-f nodes of largest (log V desc, creation asc);
 *     frontier slot s is expanded with draft row 1 + (f-1)k + s.  Row 0 expands the root.
 *   - Creation index: depth-1 children 0..k-1 in child-rank order, then per depth, per frontier
 *     slot, per child rank.  Rerank key: (log V desc, depth asc, creation asc).
 *   - Flattened order: root = node 0, then kept nodes by creation index (parents first).
 *   - The root is an ancestor of every node; every node sees itself.
 *   - Verify at T > 0: children of a node are tested in ascending flattened index; accept iff
 *     u[c] < p(t)/q(t) (q(t) = 0 counts as +inf); on rejection p <- max(0, p-q)/sum, q kept;
 *     if the sum is 0 p is kept.  The final token is drawn by inverse CDF with u[0].
 *   - Verify at T = 0: follow the child whose token is the target argmax (ties to lower id);
 *     otherwise commit the argmax and stop.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_OK 0
#define ORC_BAD_ARG 1
#define ORC_NOT_CLOSED 2
#define ORC_BAD_TREE 3

#define DT_F32 0
#define DT_BF16 1

/* ------------------------------------------------------------------------------------------ */
/* small helpers                                                                              */
/* ------------------------------------------------------------------------------------------ */

/* log-sum-exp of x/T over a row, plain two-pass form. */
static double row_logsumexp(const float *x, int V, double T)
{
    double mx = -INFINITY;
    for (int t = 0; t < V; ++t) {
        double v = (double)x[t] / T;
        if (v > mx) mx = v;
    }
    double s = 0.0;
    for (int t = 0; t < V; ++t) s += exp((double)x[t] / T - mx);
    return mx + log(s);
}

/* The k largest entries of x, largest first; equal values go to the lower token id.
 * Plain repeated selection under the total order (value desc, id asc): pass j takes the best
 * entry that comes strictly after the entry taken by pass j-1. */
static void row_topk(const float *x, int V, int k, int *out)
{
    for (int j = 0; j < k; ++j) {
        int best = -1;
        for (int t = 0; t < V; ++t) {
            if (j > 0) {
                int prev = out[j - 1];
                int after = x[t] < x[prev] || (x[t] == x[prev] && t > prev);
                if (!after) continue;
            }
            if (best < 0 || x[t] > x[best]) best = t; /* strict '>' keeps the lower id on ties */
        }
        out[j] = best;
    }
}

/* argmax with ties to the lower token id */
static int row_argmax(const float *x, int V)
{
    int best = 0;
    for (int t = 1; t < V; ++t)
        if (x[t] > x[best]) best = t;
    return best;
}

static int inverse_cdf(const double *p, int V, double u, double *gap);

/* The children of one draft row in the non-greedy setting ([EAGLE-1 notes] appendix A.1: k
 * tokens are sampled instead of the top k).  Reading: k independent draws from the row's draft
 * distribution q = softmax(x/T), with replacement (a token may be drawn twice), draw j by
 * inverse CDF over ascending token id with the caller's uniform u[j]; the children keep draw
 * order.  q_buf: V doubles of scratch.  *gap is lowered to the smallest distance of a u[j] to the
 * CDF step that decided its draw. */
static void row_sample(const float *x, int V, double T, int k, const float *u, int *out, double *q_buf,
                       double *gap)
{
    const double lse = row_logsumexp(x, V, T);
    for (int t = 0; t < V; ++t) q_buf[t] = exp((double)x[t] / T - lse);
    for (int j = 0; j < k; ++j) {
        double g = INFINITY;
        out[j] = inverse_cdf(q_buf, V, (double)u[j], &g);
        if (g < *gap) *gap = g;
    }
}

/* A row's k children: the top k (u == NULL) or k draws (u = the row's k uniforms). */
static void row_children(const float *x, int V, double T, int k, const float *u, int *out, double *q_buf,
                         double *gap)
{
    if (u)
        row_sample(x, V, T, k, u, out, q_buf, gap);
    else
        row_topk(x, V, k, out);
}

static double bf16_to_double(uint16_t h)
{
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double load_elem(const void *base, size_t idx, int dtype)
{
    if (dtype == DT_F32) return (double)((const float *)base)[idx];
    return bf16_to_double(((const uint16_t *)base)[idx]);
}

/* ------------------------------------------------------------------------------------------ */
/* 1. Draft-tree build  ([EAGLE-2 notes] Expanding / Rerank / Tree Attention Mask)             */
/* ------------------------------------------------------------------------------------------ */

typedef struct {
    double logv;  /* log V_i = sum of log-confidences along root -> node */
    int depth;    /* 1..D */
    int creation; /* creation index, see the header */
    int parent;   /* creation index of the parent, -1 for a depth-1 node (parent = root) */
    int token;
    int row;      /* draft row that expanded this node, -1 if it was never expanded */
} cand_t;

/* Total order used for the frontier and the rerank: log V descending, then depth ascending,
 * then creation index ascending ([EAGLE-2 notes] Rerank: equal value -> shallower first). */
static int cand_before(const cand_t *a, const cand_t *b)
{
    if (a->logv != b->logv) return a->logv > b->logv;
    if (a->depth != b->depth) return a->depth < b->depth;
    return a->creation < b->creation;
}

static int cand_cmp(const void *pa, const void *pb)
{
    const cand_t *a = *(const cand_t *const *)pa;
    const cand_t *b = *(const cand_t *const *)pb;
    if (cand_before(a, b)) return -1;
    if (cand_before(b, a)) return 1;
    return 0;
}

/* Relative gap between two neighbouring keys of a selection.  Two keys that are equal because
 * they come from equal logits of one draft row (siblings) are decided identically by any exact
 * implementation, so they do not count as a near tie. */
static double key_gap(const cand_t *a, const cand_t *b)
{
    if (a->logv == b->logv && a->parent == b->parent) return INFINITY;
    double den = fmax(fabs(a->logv), fabs(b->logv));
    if (den < 1e-300) den = 1e-300;
    return fabs(a->logv - b->logv) / den;
}

/*
 * Build one sequence's tree.
 *   x: draft logits of this sequence, [R][V] with R = 1 + (D-1)k.
 *   outputs of length n = m + 1 (mask: n * W words, W = ceil(n/64)).
 *   margin: smallest relative key gap at any selection boundary that decides the result.
 */
static int build_one(int V, int D, int k, int m, double Tt, const float *x, const float *u, int32_t root_tok,
                     int32_t *tokens, int32_t *parents, int32_t *depths, int32_t *node_row,
                     uint64_t *mask, double *node_logv, double *margin, double *draw_gap,
                     int32_t *front_tok, int32_t *front_par)
{
    const int R = 1 + (D - 1) * k;
    const int P = k + (D - 1) * k * k;
    const int n = m + 1;
    const int W = (n + 63) / 64;
    double gap_min = INFINITY;

    cand_t *pool = (cand_t *)calloc((size_t)P, sizeof(cand_t));
    cand_t **order = (cand_t **)calloc((size_t)P, sizeof(cand_t *));
    int *kids = (int *)calloc((size_t)k, sizeof(int));
    int *flat = (int *)calloc((size_t)P, sizeof(int));
    double *qbuf = u ? (double *)calloc((size_t)V, sizeof(double)) : NULL;
    double dgap = INFINITY;
    if (!pool || !order || !kids || !flat || (u && !qbuf)) {
        free(pool); free(order); free(kids); free(flat); free(qbuf);
        return ORC_BAD_ARG;
    }

    /* depth 1: the root's children from row 0 */
    int np = 0;
    {
        const float *row = x;
        double lse = row_logsumexp(row, V, Tt);
        row_children(row, V, Tt, k, u, kids, qbuf, &dgap);
        for (int r = 0; r < k; ++r) {
            cand_t *c = &pool[np];
            c->logv = (double)row[kids[r]] / Tt - lse; /* log confidence; log V_parent(root) = 0 */
            c->depth = 1;
            c->creation = np;
            c->parent = -1;
            c->token = kids[r];
            c->row = -1;
            ++np;
        }
    }
    /* depths 2..D: expand the top-k frontier of the previous depth */
    int level_begin = 0, level_count = k;
    for (int f = 1; f <= D - 1; ++f) {
        for (int i = 0; i < level_count; ++i) order[i] = &pool[level_begin + i];
        qsort(order, (size_t)level_count, sizeof(cand_t *), cand_cmp);
        int nf = level_count < k ? level_count : k;
        for (int s = 0; s + 1 < level_count && s < k; ++s) {
            double g = key_gap(order[s], order[s + 1]);
            if (g < gap_min) gap_min = g;
        }
        int next_begin = np;
        /* the frontier of depth f in slot order, with each node's parent slot at depth f - 1 */
        for (int s = 0; front_tok && s < nf; ++s) {
            front_tok[(size_t)(f - 1) * k + s] = order[s]->token;
            front_par[(size_t)(f - 1) * k + s] =
                order[s]->parent < 0 ? -1 : pool[order[s]->parent].row - 1 - (f - 2) * k;
        }
        for (int s = 0; s < nf; ++s) {
            cand_t *par = order[s];
            par->row = 1 + (f - 1) * k + s;
            const float *row = x + (size_t)par->row * V;
            double lse = row_logsumexp(row, V, Tt);
            row_children(row, V, Tt, k, u ? u + (size_t)par->row * k : NULL, kids, qbuf, &dgap);
            for (int r = 0; r < k; ++r) {
                cand_t *c = &pool[np];
                c->logv = par->logv + ((double)row[kids[r]] / Tt - lse);
                c->depth = f + 1;
                c->creation = np;
                c->parent = par->creation;
                c->token = kids[r];
                c->row = -1;
                ++np;
            }
        }
        level_begin = next_begin;
        level_count = np - next_begin;
    }
    (void)R;

    /* rerank: keep the first m of the whole pool under the total order */
    for (int i = 0; i < np; ++i) order[i] = &pool[i];
    qsort(order, (size_t)np, sizeof(cand_t *), cand_cmp);
    if (m < np) {
        double g = key_gap(order[m - 1], order[m]);
        if (g < gap_min) gap_min = g;
    }
    char *kept = (char *)calloc((size_t)np, 1);
    for (int i = 0; i < m && i < np; ++i) kept[order[i]->creation] = 1;

    /* flatten: root first, then kept nodes in creation order (a parent is created before its
     * children, so every parent precedes its children) */
    tokens[0] = root_tok;
    parents[0] = -1;
    depths[0] = 0;
    node_row[0] = 0;
    node_logv[0] = 0.0;
    for (int w = 0; w < W; ++w) mask[w] = 0;
    mask[0] = 1ull;
    int next = 1;
    int status = ORC_OK;
    for (int c = 0; c < np; ++c) {
        if (!kept[c]) { flat[c] = -1; continue; }
        const cand_t *nd = &pool[c];
        int i = next++;
        flat[c] = i;
        int par = 0;
        if (nd->parent >= 0) {
            par = flat[nd->parent];
            if (par < 0) { status = ORC_NOT_CLOSED; par = 0; }
        }
        tokens[i] = nd->token;
        parents[i] = par;
        depths[i] = nd->depth;
        node_row[i] = nd->row;
        node_logv[i] = nd->logv;
        for (int w = 0; w < W; ++w) mask[(size_t)i * W + w] = mask[(size_t)par * W + w];
        mask[(size_t)i * W + i / 64] |= 1ull << (i % 64);
    }
    *margin = gap_min;
    if (draw_gap) *draw_gap = dgap;
    free(qbuf);
    free(kept);
    free(pool);
    free(order);
    free(kids);
    free(flat);
    return status;
}

/* Batched build.  draft_logits [B][R][V]; outputs [B][n] (mask [B][n][W]).
 * child_u: NULL for top-k children, else [B][R][k] uniforms in [0, 1) (sampled children).
 * draw_gap [B] (optional): smallest distance of a uniform to the CDF step deciding its draw.
 * front_tok, front_par [B][D-1][k] (optional, both or neither): the frontier of each depth
 * f = 1..D-1 in slot order (slot s is expanded with row 1 + (f-1)k + s) and each frontier
 * node's parent slot at depth f - 1 (-1 at depth 1: the parent is the root). */
int orc_build_tree_ex(int B, int V, int D, int k, int m, double tree_temp, const float *draft_logits,
                      const float *child_u, const int32_t *root_token, int32_t *tokens, int32_t *parents,
                      int32_t *depths, int32_t *node_row, uint64_t *mask, double *node_logv, double *margin,
                      double *draw_gap, int32_t *front_tok, int32_t *front_par, int nthreads)
{
    if (B < 0 || V < 1 || D < 1 || k < 1 || k > V || m < 1 || !(tree_temp > 0)) return ORC_BAD_ARG;
    if ((front_tok == NULL) != (front_par == NULL)) return ORC_BAD_ARG;
    const int P = k + (D - 1) * k * k;
    if (m > P) return ORC_BAD_ARG;
    const int R = 1 + (D - 1) * k;
    const int n = m + 1;
    const int W = (n + 63) / 64;
    const size_t F = (size_t)(D > 1 ? D - 1 : 1) * k;
    int status = ORC_OK;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic) reduction(max : status)
#endif
    for (int b = 0; b < B; ++b) {
        double mg = INFINITY, dg = INFINITY;
        int s = build_one(V, D, k, m, tree_temp, draft_logits + (size_t)b * R * V,
                          child_u ? child_u + (size_t)b * R * k : NULL, root_token[b],
                          tokens + (size_t)b * n, parents + (size_t)b * n, depths + (size_t)b * n,
                          node_row + (size_t)b * n, mask + (size_t)b * n * W, node_logv + (size_t)b * n,
                          &mg, &dg, front_tok ? front_tok + b * F : NULL, front_par ? front_par + b * F : NULL);
        if (margin) margin[b] = mg;
        if (draw_gap) draw_gap[b] = dg;
        if (s > status) status = s;
    }
    (void)nthreads;
    return status;
}

int orc_build_tree(int B, int V, int D, int k, int m, double tree_temp, const float *draft_logits,
                   const int32_t *root_token, int32_t *tokens, int32_t *parents, int32_t *depths,
                   int32_t *node_row, uint64_t *mask, double *node_logv, double *margin, int nthreads)
{
    return orc_build_tree_ex(B, V, D, k, m, tree_temp, draft_logits, NULL, root_token, tokens, parents, depths,
                             node_row, mask, node_logv, margin, NULL, NULL, NULL, nthreads);
}

/* The children of N independent draft rows, as the builds take them: tok, lc [N][k]; u NULL for
 * the top k, else [N][k] uniforms (row_sample); gap [N][k] (optional, draws only): each draw's
 * distance to the CDF step that decided it. */
int orc_row_children(int N, int V, int k, double T, const float *x, const float *u, int32_t *tok, double *lc,
                     double *gap)
{
    if (N < 0 || V < 1 || k < 1 || k > V || !(T > 0)) return ORC_BAD_ARG;
    double *qbuf = (double *)calloc((size_t)V, sizeof(double));
    int *kids = (int *)calloc((size_t)k, sizeof(int));
    if (!qbuf || !kids) { free(qbuf); free(kids); return ORC_BAD_ARG; }
    for (int r = 0; r < N; ++r) {
        const float *row = x + (size_t)r * V;
        const double lse = row_logsumexp(row, V, T);
        for (int j = 0; j < k; ++j) {
            double g = INFINITY;
            if (u)
                row_sample(row, V, T, 1, u + (size_t)r * k + j, &kids[j], qbuf, &g);
            if (gap) gap[(size_t)r * k + j] = g;
        }
        if (!u) row_topk(row, V, k, kids);
        for (int j = 0; j < k; ++j) {
            tok[(size_t)r * k + j] = kids[j];
            lc[(size_t)r * k + j] = (double)row[kids[j]] / T - lse;
        }
    }
    free(qbuf);
    free(kids);
    return ORC_OK;
}

/* ------------------------------------------------------------------------------------------ */
/* 2. Tree attention  ([EAGLE-3 blog] section 5; [EAGLE-2 notes] Tree Attention Mask)           */
/* ------------------------------------------------------------------------------------------ */

typedef struct {
    int L, B, n, Hq, Hkv, d, S_max, W, dtype;
    double scale;
    const void *q, *k_cache, *v_cache, *k_tree, *v_tree;
    const int32_t *ctx_len;
    const uint64_t *mask;
} attn_args_t;

/* One query row: node i of sequence b, query head h, layer l.  Literal softmax over every key
 * the node may see (the whole cached context, and the tree nodes whose mask bit is set), then
 * the weighted sum of the values.  Head h reads KV head h / (Hq/Hkv). */
static void attn_row(const attn_args_t *a, int l, int b, int i, int h, double *out, double *s)
{
    const int d = a->d;
    const int G = a->Hq / a->Hkv;
    const int g = h / G;
    const int ctx = a->ctx_len[b];
    const size_t qoff = ((((size_t)l * a->B + b) * a->n + i) * a->Hq + h) * (size_t)d;
    int nk = 0;
    for (int j = 0; j < ctx; ++j) {
        size_t koff = ((((size_t)l * a->B + b) * a->S_max + j) * a->Hkv + g) * (size_t)d;
        double dot = 0.0;
        for (int e = 0; e < d; ++e) dot += load_elem(a->q, qoff + e, a->dtype) * load_elem(a->k_cache, koff + e, a->dtype);
        s[nk++] = dot * a->scale;
    }
    const uint64_t *mrow = a->mask + ((size_t)b * a->n + i) * a->W;
    for (int j = 0; j < a->n; ++j) {
        if (!((mrow[j / 64] >> (j % 64)) & 1ull)) continue;
        size_t koff = ((((size_t)l * a->B + b) * a->n + j) * a->Hkv + g) * (size_t)d;
        double dot = 0.0;
        for (int e = 0; e < d; ++e) dot += load_elem(a->q, qoff + e, a->dtype) * load_elem(a->k_tree, koff + e, a->dtype);
        s[nk++] = dot * a->scale;
    }
    double mx = -INFINITY;
    for (int j = 0; j < nk; ++j) if (s[j] > mx) mx = s[j];
    double den = 0.0;
    for (int j = 0; j < nk; ++j) { s[j] = exp(s[j] - mx); den += s[j]; }
    for (int e = 0; e < d; ++e) out[e] = 0.0;
    nk = 0;
    for (int j = 0; j < ctx; ++j) {
        size_t voff = ((((size_t)l * a->B + b) * a->S_max + j) * a->Hkv + g) * (size_t)d;
        double w = s[nk++] / den;
        for (int e = 0; e < d; ++e) out[e] += w * load_elem(a->v_cache, voff + e, a->dtype);
    }
    for (int j = 0; j < a->n; ++j) {
        if (!((mrow[j / 64] >> (j % 64)) & 1ull)) continue;
        size_t voff = ((((size_t)l * a->B + b) * a->n + j) * a->Hkv + g) * (size_t)d;
        double w = s[nk++] / den;
        for (int e = 0; e < d; ++e) out[e] += w * load_elem(a->v_tree, voff + e, a->dtype);
    }
}

static int attn_check(const attn_args_t *a)
{
    if (a->L < 1 || a->B < 0 || a->n < 1 || a->Hq < 1 || a->Hkv < 1 || a->Hq % a->Hkv || a->d < 1 || a->S_max < 0)
        return ORC_BAD_ARG;
    if (a->dtype != DT_F32 && a->dtype != DT_BF16) return ORC_BAD_ARG;
    for (int b = 0; b < a->B; ++b)
        if (a->ctx_len[b] < 0 || a->ctx_len[b] > a->S_max) return ORC_BAD_ARG;
    return ORC_OK;
}

/* Full attention for layers [l0, l1): out [L][B][n][Hq][d] (only those layers written). */
int orc_tree_attention(int L, int B, int n, int Hq, int Hkv, int d, int S_max, int dtype, double scale,
                       const void *q, const void *k_cache, const void *v_cache, const int32_t *ctx_len,
                       const void *k_tree, const void *v_tree, const uint64_t *mask, double *out,
                       int l0, int l1, int nthreads)
{
    attn_args_t a = {L, B, n, Hq, Hkv, d, S_max, (n + 63) / 64, dtype, scale,
                     q, k_cache, v_cache, k_tree, v_tree, ctx_len, mask};
    int st = attn_check(&a);
    if (st) return st;
    if (l0 < 0 || l1 > L || l0 > l1) return ORC_BAD_ARG;
    const long units = (long)(l1 - l0) * B * n * Hq;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel
#endif
    {
        double *s = (double *)malloc(sizeof(double) * ((size_t)S_max + n + 1));
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 4)
#endif
        for (long u = 0; u < units; ++u) {
            int h = (int)(u % Hq);
            int i = (int)((u / Hq) % n);
            int b = (int)((u / Hq / n) % B);
            int l = l0 + (int)(u / Hq / n / B);
            double *o = out + ((((size_t)l * B + b) * n + i) * Hq + h) * (size_t)d;
            attn_row(&a, l, b, i, h, o, s);
        }
        free(s);
    }
    (void)nthreads;
    return ORC_OK;
}

/* Selected rows only: rows[r] = (l, b, i, h); out [count][d]. */
int orc_tree_attention_rows(int L, int B, int n, int Hq, int Hkv, int d, int S_max, int dtype, double scale,
                            const void *q, const void *k_cache, const void *v_cache, const int32_t *ctx_len,
                            const void *k_tree, const void *v_tree, const uint64_t *mask,
                            const int32_t *rows, int count, double *out, int nthreads)
{
    attn_args_t a = {L, B, n, Hq, Hkv, d, S_max, (n + 63) / 64, dtype, scale,
                     q, k_cache, v_cache, k_tree, v_tree, ctx_len, mask};
    int st = attn_check(&a);
    if (st) return st;
    for (int r = 0; r < count; ++r) {
        const int32_t *x = rows + 4 * (size_t)r;
        if (x[0] < 0 || x[0] >= L || x[1] < 0 || x[1] >= B || x[2] < 0 || x[2] >= n || x[3] < 0 || x[3] >= Hq)
            return ORC_BAD_ARG;
    }
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel
#endif
    {
        double *s = (double *)malloc(sizeof(double) * ((size_t)S_max + n + 1));
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int r = 0; r < count; ++r) {
            const int32_t *x = rows + 4 * (size_t)r;
            attn_row(&a, x[0], x[1], x[2], x[3], out + (size_t)r * d, s);
        }
        free(s);
    }
    (void)nthreads;
    return ORC_OK;
}

/* ------------------------------------------------------------------------------------------ */
/* 3. Tree verification  ([EAGLE-1 notes] A3, 3.3, A.2; [EAGLE-3 blog] sections 1, 2, 5)      */
/* ------------------------------------------------------------------------------------------ */

/* p = softmax(x / T) */
static void softmax_T(const float *x, int V, double T, double *p)
{
    double lse = row_logsumexp(x, V, T);
    for (int t = 0; t < V; ++t) p[t] = exp((double)x[t] / T - lse);
}

/* Accept test of speculative sampling: ratio p(t)/q(t), +inf when q(t) = 0. */
static double accept_ratio(const double *p, const double *q, int t)
{
    if (q[t] > 0.0) return p[t] / q[t];
    return INFINITY;
}

/* After a rejection: p <- norm(max(0, p - q)); kept unchanged when the residual mass is 0. */
static void residual_update(double *p, const double *q, int V, double *tmp)
{
    double z = 0.0;
    for (int t = 0; t < V; ++t) {
        tmp[t] = p[t] - q[t] > 0.0 ? p[t] - q[t] : 0.0;
        z += tmp[t];
    }
    if (z > 0.0)
        for (int t = 0; t < V; ++t) p[t] = tmp[t] / z;
}

/* Inverse-CDF draw over ascending token id: the smallest j with sum_{t<=j} p_t > u, clamped to
 * the last token of non-zero probability.  *gap = distance of u to the nearest CDF step that
 * decided the draw. */
static int inverse_cdf(const double *p, int V, double u, double *gap)
{
    double c = 0.0, prev = 0.0;
    int last_pos = 0;
    for (int t = 0; t < V; ++t) {
        if (p[t] > 0.0) last_pos = t;
        prev = c;
        c += p[t];
        if (c > u) {
            double g1 = u - prev, g2 = c - u;
            *gap = g1 < g2 ? g1 : g2;
            return t;
        }
    }
    *gap = fabs(c - u);
    return last_pos;
}

static int kept_children(const int32_t *parents, int n, int a, int *out)
{
    int c = 0;
    for (int i = 1; i < n; ++i)
        if (parents[i] == a) out[c++] = i;
    return c;
}

static int verify_one(int V, int R, int n, int max_commit, double T, const float *target, const float *draft,
                      const int32_t *tokens, const int32_t *parents, const int32_t *node_row, const float *u,
                      int32_t *out_tokens, int32_t *out_len, int32_t *out_path, double *out_ratio, double *margin)
{
    double *p = (double *)malloc(sizeof(double) * V);
    double *q = (double *)malloc(sizeof(double) * V);
    double *tmp = (double *)malloc(sizeof(double) * V);
    int *kids = (int *)malloc(sizeof(int) * n);
    int status = ORC_OK;
    double mg = INFINITY;

    for (int i = 0; i < n; ++i) {
        if (i > 0 && (parents[i] < 0 || parents[i] >= i)) status = ORC_BAD_TREE;
        if (tokens[i] < 0 || tokens[i] >= V) status = ORC_BAD_TREE;
    }
    for (int j = 0; j < max_commit; ++j) out_tokens[j] = -1;
    for (int j = 0; j + 1 < max_commit; ++j) out_path[j] = -1;
    if (status) goto done;

    /* out_ratio: for every non-root node c, the ratio it is tested with when all of its earlier
     * siblings were rejected (the accept test never depends on u before it is reached). */
    if (out_ratio) {
        for (int i = 0; i < n; ++i) out_ratio[i] = NAN;
        if (T > 0.0) {
            for (int a = 0; a < n; ++a) {
                int nk = kept_children(parents, n, a, kids);
                if (nk == 0) continue;
                if (node_row[a] < 0 || node_row[a] >= R) { status = ORC_BAD_TREE; goto done; }
                softmax_T(target + (size_t)a * V, V, T, p);
                softmax_T(draft + (size_t)node_row[a] * V, V, T, q);
                for (int j = 0; j < nk; ++j) {
                    out_ratio[kids[j]] = accept_ratio(p, q, tokens[kids[j]]);
                    residual_update(p, q, V, tmp);
                }
            }
        }
    }

    int a = 0, len = 0;
    for (;;) {
        int nk = kept_children(parents, n, a, kids);
        if (T <= 0.0) {
            /* greedy: the target's argmax decides; follow the first child holding it */
            int g = row_argmax(target + (size_t)a * V, V);
            int next = -1;
            for (int j = 0; j < nk; ++j)
                if (tokens[kids[j]] == g) { next = kids[j]; break; }
            out_tokens[len] = g;
            if (next < 0) { ++len; break; }
            if (len + 1 >= max_commit) { status = ORC_BAD_TREE; break; }
            out_path[len] = next;
            ++len;
            a = next;
            continue;
        }
        softmax_T(target + (size_t)a * V, V, T, p);
        int accepted = -1;
        if (nk > 0) {
            if (node_row[a] < 0 || node_row[a] >= R) { status = ORC_BAD_TREE; break; }
            softmax_T(draft + (size_t)node_row[a] * V, V, T, q);
            for (int j = 0; j < nk; ++j) {
                int c = kids[j];
                double r = accept_ratio(p, q, tokens[c]);
                double gap = fabs((double)u[c] - r);
                if (gap < mg) mg = gap;
                if ((double)u[c] < r) { accepted = c; break; }
                residual_update(p, q, V, tmp);
            }
        }
        if (accepted >= 0) {
            if (len + 1 >= max_commit) { status = ORC_BAD_TREE; break; }
            out_tokens[len] = tokens[accepted];
            out_path[len] = accepted;
            ++len;
            a = accepted;
            continue;
        }
        double gap;
        out_tokens[len++] = inverse_cdf(p, V, (double)u[0], &gap);
        if (gap < mg) mg = gap;
        break;
    }
    *out_len = len;
done:
    if (margin) *margin = mg;
    free(p);
    free(q);
    free(tmp);
    free(kids);
    return status;
}

/*
 * Batched verification.
 *   target [B][n][V]: target logits of every tree node (row i = distribution after node i).
 *   draft  [B][R][V]: draft logits; node_row[i] names the row that proposed node i's children.
 *   u [B][n]: u[0] draws the final token, u[i>=1] is node i's accept test.
 *   outputs: out_tokens [B][max_commit], out_path [B][max_commit-1] (node ids), out_len [B],
 *            out_ratio [B][n] (optional), margin [B] (optional: smallest |u - decision value|).
 */
int orc_tree_verify(int B, int V, int R, int n, int max_commit, double T, const float *target,
                    const float *draft, const int32_t *tokens, const int32_t *parents, const int32_t *node_row,
                    const float *u, int32_t *out_tokens, int32_t *out_len, int32_t *out_path,
                    double *out_ratio, double *margin, int nthreads)
{
    if (B < 0 || V < 1 || R < 1 || n < 1 || max_commit < 1 || T < 0.0) return ORC_BAD_ARG;
    int status = ORC_OK;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 16) reduction(max : status)
#endif
    for (long b = 0; b < B; ++b) {
        int s = verify_one(V, R, n, max_commit, T, target + (size_t)b * n * V, draft + (size_t)b * R * V,
                           tokens + (size_t)b * n, parents + (size_t)b * n, node_row + (size_t)b * n,
                           u + (size_t)b * n, out_tokens + (size_t)b * max_commit, out_len + b,
                           out_path + (size_t)b * (max_commit > 1 ? max_commit - 1 : 1),
                           out_ratio ? out_ratio + (size_t)b * n : NULL, margin ? margin + b : NULL);
        if (s > status) status = s;
    }
    (void)nthreads;
    return status;
}

/* ------------------------------------------------------------------------------------------ */
/* Static tree and chain  ([EAGLE-1 notes] appendix A.1, section 4.3.1)                        */
/* ------------------------------------------------------------------------------------------ */

/* EAGLE-1 drafts a fixed tree: in the greedy setting a node's children are the top tokens of the
 * draft distribution at that node (appendix A.1); the chain of section 4.3.1 has one child per
 * node.  The tree is drawn only as a figure, so it is a template here (reading): tmpl[0] = -1,
 * tmpl[i] in [0, i).  The template nodes with children own the draft rows, in ascending index
 * (row r = the r-th such node); node p's children, in ascending index, take ranks 0, 1, ... of
 * its row's tokens under (value desc, id asc).  log V of a node is the sum of the
 * log-confidences (x/T - logsumexp(x/T) of the row) along its path; the root has 0. */
/* Sampled children (child_u != NULL, [B][R][kmax] with kmax = the most children of one template
 * node): node p's children, in ascending index, are draws 0, 1, ... of its row (row_sample),
 * draw j with child_u[b][row(p)][j].  draw_gap [B] (optional) as in orc_build_tree_ex. */
int orc_build_static_tree_ex(int B, int V, int n, const int32_t *tmpl, double tree_temp, const float *draft,
                             const float *child_u, const int32_t *root_token, int32_t *tokens, int32_t *parents,
                             int32_t *depths, int32_t *node_row, uint64_t *mask, double *node_logv,
                             double *draw_gap)
{
    if (B < 1 || V < 1 || n < 1 || n > 64 || !(tree_temp > 0.0) || tmpl[0] != -1) return ORC_BAD_ARG;
    int kids[64] = {0}, row_of[64];
    for (int i = 1; i < n; ++i) {
        if (tmpl[i] < 0 || tmpl[i] >= i) return ORC_BAD_ARG;
        ++kids[tmpl[i]];
    }
    int R = 0, kmax = 0;
    for (int i = 0; i < n; ++i) {
        if (kids[i] > V) return ORC_BAD_ARG;
        row_of[i] = kids[i] > 0 ? R++ : -1;
        if (kids[i] > kmax) kmax = kids[i];
    }
    int top[64][64];
    double lse[64];
    double *qbuf = child_u ? (double *)calloc((size_t)V, sizeof(double)) : NULL;
    if (child_u && !qbuf) return ORC_BAD_ARG;
    for (int b = 0; b < B; ++b) {
        double dg = INFINITY;
        for (int p = 0; p < n; ++p)
            if (row_of[p] >= 0) {
                const float *row = draft + ((size_t)b * R + row_of[p]) * V;
                lse[p] = row_logsumexp(row, V, tree_temp);
                row_children(row, V, tree_temp, kids[p],
                             child_u ? child_u + ((size_t)b * R + row_of[p]) * kmax : NULL, top[p], qbuf, &dg);
            }
        if (draw_gap) draw_gap[b] = dg;
        int32_t *tok = tokens + (size_t)b * n, *par = parents + (size_t)b * n, *dep = depths + (size_t)b * n;
        int32_t *nr = node_row + (size_t)b * n;
        uint64_t *mk = mask + (size_t)b * n;
        double *lv = node_logv + (size_t)b * n;
        tok[0] = root_token[b];
        par[0] = -1;
        dep[0] = 0;
        lv[0] = 0.0;
        mk[0] = 1ull;
        for (int i = 0; i < n; ++i) nr[i] = row_of[i];
        for (int i = 1; i < n; ++i) {  /* parents come first, so their values are already set */
            const int p = tmpl[i];
            int rank = 0;
            for (int j = p + 1; j < i; ++j) rank += tmpl[j] == p;
            const float *row = draft + ((size_t)b * R + row_of[p]) * V;
            tok[i] = top[p][rank];
            par[i] = p;
            dep[i] = dep[p] + 1;
            lv[i] = lv[p] + ((double)row[tok[i]] / tree_temp - lse[p]);
            mk[i] = mk[p] | (1ull << i);
        }
    }
    free(qbuf);
    return ORC_OK;
}

int orc_build_static_tree(int B, int V, int n, const int32_t *tmpl, double tree_temp, const float *draft,
                          const int32_t *root_token, int32_t *tokens, int32_t *parents, int32_t *depths,
                          int32_t *node_row, uint64_t *mask, double *node_logv)
{
    return orc_build_static_tree_ex(B, V, n, tmpl, tree_temp, draft, NULL, root_token, tokens, parents, depths,
                                    node_row, mask, node_logv, NULL);
}

/* ------------------------------------------------------------------------------------------ */
/* KV commit of the accepted path                                                             */
/* ------------------------------------------------------------------------------------------ */

/* After a round the committed tokens extend each sequence ([EAGLE-3 blog] section 1: the
 * accepted drafts and one more token; section 5: the tree pass computed every node's keys and
 * values at position ctx + depth).  Reading: the cache gains the root (node 0, position ctx_b)
 * and then the accepted nodes in path order (path entry i at position ctx_b + 1 + i), i.e. the
 * out_len[b] nodes root, path[0 .. out_len[b] - 2]; the last committed token has no keys or
 * values yet (it is the next round's root), so the new length is ctx_b + out_len[b].  A
 * sequence with out_len 0 (nothing committed) keeps its cache and length.  A sequence whose
 * count exceeds D + 1, whose path holds an id outside [1, n), or whose new length exceeds S_max
 * is also left as it was, and the call returns ORC_BAD_ARG.  Copies are bytewise (esize bytes
 * per element), one row of Hkv * d elements at a time. */
int orc_kv_commit(int L, int B, int n, int Hkv, int d, int S_max, int D, int esize, const void *k_tree,
                  const void *v_tree, const int32_t *out_path, const int32_t *out_len, const int32_t *ctx_len,
                  void *k_cache, void *v_cache, int32_t *new_ctx_len)
{
    if (L < 1 || B < 1 || n < 1 || Hkv < 1 || d < 1 || S_max < 1 || D < 0 || (esize != 2 && esize != 4))
        return ORC_BAD_ARG;
    const size_t row = (size_t)Hkv * d * esize;
    int status = ORC_OK;
    for (int b = 0; b < B; ++b) {
        const int ctx = ctx_len[b], len = out_len[b];
        new_ctx_len[b] = ctx;
        if (len == 0) continue;
        int ok = len >= 1 && len <= D + 1 && ctx >= 0 && ctx + len <= S_max;
        for (int i = 0; ok && i < len - 1; ++i) {
            const int node = out_path[(size_t)b * D + i];
            if (node < 1 || node >= n) ok = 0;
        }
        if (!ok) {
            status = ORC_BAD_ARG;
            continue;
        }
        for (int l = 0; l < L; ++l)
            for (int i = 0; i < len; ++i) {
                const int node = i == 0 ? 0 : out_path[(size_t)b * D + i - 1];
                const size_t src = (((size_t)l * B + b) * n + node) * row;
                const size_t dst = (((size_t)l * B + b) * S_max + ctx + i) * row;
                memcpy((char *)k_cache + dst, (const char *)k_tree + src, row);
                memcpy((char *)v_cache + dst, (const char *)v_tree + src, row);
            }
        new_ctx_len[b] = ctx + len;
    }
    return status;
}

int orc_version(void) { return 1; }
