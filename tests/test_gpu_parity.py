"""GPU parity: every stage through the C ABI against the fp64 oracle on the same seeded inputs.

Small cases compare every output element; the five workloads run at full size with every tree
index and committed token compared, and attention compared on sampled rows (launch configuration
identical to the benchmark's)."""
import numpy as np
import pytest
import torch

import datagen
import eagle_draft_tree_gb300 as eg
import oracle
from tests.gpu_parity import (ATTN_TOL, attention_sample_rows, compare_build, compare_verify, gpu_build, np_,
                              oracle_attention_rows, oracle_tree_tensors)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _draft(wl, seed, device=DEV):
    return datagen.draft_logits(wl.batch, wl.rows, wl.vocab, seed, device), datagen.root_tokens(wl.batch, wl.vocab, seed, device)


# ---------------------------------------------------------------- build

BUILD_SHAPES = [
    # (B, V, D, k, m)
    (1, 1000, 3, 4, 10), (3, 1000, 3, 4, 10), (2, 32000, 6, 10, 50), (2, 128256, 8, 10, 60),
    (4, 16, 2, 3, 12), (2, 500, 1, 5, 5), (2, 300, 5, 1, 5), (2, 4096, 4, 16, 63), (5, 777, 3, 7, 30),
    (2, 2048, 2, 2, 1), (2, 300, 64, 1, 63), (1, 2000, 11, 10, 63),
    # the full vocabulary over 101 rows (the largest pool at k = 10) and a depth-64 chain, and
    # 304 rows in all
    (1, 128256, 11, 10, 63), (1, 128256, 64, 1, 63), (4, 2000, 16, 5, 60),
]


@pytest.mark.parametrize("shape", BUILD_SHAPES)
@pytest.mark.parametrize("seed", [0, 1])
def test_build_tree_matches_oracle(shape, seed):
    B, V, D, k, m = shape
    wl = datagen.WORKLOADS["tiny_f32"].with_(batch=B, vocab=V, depth=D, topk=k, keep=m)
    draft, root = _draft(wl, 100 + seed)
    g = gpu_build(draft, root, wl)
    o = oracle.build_tree(np_(draft), np_(root), D, k, m)
    log = []
    excused = compare_build(g, o, log)
    assert len(excused) <= max(1, B // 8), log


def test_build_tree_equal_logit_ties():
    """Rows with repeated values: ties must go to the lower token id exactly as in the oracle."""
    wl = datagen.WORKLOADS["tiny_f32"].with_(batch=3, vocab=64, depth=3, topk=4, keep=12)
    g = torch.Generator().manual_seed(5)
    draft = torch.randint(-3, 3, (3, wl.rows, 64), generator=g).float().to(DEV)
    root = torch.zeros(3, dtype=torch.int32, device=DEV)
    gb = gpu_build(draft, root, wl)
    o = oracle.build_tree(np_(draft), np_(root), wl.depth, wl.topk, wl.keep)
    # integer logits produce exact value ties across parents only through equal log-sums; the
    # frontier/rerank then decide by creation order on both sides
    compare_build(gb, o)


def test_build_tree_bad_root_token_sets_status():
    wl = datagen.WORKLOADS["tiny_f32"]
    draft, _ = _draft(wl, 3)
    ws = eg.Workspace()
    root = torch.tensor([wl.vocab + 5], dtype=torch.int32, device=DEV)
    eg.build_tree(draft, root, depth=wl.depth, topk=wl.topk, keep=wl.keep, ws=ws)
    assert ws.status() == eg.EAGLE_ERR_DEVICE_INPUT
    assert ws.status() == eg.EAGLE_OK  # reading clears it


# ---------------------------------------------------------------- attention

ATTN_CASES = [
    # (L, B, n, Hq, Hkv, d, ctx list, dtype)
    (1, 1, 11, 4, 2, 64, [128], "f32"),
    (2, 3, 11, 4, 2, 64, [0, 1, 200], "f32"),
    (2, 2, 61, 8, 2, 128, [130, 64], "bf16"),
    (1, 3, 1, 4, 4, 128, [0, 63, 65], "bf16"),
    (2, 2, 64, 8, 1, 128, [191, 257], "bf16"),
    (1, 2, 49, 16, 2, 128, [300, 5], "bf16"),
    (2, 2, 20, 6, 6, 64, [77, 128], "bf16"),
    (1, 1, 51, 2, 2, 128, [1000], "bf16"),
    # query-head groups that do not divide 128: an M-tile holds floor(128 / G) whole nodes
    (2, 2, 61, 40, 8, 128, [300, 129], "bf16"),  # G = 5: 125-row tiles, a CTA's second tile partial
    (1, 2, 64, 21, 3, 128, [257, 0], "bf16"),    # G = 7: 126-row tiles, two CTAs a unit
    (1, 1, 30, 24, 8, 128, [130], "bf16"),       # G = 3: one 90-row tile
    (1, 1, 61, 40, 8, 128, [2048], "bf16"),      # G = 5 with the context split and its merge
    # d = 64 on the tensor cores (a zero upper half through the tensor maps' out-of-range fill)
    (2, 2, 61, 32, 8, 64, [300, 129], "bf16"),
    (1, 1, 40, 16, 4, 64, [2048], "bf16"),        # with the context split
]


def _attn_inputs(L, B, n, Hq, Hkv, d, ctx, dtype, seed):
    S = max(max(ctx), 1)
    wl = datagen.WORKLOADS["tiny_f32"].with_(layers=L, batch=B, keep=n - 1, heads_q=Hq, heads_kv=Hkv, head_dim=d,
                                             ctx=S, ctx_min=S, kv_dtype=dtype)
    inp = datagen.attention_inputs(wl, seed, DEV)
    inp["ctx_len"] = torch.tensor(ctx, dtype=torch.int32, device=DEV)
    # a random tree for the mask
    rng = np.random.default_rng(seed)
    par = [[-1] + [int(rng.integers(0, i)) for i in range(1, n)] for _ in range(B)]
    mask = np.zeros((B, n, 1), np.uint64)
    for b in range(B):
        for i in range(n):
            j, w = i, 0
            while j >= 0:
                w |= 1 << j
                j = par[b][j]
            mask[b, i, 0] = w
    return wl, inp, mask


@pytest.mark.parametrize("case", ATTN_CASES, ids=lambda c: f"L{c[0]}B{c[1]}n{c[2]}G{c[3]//c[4]}d{c[5]}{c[7]}")
def test_tree_attention_matches_oracle(case):
    L, B, n, Hq, Hkv, d, ctx, dtype = case
    wl, inp, mask = _attn_inputs(L, B, n, Hq, Hkv, d, ctx, dtype, seed=17 + n)
    mask_t = torch.from_numpy(mask.reshape(B, n).view(np.int64).copy()).to(DEV)
    out = eg.tree_attention(inp["q"], inp["k_cache"], inp["v_cache"], inp["ctx_len"], inp["k_tree"],
                            inp["v_tree"], mask_t)
    torch.cuda.synchronize()
    ref = oracle.tree_attention(np_(inp["q"]), np_(inp["k_cache"]), np_(inp["v_cache"]), np_(inp["ctx_len"]),
                                np_(inp["k_tree"]), np_(inp["v_tree"]), mask)
    got = out.float().cpu().numpy().astype(np.float64)
    err = np.abs(got - ref).max()
    assert err <= ATTN_TOL[dtype], err


@pytest.mark.parametrize("d", [64, 128])
def test_bf16_attention_takes_the_tensor_core_path(d):
    """Few units: the tensor-core kernel splits the context and merges (two launches); the
    mma.sync kernel it would otherwise fall back to is one launch."""
    wl, inp, mask = _attn_inputs(1, 1, 40, 16, 4, d, [2048], "bf16", seed=5)
    mask_t = torch.from_numpy(mask.reshape(1, 40).view(np.int64).copy()).to(DEV)
    eg.tree_attention(inp["q"], inp["k_cache"], inp["v_cache"], inp["ctx_len"], inp["k_tree"], inp["v_tree"], mask_t)
    torch.cuda.synchronize()
    assert eg.last_launch_count() == 2


@pytest.mark.parametrize("case", [c for c in ATTN_CASES if min(c[6]) < max(c[6])],
                         ids=lambda c: f"L{c[0]}B{c[1]}n{c[2]}G{c[3]//c[4]}d{c[5]}{c[7]}")
def test_tree_attention_ignores_cache_past_context(case):
    """Cache positions at or past ctx_len[b] may hold anything, NaN included: the output is unchanged."""
    L, B, n, Hq, Hkv, d, ctx, dtype = case
    wl, inp, mask = _attn_inputs(L, B, n, Hq, Hkv, d, ctx, dtype, seed=5 + n)
    mask_t = torch.from_numpy(mask.reshape(B, n).view(np.int64).copy()).to(DEV)
    args = lambda: (inp["q"], inp["k_cache"], inp["v_cache"], inp["ctx_len"], inp["k_tree"], inp["v_tree"], mask_t)
    clean = eg.tree_attention(*args())
    for b, c in enumerate(ctx):
        inp["k_cache"][:, b, c:] = float("nan")
        inp["v_cache"][:, b, c:] = float("nan")
    dirty = eg.tree_attention(*args())
    torch.cuda.synchronize()
    assert torch.isfinite(dirty.float()).all()
    assert torch.equal(dirty, clean)


def test_tree_attention_chain_equals_causal_on_gpu():
    """A chain tree through the library equals causal attention computed by torch in fp64."""
    L, B, n, Hq, Hkv, d = 1, 1, 12, 4, 2, 128
    wl, inp, _ = _attn_inputs(L, B, n, Hq, Hkv, d, [96], "bf16", seed=3)
    mask = np.array([[(1 << (i + 1)) - 1 for i in range(n)]], np.int64)
    out = eg.tree_attention(inp["q"], inp["k_cache"], inp["v_cache"], inp["ctx_len"], inp["k_tree"], inp["v_tree"],
                            torch.from_numpy(mask).to(DEV))
    k = torch.cat([inp["k_cache"][0, 0, :96], inp["k_tree"][0, 0]], 0).double().transpose(0, 1)
    v = torch.cat([inp["v_cache"][0, 0, :96], inp["v_tree"][0, 0]], 0).double().transpose(0, 1)
    q = inp["q"][0, 0].double().transpose(0, 1)
    allowed = torch.ones((n, 96 + n), dtype=torch.bool, device=DEV)
    allowed[:, 96:] = torch.tril(torch.ones((n, n), dtype=torch.bool, device=DEV))
    ref = torch.nn.functional.scaled_dot_product_attention(q, k.repeat_interleave(2, 0), v.repeat_interleave(2, 0),
                                                           attn_mask=allowed).transpose(0, 1)
    assert (out[0, 0].double() - ref).abs().max().item() <= 2e-2


def test_tree_attention_bad_context_sets_status():
    wl, inp, mask = _attn_inputs(1, 2, 5, 2, 1, 64, [10, 10], "bf16", seed=1)
    inp["ctx_len"] = torch.tensor([10, 11], dtype=torch.int32, device=DEV)  # 11 > S_max
    ws = eg.Workspace()
    eg.tree_attention(inp["q"], inp["k_cache"], inp["v_cache"], inp["ctx_len"], inp["k_tree"], inp["v_tree"],
                      torch.from_numpy(mask.reshape(2, 5).view(np.int64).copy()).to(DEV), ws=ws)
    assert ws.status() == eg.EAGLE_ERR_DEVICE_INPUT


# ---------------------------------------------------------------- verify

def _verify_case(wl, seed, T, with_ratio=True):
    draft, root = _draft(wl, seed)
    o_tree = oracle.build_tree(np_(draft), np_(root), wl.depth, wl.topk, wl.keep)
    sig = datagen.noise_sigmas(wl, seed)
    target = datagen.target_logits(draft, torch.from_numpy(o_tree["node_row"]).to(DEV), sig, seed)
    u = datagen.uniforms(wl.batch, wl.nodes, seed, DEV)
    tree = oracle_tree_tensors(o_tree, DEV)
    g = eg.tree_verify(target, draft, tree, u, temperature=T, depth=wl.depth, topk=wl.topk, with_ratio=with_ratio)
    torch.cuda.synchronize()
    g = {k: np_(v) for k, v in g.items() if v is not None}
    o = oracle.tree_verify(np_(target), np_(draft), o_tree["tokens"], o_tree["parents"], o_tree["node_row"], np_(u),
                           T, wl.depth + 1)
    o["parents"] = o_tree["parents"]
    return g, o


VERIFY_SHAPES = [(4, 1000, 3, 4, 10), (2, 32000, 6, 10, 50), (2, 128256, 8, 10, 60), (8, 64, 3, 3, 12),
                 (3, 5000, 1, 6, 6), (3, 999, 4, 1, 4)]


@pytest.mark.parametrize("shape", VERIFY_SHAPES)
@pytest.mark.parametrize("T", [1.0, 0.7, 0.0])
@pytest.mark.parametrize("with_ratio", [True, False], ids=["ratios", "first-accept"])
def test_tree_verify_matches_oracle(shape, T, with_ratio):
    """With every child's ratio requested the prep tests every child; without, a node's chain
    stops at its first accepted child.  The committed tokens and path are the same either way."""
    B, V, D, k, m = shape
    wl = datagen.WORKLOADS["tiny_f32"].with_(batch=B, vocab=V, depth=D, topk=k, keep=m)
    for seed in (0, 1):
        g, o = _verify_case(wl, 40 + seed, T, with_ratio)
        log = []
        excused = compare_verify(g, o, log)
        assert len(excused) <= max(1, B // 8), log


def test_tree_verify_low_noise_accepts_deep_paths():
    """With the target equal to the draft the path is accepted to depth D almost always; this
    drives the walk through every depth (parity still exact)."""
    wl = datagen.WORKLOADS["tiny_f32"].with_(batch=8, vocab=500, depth=5, topk=3, keep=20, noise=0.0)
    g, o = _verify_case(wl, 9, 1.0)
    compare_verify(g, o)
    assert o["out_len"].max() >= 4


@pytest.mark.parametrize("shape", [(4, 128256, 8, 10, 60), (3, 150000, 4, 4, 20), (6, 1000, 3, 4, 10)])
@pytest.mark.parametrize("T", [1.0, 0.7])
@pytest.mark.parametrize("with_ratio", [True, False], ids=["ratios", "first-accept"])
def test_tree_verify_bonus_token_at_a_leaf(shape, T, with_ratio):
    """Target rows equal to their draft rows make every accept ratio exactly 1, so every walk
    accepts down to a leaf and ends with the bonus token drawn from that leaf's target
    distribution (the draw made for that one leaf after the walk).  Both slice widths (8 and 16
    CTAs per row) are covered."""
    B, V, D, k, m = shape
    wl = datagen.WORKLOADS["tiny_f32"].with_(batch=B, vocab=V, depth=D, topk=k, keep=m, noise=0.0)
    g, o = _verify_case(wl, 77, T, with_ratio)
    assert not compare_verify(g, o)
    draft, root = _draft(wl, 77)
    parents = oracle.build_tree(np_(draft), np_(root), D, k, m)["parents"]
    for b in range(B):
        L = int(g["out_len"][b])
        path = [int(x) for x in g["out_path"][b][:L - 1]]
        end = path[-1] if path else 0
        assert end not in set(int(x) for x in parents[b]), f"sequence {b} did not end at a leaf"
        assert int(g["out_tokens"][b][L - 1]) >= 0


@pytest.mark.parametrize("T", [1.0, 0.0])
def test_tree_verify_repeated_calls_on_a_stale_workspace(T):
    """Repeated calls on one workspace, and calls on a workspace whose body holds stale bytes
    (another call's scratch), commit the same tokens; launches: the prep and the walk, plus the
    bonus launch when sampling with every ratio wanted."""
    wl = datagen.WORKLOADS["tiny_f32"].with_(batch=3, vocab=32000, depth=6, topk=10, keep=50)
    seed = 5
    draft, root = _draft(wl, seed)
    o_tree = oracle.build_tree(np_(draft), np_(root), wl.depth, wl.topk, wl.keep)
    target = datagen.target_logits(draft, torch.from_numpy(o_tree["node_row"]).to(DEV),
                                   datagen.noise_sigmas(wl, seed), seed)
    u = datagen.uniforms(wl.batch, wl.nodes, seed, DEV)
    tree = oracle_tree_tensors(o_tree, DEV)
    ws = eg.Workspace()
    args = (target, draft, tree, u)
    kw = dict(temperature=T, depth=wl.depth, topk=wl.topk, ws=ws)
    ref = eg.tree_verify(*args, with_ratio=True, **kw)
    assert eg.last_launch_count() == (2 if T == 0.0 else 3)
    ref = {k: v.clone() for k, v in ref.items() if v is not None}
    o = oracle.tree_verify(np_(target), np_(draft), o_tree["tokens"], o_tree["parents"], o_tree["node_row"], np_(u),
                           T, wl.depth + 1)
    o["parents"] = o_tree["parents"]
    compare_verify({k: np_(v) for k, v in ref.items()}, o)
    for fill in (None, None, 0xFF, 0x00, 0x5A):
        if fill is not None:  # everything past the status header
            off = ws.ptr.value - ws.buf.data_ptr()
            ws.buf[off + 256:].fill_(fill)
        g = eg.tree_verify(*args, with_ratio=False, **kw)
        assert eg.last_launch_count() == 2
        for key in ("out_tokens", "out_len", "out_path"):
            assert torch.equal(g[key], ref[key]), (fill, key)
    assert ws.status() == eg.EAGLE_OK


def test_tree_verify_bad_tree_sets_status():
    wl = datagen.WORKLOADS["tiny_f32"].with_(batch=2)
    draft, root = _draft(wl, 1)
    o_tree = oracle.build_tree(np_(draft), np_(root), wl.depth, wl.topk, wl.keep)
    tree = oracle_tree_tensors(o_tree, DEV)
    tree["parents"][1, 3] = 7  # parent after child
    target = datagen.target_logits(draft, tree["node_row"], datagen.noise_sigmas(wl, 1), 1)
    u = datagen.uniforms(wl.batch, wl.nodes, 1, DEV)
    ws = eg.Workspace()
    r = eg.tree_verify(target, draft, tree, u, temperature=1.0, depth=wl.depth, topk=wl.topk, ws=ws)
    assert ws.status() == eg.EAGLE_ERR_DEVICE_INPUT
    assert int(r["out_len"][1]) == 0 and int(r["out_len"][0]) >= 1
