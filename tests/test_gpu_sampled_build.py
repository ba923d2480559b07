"""GPU parity of the sampled-children builds (eagle_build_tree_sampled,
eagle_build_static_tree_sampled) and of the stepwise build (eagle_build_begin / _expand /
_finalize) against the oracle, plus end-to-end losslessness of build -> verify on the GPU.

Tolerances: tree indices and masks bit-exact.  A sequence may differ only where the oracle's
smallest relative key gap at a selection boundary is < 1e-6 or one of its uniforms lies within
draw_excuse(V) of the CDF step that decided its draw.  The kernel forms each weight's exponent
without rounding error (TwoSum, an FMA product, one rounding of a fraction in [-1/2, 1/2]), takes
2^f from the SFU (relative error at most EX2_BOUND, checked by eagle_selftest_exp2_error) and sums
the weights exactly as integers in units of 2^-S, S = 62 - ceil(log2 V).  A CDF step A / (A + B)
with weights off by relative errors within +-e moves by at most e / 2 (the worst case puts +e on
A and -e on B at A = B), and the truncations move it by at most V 2^-S, so a draw farther than
draw_excuse(V) from a step is decided alike.  node_logv to 1e-5 relative.  The stepwise build must
equal the one-call build bit for bit, on the same rows.
"""
import math
import numpy as np
import pytest
import torch
from scipy.special import softmax
from scipy.stats import chisquare

import datagen
import eagle_draft_tree_gb300 as eg
import oracle
from tests.gpu_parity import BUILD_EXCUSE, np_
from tests.test_oracle_static_tree import random_template

pytestmark = pytest.mark.gpu
DEV = "cuda"
EX2_BOUND = 1.5e-7  # the SFU's 2^f on |f| <= 1/2: eagle_selftest_exp2_error measured 1.46e-7 on GB300


def draw_excuse(V):
    """Largest distance from a uniform to a CDF step at which the kernel's draw may differ."""
    S = 62 - math.ceil(math.log2(V))
    return (EX2_BOUND + 2.0 ** -25 * math.log(2.0)) / 2 + V * 2.0 ** -S
KEYS = ("tokens", "parents", "depths", "node_row", "mask")


def _same(g, o, b):
    gm = np_(g["mask"]).view(np.uint64).reshape(o["mask"].shape[0], -1)
    return (all(np.array_equal(np_(g[k])[b], o[k][b]) for k in KEYS[:4])
            and np.array_equal(gm[b], o["mask"][b, :, 0]))


def _valid_tree(g, B, V):
    """Structure every build output has, whatever its draws: parents precede children, depths
    step by one, masks are the ancestor closure, log V never increases along a path."""
    tok, par, dep = np_(g["tokens"]), np_(g["parents"]), np_(g["depths"])
    mask, lv = np_(g["mask"]).view(np.uint64), np_(g["node_logv"])
    for b in range(B):
        assert par[b, 0] == -1 and dep[b, 0] == 0 and mask[b, 0] == 1
        for i in range(1, tok.shape[1]):
            p = par[b, i]
            assert 0 <= p < i and dep[b, i] == dep[b, p] + 1 and 0 <= tok[b, i] < V
            assert mask[b, i] == (mask[b, p] | np.uint64(1 << i))
            assert lv[b, i] <= lv[b, p] + 1e-6 * (1.0 + abs(lv[b, p]))


def _compare(g, o, V, bounded=True):
    """Bit-exact where the oracle's decisions are clear of the excuse bands; returns the number of
    excused sequences (at most a quarter when ``bounded``)."""
    B = o["tokens"].shape[0]
    excused = 0
    for b in range(B):
        if not _same(g, o, b):
            m, dg = o["margin"][b] if "margin" in o else np.inf, o["draw_gap"][b]
            assert m < BUILD_EXCUSE or dg < draw_excuse(V), f"sequence {b} differs (margin {m:.3g}, draw gap {dg:.3g})"
            excused += 1
            continue
        np.testing.assert_allclose(np_(g["node_logv"])[b].astype(np.float64), o["node_logv"][b], rtol=1e-5,
                                   atol=1e-6)
    if bounded:
        assert excused <= B // 4, f"{excused} of {B} sequences excused"
    return excused


def _inputs(B, V, D, k, seed):
    R = 1 + (D - 1) * k
    draft = datagen.draft_logits(B, R, V, seed, DEV)
    cu = datagen.child_uniforms(B, R, k, seed, DEV)
    root = datagen.root_tokens(B, V, seed, DEV)
    return draft, cu, root


def _clear_uniforms(draft, cu, T):
    """The uniforms with every one that lies within 2 draw_excuse(V) of a step of its row's CDF
    (float64, as the oracle forms it) moved to the middle of the row's most probable token's
    interval, so that every draw of a build is decided alike by the kernel and the oracle."""
    x, u = np_(draft).astype(np.float64), np_(cu).copy()
    band = 2 * draw_excuse(x.shape[-1])
    for b in range(x.shape[0]):
        for r in range(x.shape[1]):
            cdf = np.cumsum(softmax(x[b, r] / T))
            for j in range(u.shape[2]):
                t = int(np.searchsorted(cdf, u[b, r, j], side="right"))
                lo, hi = (cdf[t - 1] if t > 0 else 0.0), cdf[min(t, len(cdf) - 1)]
                if min(u[b, r, j] - lo, hi - u[b, r, j]) < band:
                    a = int(np.argmax(x[b, r]))
                    u[b, r, j] = ((cdf[a - 1] if a > 0 else 0.0) + cdf[a]) / 2
    return torch.tensor(u, device=cu.device)


def test_the_sfu_exponential_is_within_the_bound_the_bands_assume():
    e = eg.selftest_exp2_error()
    assert 0.0 < e <= EX2_BOUND, e


ROWS = [  # rows, V, k, T: every draw compared on its own (a depth-1 build keeps all k in draw order)
    (51, 128256, 10, 1.0),   # the rows of one sequence of the 8B-vocabulary tree
    (102, 32000, 10, 1.0),
    (40, 128256, 10, 0.7),
    (200, 300000, 4, 1.0),   # two CTAs a row, 74 chunk columns each
    (64, 1003, 16, 1.0),     # V not a multiple of 4 (scalar loads); k = 16 uses every warp
    (8, 5, 5, 1.0),          # a vocabulary below one chunk column
]


@pytest.mark.parametrize("N,V,k,T", ROWS)
def test_row_draws_match_oracle(N, V, k, T):
    """Each draw is the oracle's unless its uniform lies within draw_excuse(V) of the deciding CDF
    step; such a draw must still land within draw_excuse(V) of its own CDF interval.  At V =
    128256 about 3 % of the draws are that close to a step."""
    x = datagen.draft_logits(N, 1, V, N + V, DEV)
    u = datagen.child_uniforms(N, 1, k, N + k, DEV)
    root = torch.zeros(N, dtype=torch.int32, device=DEV)
    ws = eg.Workspace(device=DEV)
    g = eg.build_tree(x, root, 1, k, k, T, ws=ws, child_u=u)
    assert ws.status() == eg.EAGLE_OK
    gt, glv = np_(g["tokens"])[:, 1:], np_(g["node_logv"])[:, 1:].astype(np.float64)
    xn, un = np_(x)[:, 0], np_(u)[:, 0]
    o = oracle.row_children(xn, k, T, child_u=un)
    band = draw_excuse(V)
    clear = o["gap"] >= band
    assert np.array_equal(gt[clear], o["tok"][clear])
    np.testing.assert_allclose(glv[clear], o["lc"][clear], rtol=1e-5, atol=1e-6)
    for r, j in zip(*np.nonzero(~clear)):
        cdf = np.cumsum(softmax(xn[r].astype(np.float64) / T))
        t = gt[r, j]
        lo_ = cdf[t - 1] if t > 0 else 0.0
        assert lo_ - band <= float(un[r, j]) < cdf[t] + band
    assert clear.mean() > (0.9 if V <= 300000 else 0.5)


SHAPES = [  # B, V, D, k, m, T: whole trees (small vocabularies: almost every draw is clear)
    (8, 1000, 3, 4, 10, 1.0),
    (4, 1003, 4, 3, 20, 0.7),     # V not a multiple of 4: scalar loads
    (6, 5000, 2, 16, 63, 1.0),    # k = 16: one warp per draw, all 16 warps
    (16, 300, 6, 10, 60, 1.0),
    (2, 300, 64, 1, 63, 1.0),     # the deepest tree: a chain of 64 depths
    (1, 2000, 11, 10, 63, 1.0),   # a pool of 1010 candidates
]


@pytest.mark.parametrize("B,V,D,k,m,T", SHAPES)
def test_sampled_build_matches_oracle(B, V, D, k, m, T):
    seed = B * 7 + D
    draft, cu, root = _inputs(B, V, D, k, seed)
    ws = eg.Workspace(device=DEV)
    g = eg.build_tree(draft, root, D, k, m, T, ws=ws, child_u=cu)
    assert ws.status() == eg.EAGLE_OK
    o = oracle.build_tree(np_(draft), np_(root), D, k, m, T, child_u=np_(cu))
    _valid_tree(g, B, V)
    _compare(g, o, V)


@pytest.mark.parametrize("B,V", [(2, 32000), (2, 128256)])
def test_sampled_build_at_full_vocabulary(B, V):
    """Full-size trees (D = 6, k = 10, m = 60) with every draw clear of the excuse band (the few
    uniforms near a step moved, see _clear_uniforms; the per-draw test above covers such
    uniforms): equal to the oracle bit for bit but for selection ties."""
    draft, cu, root = _inputs(B, V, 6, 10, 77 + B)
    cu = _clear_uniforms(draft, cu, 1.0)
    g = eg.build_tree(draft, root, 6, 10, 60, 1.0, child_u=cu)
    o = oracle.build_tree(np_(draft), np_(root), 6, 10, 60, 1.0, child_u=np_(cu))
    _valid_tree(g, B, V)
    assert (o["draw_gap"] >= draw_excuse(V)).all()
    assert _compare(g, o, V) == 0 or (o["margin"] < BUILD_EXCUSE).any()


def test_sampled_static_matches_oracle():
    for seed, (tmpl, B, V, T) in enumerate([(eg.chain_template(5), 3, 128256, 1.0),
                                           ([-1] + [0] * 16, 2, 1000, 0.8),
                                           (random_template(np.random.default_rng(4), 40), 4, 32000, 1.0)]):
        internal = len(set(tmpl[1:]))
        kmax = max(sum(1 for p in tmpl[1:] if p == q) for q in range(len(tmpl)))
        draft = datagen.draft_logits(B, internal, V, seed, DEV)
        cu = datagen.child_uniforms(B, internal, kmax, seed, DEV)
        root = datagen.root_tokens(B, V, seed, DEV)
        ws = eg.Workspace(device=DEV)
        g = eg.build_static_tree(draft, root, tmpl, T, ws=ws, child_u=cu)
        assert ws.status() == eg.EAGLE_OK
        o = oracle.build_static_tree(np_(draft), np_(root), tmpl, T, child_u=np_(cu))
        _valid_tree(g, B, V)
        _compare(g, o, V, bounded=V <= 5000)


def test_repeated_draws_of_a_peaked_row():
    """Rows where one token holds about 0.9 of the mass: siblings repeat that token.  (Not 1 - 1e-12:
    log-confidences within ~1e-7 of 0 make the values of different rows tie to within the
    kernel's log-normaliser error, and exact ties across parents only the oracle resolves.)"""
    B, V, D, k, m = 4, 2000, 3, 4, 20
    draft, cu, root = _inputs(B, V, D, k, 9)
    draft[:, :, 17] = 12.0  # e^12 against ~V e^2 for the rest
    g = eg.build_tree(draft, root, D, k, m, 1.0, child_u=cu)
    o = oracle.build_tree(np_(draft), np_(root), D, k, m, 1.0, child_u=np_(cu))
    _valid_tree(g, B, V)
    _compare(g, o, V)
    tok, par = np_(g["tokens"]), np_(g["parents"])
    assert (tok[:, 1:] == 17).mean() > 0.7
    assert any(len({(int(par[b, i]), int(tok[b, i])) for i in range(1, m + 1)}) < m for b in range(B))


def _stepwise(draft, cu, root, D, k, m, T, ws=None):
    B = draft.shape[0]
    st = eg.BuildState(B, draft.shape[2], D, k, m, T, ws=ws, device=DEV)
    fronts = []
    f = eg.build_begin(st, draft[:, 0].contiguous(), None if cu is None else cu[:, :1].contiguous())
    if f is not None:
        fronts.append(tuple(np_(t).copy() for t in f))
    for d in range(1, D):
        rows = slice(1 + (d - 1) * k, 1 + d * k)
        f = eg.build_expand(st, d, draft[:, rows].contiguous(), None if cu is None else cu[:, rows].contiguous())
        if f is not None:
            fronts.append(tuple(np_(t).copy() for t in f))
    out = eg.build_finalize(st, root)
    return out, fronts, st


@pytest.mark.parametrize("B,V,D,k,m", [(3, 1000, 1, 4, 4), (4, 1000, 2, 4, 12), (5, 32000, 4, 6, 40),
                                       (2, 128256, 6, 10, 60), (3, 1001, 5, 2, 16)])
@pytest.mark.parametrize("sampled", [False, True])
def test_stepwise_equals_one_call_and_reports_the_frontiers(B, V, D, k, m, sampled):
    draft, cu, root = _inputs(B, V, D, k, 40 + D)
    cu = cu if sampled else None
    whole = eg.build_tree(draft, root, D, k, m, 1.0, child_u=cu)
    steps, fronts, st = _stepwise(draft, cu, root, D, k, m, 1.0)
    assert st.ws.status() == eg.EAGLE_OK
    for key in ("tokens", "parents", "depths", "node_row", "mask", "node_logv"):
        assert torch.equal(whole[key], steps[key]), key
    o = oracle.build_tree(np_(draft), np_(root), D, k, m, 1.0, child_u=None if cu is None else np_(cu),
                          frontier=True)
    _compare(steps, o, V, bounded=V <= 5000)
    assert len(fronts) == max(D - 1, 0)
    for f, (ft, fp) in enumerate(fronts):
        ok = [b for b in range(B) if _same(steps, o, b)]
        assert np.array_equal(ft[ok], o["front_tok"][ok, f]) and np.array_equal(fp[ok], o["front_par"][ok, f])


@pytest.mark.parametrize("sampled", [False, True])
def test_stepwise_at_the_serving_batch(sampled):
    """The serving workload's shape (B = 64, V = 128256, D = 8, k = 10, m = 60): the stepwise build
    equals the one-call build bit for bit; trees are valid; with every draw clear of the excuse
    band, equal to the oracle but for selection ties."""
    B, V, D, k, m = 64, 128256, 8, 10, 60
    draft, cu, root = _inputs(B, V, D, k, 64)
    cu = _clear_uniforms(draft, cu, 1.0) if sampled else None
    whole = eg.build_tree(draft, root, D, k, m, 1.0, child_u=cu)
    steps, fronts, st = _stepwise(draft, cu, root, D, k, m, 1.0)
    assert st.ws.status() == eg.EAGLE_OK
    for key in ("tokens", "parents", "depths", "node_row", "mask", "node_logv"):
        assert torch.equal(whole[key], steps[key]), key
    _valid_tree(steps, B, V)
    o = oracle.build_tree(np_(draft), np_(root), D, k, m, 1.0, child_u=None if cu is None else np_(cu))
    excused = _compare(steps, o, V)
    assert excused <= int((o["margin"] < BUILD_EXCUSE).sum())


def test_finalize_on_a_fresh_state_is_flagged():
    B, V, D, k, m = 2, 500, 3, 3, 9
    root = datagen.root_tokens(B, V, 1, DEV)
    st = eg.BuildState(B, V, D, k, m, device=DEV)
    eg.build_finalize(st, root)
    assert st.ws.status() == eg.EAGLE_ERR_DEVICE_INPUT  # depth-2 slots of a zeroed state are out of range


def test_row_without_a_finite_logit_is_flagged():
    B, V, D, k, m = 2, 700, 2, 2, 4
    draft, cu, root = _inputs(B, V, D, k, 5)
    draft[1, 0] = -float("inf")
    ws = eg.Workspace(device=DEV)
    g = eg.build_tree(draft, root, D, k, m, 1.0, ws=ws, child_u=cu)
    assert ws.status() == eg.EAGLE_ERR_DEVICE_INPUT
    assert (np_(g["tokens"])[1, 1:3] == 0).all()


# ---- end to end on the GPU: sampled children, then verification, commit the target law ----

def _logits(p):
    return np.log(np.maximum(p, 1e-30)).astype(np.float32)


def test_gpu_static_sampled_build_then_verify_is_lossless():
    V, k, B, calls = 16, 3, 65535, 4
    rng = np.random.default_rng(31)
    p = rng.dirichlet(np.ones(V))
    q = rng.dirichlet(np.full(V, 0.5))
    p2 = torch.tensor(_logits(rng.dirichlet(np.ones(V), size=V)), device=DEV)
    tmpl = [-1, 0, 0, 0]
    dft = torch.tensor(_logits(q), device=DEV).expand(B, 1, V).contiguous()
    root = torch.zeros(B, dtype=torch.int32, device=DEV)
    counts = np.zeros(V, np.int64)
    for c in range(calls):
        cu = datagen.child_uniforms(B, 1, k, 100 + c, DEV)
        t = eg.build_static_tree(dft, root, tmpl, 1.0, child_u=cu)
        tgt = torch.empty((B, k + 1, V), dtype=torch.float32, device=DEV)
        tgt[:, 0] = torch.tensor(_logits(p), device=DEV)
        tgt[:, 1:] = p2[t["tokens"][:, 1:].long()]
        u = datagen.uniforms(B, k + 1, 200 + c, DEV)
        o = eg.tree_verify(tgt, dft, t, u, 1.0, depth=1, topk=k)
        counts += np.bincount(np_(o["out_tokens"])[:, 0], minlength=V)
    pe = softmax(_logits(p).astype(np.float64))
    assert chisquare(counts, pe * counts.sum()).pvalue > 1e-3


def test_gpu_stepwise_sampled_build_then_verify_is_lossless():
    """A draft 'model' that is a table q2[token] feeds each depth-1 frontier slot its row; every
    candidate kept (m = k + k^2).  First committed token ~ p; second, given an accepted first
    token t, ~ p2[t]."""
    V, k, D, B, calls = 12, 2, 2, 65535, 4
    m = k + k * k
    rng = np.random.default_rng(17)
    p = rng.dirichlet(np.ones(V))
    q = rng.dirichlet(np.full(V, 0.5))
    p2 = rng.dirichlet(np.ones(V), size=V)
    q2 = torch.tensor(_logits(rng.dirichlet(np.full(V, 0.5), size=V)), device=DEV)
    p2_t = torch.tensor(_logits(p2), device=DEV)
    p3_t = torch.tensor(_logits(rng.dirichlet(np.ones(V), size=V)), device=DEV)
    root = torch.zeros(B, dtype=torch.int32, device=DEV)
    row0 = torch.tensor(_logits(q), device=DEV).expand(B, V).contiguous()
    first = np.zeros(V, np.int64)
    second = np.zeros((V, V), np.int64)
    st = eg.BuildState(B, V, D, k, m, 1.0, device=DEV)
    for c in range(calls):
        cu = datagen.child_uniforms(B, 1 + k, k, 300 + c, DEV)
        ft, _ = eg.build_begin(st, row0, cu[:, :1].contiguous())
        rows = q2[ft.long()].contiguous()  # [B, k, V]: the draft row of each frontier slot
        assert eg.build_expand(st, 1, rows, cu[:, 1:].contiguous()) is None
        t = eg.build_finalize(st, root)
        draft = torch.cat([row0.unsqueeze(1), rows], 1).contiguous()
        tok, dep = t["tokens"].long(), t["depths"]
        tgt = torch.where((dep == 1).unsqueeze(-1), p2_t[tok], p3_t[tok])
        tgt[:, 0] = torch.tensor(_logits(p), device=DEV)
        u = datagen.uniforms(B, m + 1, 400 + c, DEV)
        o = eg.tree_verify(tgt.contiguous(), draft, t, u, 1.0, depth=D, topk=k)
        ot, ol = np_(o["out_tokens"]), np_(o["out_len"])
        first += np.bincount(ot[:, 0], minlength=V)
        acc = ol >= 2
        np.add.at(second, (ot[acc, 0], ot[acc, 1]), 1)
    pe = softmax(_logits(p).astype(np.float64))
    assert chisquare(first, pe * first.sum()).pvalue > 1e-3
    for t1 in np.argsort(-second.sum(1))[:3]:
        pe2 = softmax(_logits(p2[t1]).astype(np.float64))
        assert chisquare(second[t1], pe2 * second[t1].sum()).pvalue > 1e-3
