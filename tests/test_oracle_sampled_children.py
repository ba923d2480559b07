"""Pins of the oracle's sampled-children build (EAGLE-1 notes appendix A.1, non-greedy: a node's
k children are sampled from the draft distribution).

- a hand-worked example (tests/golden/sampled_children_worked_example.json) for the dynamic
  build, with a repeated draw and the depth-1 frontier, and for a static chain at T = 0.5;
- every draw equals numpy's searchsorted of the uniform in the cumulative library softmax;
- a grid of uniforms reproduces the library softmax as draw frequencies (within one draw);
- near one-hot rows make the sampled chain the greedy argmax chain;
- losslessness of build -> verify: with sampled children the first committed token follows the
  target distribution (chi-square), for a static tree and for a dynamic tree whose draft rows
  are chosen by the depth-1 frontier the build reports (the interleaving a real draft model
  does); with top-k children the same test fails (the test has power);
- the frontier outputs agree with the tree (tokens of the expanded nodes, parent slots);
- children drawn at the verify temperature stay lossless at T = 0.7, and drawing them at another
  temperature fails the same test.
"""
import json
import os

import numpy as np
from scipy.special import log_softmax, softmax
from scipy.stats import chisquare

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "sampled_children_worked_example.json")


def _ln_rows(rows):
    return np.log(np.array(rows, np.float64)).astype(np.float32)


def sampled_matches_golden(orc) -> bool:
    g = json.load(open(GOLDEN))
    d = g["dynamic"]
    x = _ln_rows(d["draft_rows_ln"])[None]
    u = np.array(d["child_u"], np.float32)[None]
    o = orc.build_tree(x, [d["root_token"]], d["depth"], d["topk"], d["keep"], d["tree_temp"], child_u=u,
                       frontier=True)
    e = d["expect"]
    ok = all(o[k][0].tolist() == e[k] for k in ("tokens", "parents", "depths", "node_row", "front_tok",
                                                 "front_par"))
    ok = ok and o["mask"][0, :, 0].tolist() == e["mask"]
    ok = ok and np.allclose(o["node_logv"][0], e["node_logv"], atol=1e-6)
    s = g["static_chain"]
    o = orc.build_static_tree(_ln_rows(s["draft_rows_ln"])[None], [s["root_token"]], s["template_parents"],
                              s["tree_temp"], child_u=np.array(s["child_u"], np.float32)[None])
    e = s["expect"]
    ok = ok and all(o[k][0].tolist() == e[k] for k in ("tokens", "parents", "depths", "node_row"))
    ok = ok and o["mask"][0, :, 0].tolist() == e["mask"]
    return bool(ok and np.allclose(o["node_logv"][0], e["node_logv"], atol=1e-6))


def test_worked_example():
    assert sampled_matches_golden(oracle)


def test_draws_are_library_inverse_cdf():
    rng = np.random.default_rng(5)
    B, V, k = 64, 16, 4
    for T in (1.0, 0.7):
        x = rng.normal(0, 2, (B, 1, V)).astype(np.float32)
        u = rng.random((B, 1, k), dtype=np.float32)
        o = oracle.build_tree(x, np.zeros(B, np.int32), 1, k, k, T, child_u=u)
        for b in range(B):
            cdf = np.cumsum(softmax(x[b, 0].astype(np.float64) / T))
            want = np.minimum(np.searchsorted(cdf, u[b, 0].astype(np.float64), side="right"), V - 1)
            # depth-1 nodes keep creation (= draw) order; all k are kept
            assert o["tokens"][b, 1:].tolist() == want.tolist()
            lv = log_softmax(x[b, 0].astype(np.float64) / T)[want]
            assert np.allclose(o["node_logv"][b, 1:], lv, rtol=1e-12, atol=1e-12)


def test_grid_of_uniforms_reproduces_softmax():
    """N uniforms on the grid (i + 1/2)/N: draw t must come up N q_t times, within one."""
    rng = np.random.default_rng(11)
    V, N = 16, 4096
    x = rng.normal(0, 1.5, V).astype(np.float32)
    q = softmax(x.astype(np.float64))
    grid = ((np.arange(N) + 0.5) / N).astype(np.float32)
    xb = np.broadcast_to(x, (N, 1, V)).copy()
    o = oracle.build_tree(xb, np.zeros(N, np.int32), 1, 1, 1, 1.0, child_u=grid.reshape(N, 1, 1))
    counts = np.bincount(o["tokens"][:, 1], minlength=V)
    assert np.all(np.abs(counts - N * q) <= 1.0 + 1e-9)


def test_peaked_rows_sample_the_greedy_chain():
    rng = np.random.default_rng(2)
    D, V, B = 5, 40, 8
    x = rng.normal(0, 1, (B, D, V)).astype(np.float32)
    top = rng.integers(0, V, (B, D))
    for b in range(B):
        for d in range(D):
            x[b, d, top[b, d]] = 60.0  # every other token has q < e^-55
    u = rng.random((B, D, 1), dtype=np.float32)
    tmpl = [-1] + list(range(D))
    s = oracle.build_static_tree(x, np.zeros(B, np.int32), tmpl, child_u=u)
    g = oracle.build_static_tree(x, np.zeros(B, np.int32), tmpl)
    for key in ("tokens", "parents", "depths", "node_row"):
        assert np.array_equal(s[key], g[key])
    assert np.allclose(s["node_logv"], g["node_logv"], rtol=0, atol=1e-12)
    assert s["tokens"][:, 1:].tolist() == top.tolist()


def _dists(rng, V):
    p = rng.dirichlet(np.ones(V))
    q = rng.dirichlet(np.full(V, 0.5))
    return p, q


def _logits(p):
    return np.log(np.maximum(p, 1e-30)).astype(np.float32)


def static_root_trial_pvalue(orc, sampled=True, trials=200_000, seed=21):
    """Root with k = 3 children from the static build (template [-1, 0, 0, 0]), verified at T = 1:
    the first committed token against the target distribution."""
    V, k = 16, 3
    rng = np.random.default_rng(seed)
    p, q = _dists(rng, V)
    p2 = rng.dirichlet(np.ones(V), size=V)
    B = trials
    dft = np.broadcast_to(_logits(q), (B, 1, V)).copy()
    u_child = rng.random((B, 1, k), dtype=np.float32)
    t = orc.build_static_tree(dft, np.zeros(B, np.int32), [-1, 0, 0, 0], child_u=u_child if sampled else None)
    tgt = np.empty((B, k + 1, V), np.float32)
    tgt[:, 0] = _logits(p)
    tgt[:, 1:] = _logits(p2)[t["tokens"][:, 1:]]
    u = rng.random((B, k + 1), dtype=np.float32)
    o = orc.tree_verify(tgt, dft, t["tokens"], t["parents"], t["node_row"], u, 1.0, 2)
    pe = softmax(_logits(p).astype(np.float64))
    obs = np.bincount(o["out_tokens"][:, 0], minlength=V)
    return chisquare(obs, pe * obs.sum()).pvalue


def test_static_sampled_children_are_lossless():
    assert static_root_trial_pvalue(oracle) > 1e-3


def test_topk_children_are_not_lossless():
    assert static_root_trial_pvalue(oracle, sampled=False) < 1e-6


def test_dynamic_sampled_tree_is_lossless_with_interleaved_draft_rows():
    """D = 2, k = 2, every candidate kept (m = k + k^2).  The draft and target rows below a depth-1
    node depend only on its token, as a real model's would; the build is first run with
    placeholder rows 1..k to learn the depth-1 frontier (it depends on row 0 only), then with
    each slot's row q2[token].  First token ~ p; second token, given the first was an accepted
    draft token t, ~ p2[t]."""
    V, k, D = 12, 2, 2
    m = k + k * k
    rng = np.random.default_rng(8)
    p, q = _dists(rng, V)
    p2 = rng.dirichlet(np.ones(V), size=V)
    q2 = rng.dirichlet(np.full(V, 0.5), size=V)
    p3 = rng.dirichlet(np.ones(V), size=V)
    B = 200_000
    R = 1 + (D - 1) * k
    x = np.zeros((B, R, V), np.float32)
    x[:, 0] = _logits(q)
    cu = rng.random((B, R, k), dtype=np.float32)
    first = oracle.build_tree(x, np.zeros(B, np.int32), D, k, m, child_u=cu, frontier=True)
    ft = first["front_tok"][:, 0]  # [B, k]
    x[:, 1:] = _logits(q2)[ft]
    t = oracle.build_tree(x, np.zeros(B, np.int32), D, k, m, child_u=cu, frontier=True)
    assert np.array_equal(t["front_tok"], first["front_tok"])  # row 0 alone decides depth 1
    tok, par, dep = t["tokens"], t["parents"], t["depths"]
    n = m + 1
    tgt = np.empty((B, n, V), np.float32)
    tgt[:, 0] = _logits(p)
    d1 = dep == 1
    tgt[d1] = _logits(p2)[tok[d1]]
    d2 = dep == 2
    tgt[d2] = _logits(p3)[tok[d2]]
    u = rng.random((B, n), dtype=np.float32)
    o = oracle.tree_verify(tgt, x, tok, par, t["node_row"], u, 1.0, D + 1)
    pe = softmax(_logits(p).astype(np.float64))
    obs = np.bincount(o["out_tokens"][:, 0], minlength=V)
    assert chisquare(obs, pe * obs.sum()).pvalue > 1e-3
    acc = o["out_len"] >= 2
    t1 = o["out_tokens"][:, 0]
    checked = 0
    for tok1 in np.argsort(-np.bincount(t1[acc], minlength=V))[:3]:
        sel = acc & (t1 == tok1)
        obs2 = np.bincount(o["out_tokens"][sel, 1], minlength=V)
        pe2 = softmax(_logits(p2[tok1]).astype(np.float64))
        assert chisquare(obs2, pe2 * obs2.sum()).pvalue > 1e-3
        checked += int(sel.sum())
    assert checked > 20_000


def frontier_consistent(orc, seeds=range(4)) -> bool:
    for seed in seeds:
        rng = np.random.default_rng(100 + seed)
        D, k, V, B = 4, 3, 30, 6
        m = k + (D - 1) * k * k  # keep everything: every frontier node is in the tree
        R = 1 + (D - 1) * k
        x = rng.normal(0, 2, (B, R, V)).astype(np.float32)
        for cu in (None, rng.random((B, R, k), dtype=np.float32)):
            o = orc.build_tree(x, np.zeros(B, np.int32), D, k, m, child_u=cu, frontier=True)
            for b in range(B):
                row_node = {int(o["node_row"][b, i]): i for i in range(1, m + 1) if o["node_row"][b, i] >= 0}
                for f in range(1, D):
                    for s in range(k):
                        i = row_node.get(1 + (f - 1) * k + s)
                        if i is None or o["depths"][b, i] != f or o["tokens"][b, i] != o["front_tok"][b, f - 1, s]:
                            return False
                        ps = o["front_par"][b, f - 1, s]
                        if f == 1:
                            if ps != -1 or o["parents"][b, i] != 0:
                                return False
                        elif o["parents"][b, i] != row_node.get(1 + (f - 2) * k + int(ps), -1):
                            return False
    return True


def test_frontier_outputs_match_the_tree():
    assert frontier_consistent(oracle)


def test_row_children_are_the_builds_children():
    """The per-row entry point gives the same children as a depth-1 build that keeps them all
    (sampled: in draw order; greedy: the top k in rank order)."""
    rng = np.random.default_rng(13)
    N, V, k = 12, 300, 5
    x = rng.normal(0, 2, (N, V)).astype(np.float32)
    u = rng.random((N, k), dtype=np.float32)
    for cu, T in ((u, 1.0), (u, 0.6), (None, 1.0)):
        rc = oracle.row_children(x, k, T, child_u=cu)
        b = oracle.build_tree(x[:, None], np.zeros(N, np.int32), 1, k, k, T,
                              child_u=None if cu is None else cu[:, None])
        if cu is None:  # the build flattens by creation order = rank order
            assert np.array_equal(rc["tok"], b["tokens"][:, 1:])
        else:
            assert np.array_equal(rc["tok"], b["tokens"][:, 1:])
            assert np.array_equal(rc["gap"].min(1), b["draw_gap"])
        assert np.allclose(rc["lc"], b["node_logv"][:, 1:], rtol=0, atol=0)


def _temperature_trial_pvalue(tree_temp, verify_temp, trials=200_000, seed=33):
    """Static root tree (k = 3) built at tree_temp, verified at verify_temp: the first committed
    token against the target distribution at verify_temp."""
    V, k = 16, 3
    rng = np.random.default_rng(seed)
    p, q = _dists(rng, V)
    p2 = rng.dirichlet(np.ones(V), size=V)
    B = trials
    dft = np.broadcast_to(_logits(q), (B, 1, V)).copy()
    t = oracle.build_static_tree(dft, np.zeros(B, np.int32), [-1, 0, 0, 0], tree_temp,
                                 child_u=rng.random((B, 1, k), dtype=np.float32))
    tgt = np.empty((B, k + 1, V), np.float32)
    tgt[:, 0] = _logits(p)
    tgt[:, 1:] = _logits(p2)[t["tokens"][:, 1:]]
    o = oracle.tree_verify(tgt, dft, t["tokens"], t["parents"], t["node_row"],
                           rng.random((B, k + 1), dtype=np.float32), verify_temp, 2)
    pe = softmax(_logits(p).astype(np.float64) / verify_temp)
    obs = np.bincount(o["out_tokens"][:, 0], minlength=V)
    return chisquare(obs, pe * obs.sum()).pvalue


def test_sampled_children_at_the_verify_temperature_are_lossless():
    """Children drawn at the temperature the verification uses for q: the committed token follows
    the target at that temperature ([hubwiz] section 2: both distributions are tempered)."""
    assert _temperature_trial_pvalue(0.7, 0.7) > 1e-3


def test_children_drawn_at_another_temperature_are_not():
    """The control: children drawn from q at T = 2 but tested as if drawn at T = 0.7."""
    assert _temperature_trial_pvalue(2.0, 0.7) < 1e-6
