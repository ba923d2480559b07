"""Pins for the oracle's tree verification (CPU only).

* Hand-worked fixtures (tests/golden/verify_worked_examples.json).
* Losslessness ([EAGLE-1 notes] A3, citing Leviathan et al. appendix A.1; [EAGLE-3 blog]
  section 2): with children drawn i.i.d. from q, the committed token is distributed as the
  target p for any q.  Checked by a chi-square test over 1e6 seeded trials, vocab 16.
* Greedy ([EAGLE-1 notes] results at T = 0; [EAGLE-3 blog] section 3, keep the longest agreeing
  prefix): brute force over the tree's paths.
* Counting ([EAGLE-3 blog] section 1): at least one token per round, at most accepted + 1.
"""
import json
import os
import zlib

import numpy as np
import pytest
from scipy.special import softmax
from scipy.stats import chisquare

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _logits(p):
    return np.log(np.asarray(p, np.float64)).astype(np.float32)


@pytest.mark.parametrize("case", json.load(open(os.path.join(GOLDEN, "verify_worked_examples.json")))["cases"],
                         ids=lambda c: c["name"])
def test_worked_examples(case):
    tgt = _logits(case["target_probs"])[None]
    dft = _logits(case["draft_probs"])[None]
    o = oracle.tree_verify(tgt, dft, [case["tokens"]], [case["parents"]], [case["node_row"]],
                           [case["uniforms"]], case["temperature"], case["max_commit"])
    e = case["expect"]
    assert o["out_tokens"][0].tolist() == e["out_tokens"]
    assert int(o["out_len"][0]) == e["out_len"]
    assert o["out_path"][0].tolist() == e["out_path"]
    for got, want in zip(o["out_ratio"][0], e["ratio"]):
        if want is None:
            assert np.isnan(got)
        else:
            np.testing.assert_allclose(got, want, rtol=1e-6, atol=1e-7)


def _dists(kind, rng, V):
    if kind == "dirichlet":
        return rng.dirichlet(np.ones(V)), rng.dirichlet(np.ones(V))
    if kind == "peaked":
        p = rng.dirichlet(np.full(V, 0.3))
        q = rng.dirichlet(np.full(V, 0.3))
        return p, q
    if kind == "mismatch":  # q puts its mass where p has little
        p = np.linspace(1.0, 0.01, V)
        q = p[::-1].copy()
        return p / p.sum(), q / q.sum()
    raise ValueError(kind)


def _iid_trials(rng, p, q, p2, k, trials, chunk=200_000, orc=oracle):
    """Root with k children drawn i.i.d. from q (duplicates allowed, EAGLE-1 appendix A.1 non-greedy
    drafting); every child is a leaf whose target row is p2[token].  Returns first and second
    committed tokens (second = -1 when the walk stopped at the root) and the accepted node."""
    V = len(p)
    n = k + 1
    firsts, seconds, accepted = [], [], []
    tgt_root = _logits(p)
    dft_root = _logits(q)
    p2_logits = _logits(p2)
    done = 0
    while done < trials:
        B = min(chunk, trials - done)
        kids = rng.choice(V, size=(B, k), p=q).astype(np.int32)
        tokens = np.concatenate([np.zeros((B, 1), np.int32), kids], 1)
        parents = np.tile(np.array([-1] + [0] * k, np.int32), (B, 1))
        node_row = np.tile(np.array([0] + [-1] * k, np.int32), (B, 1))
        tgt = np.empty((B, n, V), np.float32)
        tgt[:, 0] = tgt_root
        tgt[:, 1:] = p2_logits[kids]
        dft = np.broadcast_to(dft_root, (B, 1, V)).copy()
        u = rng.random((B, n), dtype=np.float32)
        o = orc.tree_verify(tgt, dft, tokens, parents, node_row, u, 1.0, 3)
        firsts.append(o["out_tokens"][:, 0])
        seconds.append(np.where(o["out_len"] == 2, o["out_tokens"][:, 1], -1))
        accepted.append(o["out_path"][:, 0])
        done += B
    return np.concatenate(firsts), np.concatenate(seconds), np.concatenate(accepted)


CHI_CASES = [(kind, k) for kind in ("dirichlet", "peaked", "mismatch") for k in (1, 2, 4)]


@pytest.mark.parametrize("kind,k", CHI_CASES)
def test_lossless_chi_square(kind, k):
    V, trials = 16, 1_000_000
    rng = np.random.default_rng(zlib.crc32(f"{kind}/{k}".encode()))
    p, q = _dists(kind, rng, V)
    p2 = rng.dirichlet(np.ones(V), size=V)  # target after each possible first token
    # what the oracle sees are float32 logits: compare against the distribution they encode
    p_eff = softmax(_logits(p).astype(np.float64))
    p2_eff = softmax(_logits(p2).astype(np.float64), axis=1)
    first, second, acc = _iid_trials(rng, p, q, p2, k, trials)
    obs = np.bincount(first, minlength=V)
    keep = p_eff * trials >= 5
    exp = p_eff * trials
    stat = chisquare(obs[keep], exp[keep] * obs[keep].sum() / exp[keep].sum())
    assert stat.pvalue > 0.01, (kind, k, stat)
    # second token, given that the first was an accepted draft token t1: distributed as p2[t1]
    pvals = []
    for t1 in np.argsort(-np.bincount(first[acc >= 0], minlength=V))[:3]:
        sel = (acc >= 0) & (first == t1)
        cnt = int(sel.sum())
        if cnt < 2000:
            continue
        o2 = np.bincount(second[sel], minlength=V)
        e2 = p2_eff[t1] * cnt
        kk = e2 >= 5
        pvals.append(chisquare(o2[kk], e2[kk] * o2[kk].sum() / e2[kk].sum()).pvalue)
    assert pvals and min(pvals) > 0.01 / len(pvals), pvals


def _random_tree_case(rng, B, V, n, D, distinct=False):
    """Random tree shapes; with ``distinct`` siblings hold different tokens (as top-k children do)."""
    parents = np.zeros((B, n), np.int32)
    depth = np.zeros((B, n), np.int32)
    tokens = rng.integers(0, V, (B, n)).astype(np.int32)
    parents[:, 0] = -1
    for b in range(B):
        for i in range(1, n):
            cand = [j for j in range(i) if depth[b, j] < D]
            parents[b, i] = cand[int(rng.integers(0, len(cand)))]
            depth[b, i] = depth[b, parents[b, i]] + 1
    if distinct:
        for b in range(B):
            for a in range(n):
                kids = [i for i in range(1, n) if parents[b, i] == a]
                if kids:
                    tokens[b, kids] = rng.choice(V, size=len(kids), replace=False)
    has_kids = np.zeros((B, n), bool)
    for b in range(B):
        for i in range(1, n):
            has_kids[b, parents[b, i]] = True
    R = n
    node_row = np.where(has_kids, np.arange(n)[None, :], -1).astype(np.int32)
    node_row[:, 0] = 0
    return tokens, parents, node_row, R


@pytest.mark.parametrize("seed", range(8))
def test_greedy_is_longest_agreeing_prefix(seed):
    """At T = 0 the committed tokens are the longest tree path whose every token is the target's
    argmax at its parent, followed by the argmax at the stop node (brute force over all paths)."""
    rng = np.random.default_rng(seed)
    B, V, n, D = 16, 10, 9, 4
    tokens, parents, node_row, R = _random_tree_case(rng, B, V, n, D, distinct=True)
    tgt = rng.normal(0, 1, (B, n, V)).astype(np.float32)
    # make agreement likely: node i's token is often the argmax of its parent's row
    for b in range(B):
        for i in range(1, n):
            if rng.random() < 0.7:
                tgt[b, parents[b, i], tokens[b, i]] = 10.0 + rng.random()
    dft = rng.normal(0, 1, (B, R, V)).astype(np.float32)
    u = rng.random((B, n), dtype=np.float32)
    o = oracle.tree_verify(tgt, dft, tokens, parents, node_row, u, 0.0, D + 1)
    for b in range(B):
        best = None
        # every node defines a path; count how many leading tokens agree with the argmax
        for i in range(n):
            path = []
            j = i
            while j > 0:
                path.append(j)
                j = parents[b, j]
            path = path[::-1]
            agree = []
            for node in path:
                if tokens[b, node] == int(np.argmax(tgt[b, parents[b, node]])):
                    agree.append(node)
                else:
                    break
            if len(agree) == len(path) and (best is None or len(path) > len(best)):
                best = path
        stop = best[-1] if best else 0
        want = [int(tokens[b, j]) for j in best] + [int(np.argmax(tgt[b, stop]))]
        L = int(o["out_len"][b])
        assert o["out_tokens"][b, :L].tolist() == want
        assert o["out_path"][b, :L - 1].tolist() == best


@pytest.mark.parametrize("T", [1.0, 0.7, 0.0])
def test_counts_and_path_shape(T):
    rng = np.random.default_rng(int(T * 10))
    B, V, n, D = 64, 12, 10, 4
    tokens, parents, node_row, R = _random_tree_case(rng, B, V, n, D)
    tgt = rng.normal(0, 2, (B, n, V)).astype(np.float32)
    dft = rng.normal(0, 2, (B, R, V)).astype(np.float32)
    u = rng.random((B, n), dtype=np.float32)
    o = oracle.tree_verify(tgt, dft, tokens, parents, node_row, u, T, D + 1)
    for b in range(B):
        L = int(o["out_len"][b])
        assert 1 <= L <= D + 1
        path = o["out_path"][b, :L - 1].tolist()
        prev = 0
        for j, node in enumerate(path):
            assert parents[b, node] == prev
            assert o["out_tokens"][b, j] == tokens[b, node]
            prev = node
        assert (o["out_tokens"][b, L:] == -1).all()
        assert 0 <= o["out_tokens"][b, L - 1] < V


def test_first_child_ratio_is_p_over_q():
    """The first child of a node is tested with p(t)/q(t) of the temperature-scaled softmaxes."""
    rng = np.random.default_rng(4)
    B, V, n, D = 8, 20, 8, 3
    tokens, parents, node_row, R = _random_tree_case(rng, B, V, n, D)
    tgt = rng.normal(0, 2, (B, n, V)).astype(np.float32)
    dft = rng.normal(0, 2, (B, R, V)).astype(np.float32)
    u = rng.random((B, n), dtype=np.float32)
    for T in (1.0, 0.5):
        o = oracle.tree_verify(tgt, dft, tokens, parents, node_row, u, T, D + 1)
        for b in range(B):
            seen = set()
            for i in range(1, n):
                a = parents[b, i]
                if a in seen:
                    continue
                seen.add(a)
                p = softmax(tgt[b, a].astype(np.float64) / T)
                q = softmax(dft[b, node_row[b, a]].astype(np.float64) / T)
                np.testing.assert_allclose(o["out_ratio"][b, i], p[tokens[b, i]] / q[tokens[b, i]], rtol=1e-12)


def test_two_token_closed_form():
    """V = 2, one child: P(commit token t) must equal p(t) exactly in expectation.  With the child's
    token a and u below/above the ratio, the two branches are checked against the closed form:
    accept iff u < p(a)/q(a); the residual then puts all mass on the other token."""
    p = np.array([0.3, 0.7])
    q = np.array([0.6, 0.4])
    tgt = _logits([p, [0.5, 0.5]])[None]
    dft = _logits([q])[None]
    ratio = p[0] / q[0]  # child token 0: 0.5
    for u1, want in ((ratio - 1e-3, 0), (ratio + 1e-3, 1)):
        o = oracle.tree_verify(tgt, dft, [[1, 0]], [[-1, 0]], [[0, -1]], [[0.99, u1]], 1.0, 2)
        assert int(o["out_tokens"][0, 0]) == want
