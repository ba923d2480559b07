"""Pins for the oracle's EAGLE-2 draft-tree build (CPU only).

Each test checks the oracle against something other than itself: a hand-worked fixture, a
brute-force enumeration of token paths on tiny inputs, library softmax/sort, or an invariant the
pages state ([EAGLE-2 notes] "Expanding the Draft Tree", "Rerank draft tokens", "Tree Attention
Mask").
"""
import itertools
import json
import os

import numpy as np
import pytest
from scipy.special import softmax

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(rng, B, R, V, sigma=2.0, plant=6.0):
    x = rng.normal(0.0, sigma, (B, R, V)).astype(np.float32)
    idx = rng.integers(0, V, (B, R))
    np.add.at(x, (np.arange(B)[:, None], np.arange(R)[None, :], idx), np.float32(plant))
    return x


def test_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "build_worked_example.json")))
    x = np.log(np.array(g["probs"], np.float64)).astype(np.float32)[None]
    o = oracle.build_tree(x, [g["root_token"]], g["depth"], g["topk"], g["keep"])
    e = g["expect"]
    assert o["tokens"][0].tolist() == e["tokens"]
    assert o["parents"][0].tolist() == e["parents"]
    assert o["depths"][0].tolist() == e["depths"]
    assert o["node_row"][0].tolist() == e["node_row"]
    assert o["mask"][0, :, 0].tolist() == e["mask"]
    np.testing.assert_allclose(np.exp(o["node_logv"][0]), e["node_value"], rtol=1e-6)


def _ancestors(parents, i):
    out = []
    while i >= 0:
        out.append(i)
        i = parents[i]
    return out


@pytest.mark.parametrize("shape", [(3, 1000, 3, 4, 10), (2, 500, 8, 10, 60), (2, 300, 6, 10, 50),
                                   (2, 64, 4, 3, 20), (2, 50, 5, 1, 4), (2, 40, 1, 5, 3)])
def test_structure_invariants(shape):
    """Ancestor closure, V_child <= V_parent, V = product of softmax confidences along the path,
    depth = parent depth + 1, mask = ancestor-or-self set, children = top-k of the expanding row."""
    B, V, D, k, m = shape
    R = 1 + (D - 1) * k
    rng = np.random.default_rng(1234 + D * 7 + k)
    x = _rows(rng, B, R, V)
    root = rng.integers(0, V, B).astype(np.int32)
    o = oracle.build_tree(x, root, D, k, m)
    n = m + 1
    for b in range(B):
        tok, par, dep, row = o["tokens"][b], o["parents"][b], o["depths"][b], o["node_row"][b]
        lv, msk = o["node_logv"][b], o["mask"][b, :, 0]
        assert tok[0] == root[b] and par[0] == -1 and dep[0] == 0 and row[0] == 0 and lv[0] == 0
        probs = {r: softmax(x[b, r].astype(np.float64)) for r in range(R)}
        for i in range(1, n):
            p = par[i]
            assert 0 <= p < i, "parents precede children (ancestor-closed, flattened parents first)"
            assert dep[i] == dep[p] + 1 and 1 <= dep[i] <= D
            assert lv[i] <= lv[p]
            # V_i = product of confidences along root -> i (the page's definition, product form)
            prod = 1.0
            j = i
            while j > 0:
                prod *= probs[row[par[j]]][tok[j]]
                j = par[j]
            np.testing.assert_allclose(np.exp(lv[i]), prod, rtol=1e-10)
            want = 0
            for a in _ancestors(par, i):
                want |= 1 << int(a)
            assert int(msk[i]) == want
        # children of every node are among the top-k tokens of the row that expanded it, and a
        # node that has kept children was expanded
        for a in range(n):
            kids = [i for i in range(1, n) if par[i] == a]
            if not kids:
                continue
            assert row[a] >= 0
            order = np.lexsort((np.arange(V), -x[b, row[a]].astype(np.float64)))[:k]
            assert set(tok[kids].tolist()) <= set(order.tolist())
            # flattened order among siblings follows child rank (descending logit)
            ranks = [order.tolist().index(t) for t in tok[kids]]
            assert ranks == sorted(ranks)
        # mask words: n <= 64 here, so one word per node
        assert o["mask"].shape[2] == 1


def _brute_force_tree(x, D, k, m):
    """Independent restatement over token paths: enumerate every candidate path with its value
    computed as a product of softmax probabilities; expand the k best paths per depth; keep the m
    best paths overall (value desc, shallower first, then creation order)."""
    R = x.shape[0]
    probs = [softmax(x[r].astype(np.float64)) for r in range(R)]

    def topk(r):
        return sorted(range(x.shape[1]), key=lambda t: (-float(x[r][t]), t))[:k]

    # candidate = (path tuple, value, creation, row used to expand or None)
    cands = []
    level = []
    for t in topk(0):
        c = dict(path=(t,), v=probs[0][t], creation=len(cands))
        cands.append(c)
        level.append(c)
    for f in range(1, D):
        frontier = sorted(level, key=lambda c: (-c["v"], c["creation"]))[:k]
        level = []
        for s, par in enumerate(frontier):
            r = 1 + (f - 1) * k + s
            par["row"] = r
            for t in topk(r):
                c = dict(path=par["path"] + (t,), v=par["v"] * probs[r][t], creation=len(cands))
                cands.append(c)
                level.append(c)
    kept = sorted(cands, key=lambda c: (-c["v"], len(c["path"]), c["creation"]))[:m]
    return cands, kept


@pytest.mark.parametrize("seed", range(12))
def test_brute_force_tiny(seed):
    rng = np.random.default_rng(seed)
    D = int(rng.integers(1, 4))
    k = int(rng.integers(1, 4))
    V = int(rng.integers(max(k, 2), 9))
    P = k + (D - 1) * k * k
    m = int(rng.integers(1, P + 1))
    R = 1 + (D - 1) * k
    x = rng.normal(0, 2, (1, R, V)).astype(np.float32)
    o = oracle.build_tree(x, [0], D, k, m)
    cands, kept = _brute_force_tree(x[0], D, k, m)
    # paths of the oracle's nodes
    par, tok = o["parents"][0], o["tokens"][0]
    got = set()
    for i in range(1, m + 1):
        path = []
        j = i
        while j > 0:
            path.append(int(tok[j]))
            j = par[j]
        got.add(tuple(reversed(path)))
    want = {c["path"] for c in kept}
    if o["margin"][0] > 1e-9:
        assert got == want
    # flattened order = creation order of the kept paths
    want_order = [c["path"] for c in sorted(kept, key=lambda c: c["creation"])]
    got_order = []
    for i in range(1, m + 1):
        path = []
        j = i
        while j > 0:
            path.append(int(tok[j]))
            j = par[j]
        got_order.append(tuple(reversed(path)))
    if o["margin"][0] > 1e-9:
        assert got_order == want_order


def test_frontier_slot_uses_row_convention():
    """Frontier slot s at depth f is expanded with draft row 1 + (f-1)k + s: row r carries a
    planted token 100 + r far above the rest, so the best child of the node row r expanded must
    be token 100 + r."""
    D, k, V = 4, 3, 200
    R = 1 + (D - 1) * k
    rng = np.random.default_rng(7)
    x = rng.normal(0, 1, (1, R, V)).astype(np.float32)
    for r in range(R):
        x[0, r, 100 + r] = 30.0
    P = k + (D - 1) * k * k
    o = oracle.build_tree(x, [1], D, k, P)
    tok, par, row, lv, dep = (o[key][0] for key in ("tokens", "parents", "node_row", "node_logv", "depths"))
    for a in range(len(tok)):
        kids = [i for i in range(1, len(tok)) if par[i] == a]
        if not kids:
            continue
        assert tok[kids[0]] == 100 + row[a]
    for f in range(1, D):
        nodes = [i for i in range(len(tok)) if dep[i] == f]
        ranked = sorted(nodes, key=lambda i: -lv[i])[:k]
        for s, i in enumerate(ranked):
            assert row[i] == 1 + (f - 1) * k + s


def test_tie_breaks():
    """Equal logits: the lower token id is the better child.  Equal values across depths: the
    shallower node wins the last kept slot ([EAGLE-2 notes] Rerank)."""
    V = 8
    # root row: tokens 3 and 5 tie for first; both get value 0.4 ... (ties to lower id: 3 first)
    r0 = np.full(V, -50.0, np.float32)
    r0[[3, 5]] = 0.0
    r0[1] = -0.5
    # row 1 expands node 'token 3': one certain child (log-confidence exactly 0)
    r1 = np.full(V, -200.0, np.float32)
    r1[6] = 0.0
    r2 = np.full(V, -200.0, np.float32)
    r2[2] = 0.0
    r3 = np.zeros(V, np.float32)
    x = np.stack([r0, r1, r2, r3])[None]
    o = oracle.build_tree(x, [0], 2, 3, 3)
    tok, par, dep = o["tokens"][0], o["parents"][0], o["depths"][0]
    # children of root in rank order: 3, 5 (tie -> lower id), then 1
    assert tok[1:3].tolist() == [3, 5]
    # node 3 has value v(3) = v(5) = v(child 6 of 3) = v(child 2 of 5): the two depth-1 nodes win
    # the tie over their depth-2 children, so the third kept slot goes to the best remaining key:
    # the depth-2 child of token 3 (same value as its parent, created before the child of 5)
    assert dep[1:].tolist() == [1, 1, 2]
    assert tok[3] == 6 and par[3] == 1


def test_degenerate_shapes():
    rng = np.random.default_rng(3)
    # D = 1: only the root's top-k, keep m of them
    x = rng.normal(0, 2, (2, 1, 30)).astype(np.float32)
    o = oracle.build_tree(x, [0, 1], 1, 5, 3)
    for b in range(2):
        want = np.lexsort((np.arange(30), -x[b, 0].astype(np.float64)))[:3]
        assert o["tokens"][b, 1:].tolist() == want.tolist()
        assert (o["parents"][b, 1:] == 0).all()
    # k = 1: a chain of depth min(D, m)
    x = rng.normal(0, 2, (1, 5, 30)).astype(np.float32)
    o = oracle.build_tree(x, [0], 5, 1, 5)
    assert o["parents"][0].tolist() == [-1, 0, 1, 2, 3, 4]
    assert o["node_row"][0].tolist() == [0, 1, 2, 3, 4, -1]
    # m = P keeps the whole pool
    x = rng.normal(0, 2, (1, 1 + 2 * 3, 40)).astype(np.float32)
    o = oracle.build_tree(x, [0], 3, 3, 3 + 2 * 9)
    assert (o["depths"][0] == np.array([0] + [1] * 3 + [2] * 9 + [3] * 9)).all()


def test_bad_args():
    x = np.zeros((1, 3, 10), np.float32)
    with pytest.raises(oracle.OracleError):
        oracle.build_tree(x, [0], 2, 2, 100)  # m larger than the pool
