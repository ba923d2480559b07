"""Pins of the oracle's static tree / chain build: a hand-worked example, the chain as a greedy
argmax sequence, and invariants over random templates (each sibling group is the top of its
parent's row in descending order; each node's log V step is the library log-softmax of its
parent's row at its token; masks are the ancestor closure)."""
import json
import os

import numpy as np
from scipy.special import log_softmax

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "static_tree_worked_example.json")


def static_matches_golden(orc) -> bool:
    g = json.load(open(GOLDEN))
    x = np.array([g["draft_rows"]], np.float32)
    o = orc.build_static_tree(x, np.array([g["root_token"]], np.int32), g["template_parents"], g["tree_temp"])
    e = g["expect"]
    return bool(all(list(o[k][0]) == e[k] for k in ("tokens", "parents", "depths", "node_row"))
                and list(o["mask"][0, :, 0]) == e["mask"]
                and np.allclose(o["node_logv"][0], e["node_logv"], atol=1e-6))


def test_worked_example():
    assert static_matches_golden(oracle)


def test_chain_is_the_greedy_argmax_sequence():
    rng = np.random.default_rng(0)
    for D in (1, 3, 8):
        x = rng.normal(0, 2, (3, D, 50)).astype(np.float32)
        x[:, :, 7] = x[:, :, 9] = x.max() + 1  # a tie: the lower id wins
        o = oracle.build_static_tree(x, np.arange(3, dtype=np.int32), [-1] + list(range(D)))
        for b in range(3):
            assert list(o["tokens"][b, 1:]) == [7] * D
            assert list(o["depths"][b]) == list(range(D + 1))
            assert list(o["node_row"][b]) == list(range(D)) + [-1]
        x = rng.normal(0, 2, (2, D, 50)).astype(np.float32)
        o = oracle.build_static_tree(x, np.zeros(2, np.int32), [-1] + list(range(D)))
        for b in range(2):
            assert list(o["tokens"][b, 1:]) == [int(np.argmax(x[b, d])) for d in range(D)]


def random_template(rng, n, max_kids=16):
    par = [-1]
    kids = [0]
    for i in range(1, n):
        choices = [p for p in range(i) if kids[p] < max_kids]
        p = int(rng.choice(choices))
        par.append(p)
        kids[p] += 1
        kids.append(0)
    return par


def static_invariants_hold(orc, seeds=range(6)) -> bool:
    for seed in seeds:
        rng = np.random.default_rng(seed)
        n = int(rng.integers(2, 40))
        tmpl = random_template(rng, n)
        internal = sorted(set(tmpl[1:]))
        B, V, T = 2, 64, float(rng.choice([0.7, 1.0, 1.5]))
        x = rng.normal(0, 2, (B, len(internal), V)).astype(np.float32)
        o = orc.build_static_tree(x, np.arange(B, dtype=np.int32), tmpl, T)
        for b in range(B):
            for p in internal:
                kids = [i for i in range(1, n) if tmpl[i] == p]
                row = x[b, internal.index(p)]
                order = sorted(range(V), key=lambda t: (-float(row[t]), t))
                if [int(o["tokens"][b, i]) for i in kids] != order[:len(kids)]:
                    return False
                ls = log_softmax(row.astype(np.float64) / T)
                for i in kids:
                    if abs(o["node_logv"][b, i] - o["node_logv"][b, p] - ls[o["tokens"][b, i]]) > 1e-9:
                        return False
            for i in range(n):
                anc, j = 0, i
                while j >= 0:
                    anc |= 1 << j
                    j = tmpl[j]
                if int(o["mask"][b, i, 0]) != anc or int(o["node_row"][b, i]) != (internal.index(i) if i in internal else -1):
                    return False
    return True


def test_random_templates_invariants():
    assert static_invariants_hold(oracle)
