"""Pins of the oracle's KV commit: a hand-worked example, invariants over real oracle rounds, and
the refused cases.  The commit is a definition (copies in a fixed order), so these pins fix the
order, the positions and the new length."""
import json
import os

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "kv_commit_worked_example.json")


def _golden_case():
    g = json.load(open(GOLDEN))
    L, B, n, H, d, S = g["L"], g["B"], g["n"], g["Hkv"], g["d"], g["S_max"]
    kt = np.zeros((L, B, n, H, d), np.float32)
    for b in range(B):
        for i in range(n):
            kt[:, b, i, 0] = [10 * b + i, -(10 * b + i)]
    vt = kt + 100
    kc = np.full((L, B, S, H, d), -1, np.float32)
    vc = kc.copy()
    return g, kt, vt, kc, vc


def commit_matches_golden(orc) -> bool:
    g, kt, vt, kc, vc = _golden_case()
    k2, v2, nc, ok = orc.kv_commit(kt, vt, np.array(g["out_path"], np.int32), np.array(g["out_len"], np.int32),
                                   np.array(g["ctx_len"], np.int32), kc, vc)
    exp_k = np.array(g["expect"]["k_rows"], np.float32)
    exp_v = np.where(exp_k == -1, -1, exp_k + 100)
    return bool(ok and list(nc) == g["expect"]["new_ctx_len"] and np.array_equal(k2[0, :, :, 0], exp_k)
                and np.array_equal(v2[0, :, :, 0], exp_v))


def test_worked_example():
    assert commit_matches_golden(oracle)


def _round(seed, B=3, V=200, D=4, k=3, m=9, L=2, H=2, d=8, S=40):
    rng = np.random.default_rng(seed)
    R = 1 + (D - 1) * k
    draft = rng.normal(0, 2, (B, R, V)).astype(np.float32)
    tree = oracle.build_tree(draft, rng.integers(0, V, B).astype(np.int32), D, k, m)
    n = m + 1
    target = (draft[np.arange(B)[:, None], np.maximum(tree["node_row"], 0)] +
              rng.normal(0, 0.3, (B, n, V))).astype(np.float32)
    ver = oracle.tree_verify(target, draft, tree["tokens"], tree["parents"], tree["node_row"],
                             rng.random((B, n)).astype(np.float32), 1.0, D + 1)
    kt = rng.standard_normal((L, B, n, H, d)).astype(np.float32)
    vt = rng.standard_normal((L, B, n, H, d)).astype(np.float32)
    kc = rng.standard_normal((L, B, S, H, d)).astype(np.float32)
    vc = rng.standard_normal((L, B, S, H, d)).astype(np.float32)
    ctx = rng.integers(0, S - D - 1, B).astype(np.int32)
    return tree, ver, kt, vt, kc, vc, ctx


def test_commit_of_real_rounds_follows_the_path():
    for seed in range(6):
        tree, ver, kt, vt, kc, vc, ctx = _round(seed)
        k2, v2, nc, ok = oracle.kv_commit(kt, vt, ver["out_path"], ver["out_len"], ctx, kc, vc)
        assert ok
        B = ctx.shape[0]
        for b in range(B):
            ln = int(ver["out_len"][b])
            assert nc[b] == ctx[b] + ln
            nodes = [0] + [int(x) for x in ver["out_path"][b][:ln - 1]]
            # the path is a chain from the root, in depth order, so position ctx + i holds depth i
            assert [int(tree["depths"][b][x]) for x in nodes] == list(range(ln))
            for i, node in enumerate(nodes):
                assert np.array_equal(k2[:, b, ctx[b] + i], kt[:, b, node])
                assert np.array_equal(v2[:, b, ctx[b] + i], vt[:, b, node])
            untouched = [s for s in range(kc.shape[2]) if not ctx[b] <= s < ctx[b] + ln]
            assert np.array_equal(k2[:, b, untouched], kc[:, b, untouched])
            assert np.array_equal(v2[:, b, untouched], vc[:, b, untouched])


def test_bf16_bytes_copied_unchanged():
    tree, ver, kt, vt, kc, vc, ctx = _round(11)
    as16 = lambda a: (a.view(np.uint32) >> 16).astype(np.uint16)  # noqa: E731
    k2, v2, nc, ok = oracle.kv_commit(as16(kt), as16(vt), ver["out_path"], ver["out_len"], ctx, as16(kc), as16(vc))
    k3, v3, nc3, ok3 = oracle.kv_commit(kt, vt, ver["out_path"], ver["out_len"], ctx, kc, vc)
    assert ok and ok3 and np.array_equal(nc, nc3)
    assert np.array_equal(k2, as16(k3)) and np.array_equal(v2, as16(v3))


def test_refused_commits_leave_the_sequence_unchanged():
    g, kt, vt, kc, vc = _golden_case()
    path = np.array(g["out_path"], np.int32)
    ctx = np.array(g["ctx_len"], np.int32)
    # (committed counts, path, the refused sequence)
    cases = [
        (np.array([3, 5], np.int32), path, 1),                                             # 5 > D + 1
        (np.array([3, 1], np.int32), np.array([[3, 5, -1], [-1, -1, -1]], np.int32), 0),  # node 5 >= n
        (np.array([3, 1], np.int32), np.array([[0, 4, -1], [-1, -1, -1]], np.int32), 0),  # the root in the path
        (np.array([3, 3], np.int32), np.array([[3, 4, -1], [1, 2, -1]], np.int32), 1),    # 6 + 3 > S_max
    ]
    for ln, p, bad in cases:
        k2, v2, nc, ok = oracle.kv_commit(kt, vt, p, ln, ctx, kc, vc)
        assert not ok
        assert nc[bad] == ctx[bad]
        assert np.array_equal(k2[:, bad], kc[:, bad]) and np.array_equal(v2[:, bad], vc[:, bad])
        good = 1 - bad
        assert nc[good] == ctx[good] + ln[good]
        assert not np.array_equal(k2[:, good], kc[:, good])


def test_nothing_committed_is_a_no_op():
    g, kt, vt, kc, vc = _golden_case()
    k2, v2, nc, ok = oracle.kv_commit(kt, vt, np.full((2, 3), -1, np.int32), np.zeros(2, np.int32),
                                      np.array(g["ctx_len"], np.int32), kc, vc)
    assert ok and list(nc) == g["ctx_len"]
    assert np.array_equal(k2, kc) and np.array_equal(v2, vc)
