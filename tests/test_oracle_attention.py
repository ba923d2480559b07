"""Pins for the oracle's tree attention (CPU only).

The pages fix two facts ([EAGLE-3 blog] section 5; [EAGLE-2 notes] "Tree Attention Mask"):
a token sees only its ancestors and the context, never a sibling branch, so one pass scores every
root-to-leaf path as if it ran alone; and a chain-shaped draft is plain causal drafting
([EAGLE-1 notes] ablation, appendix A.1).  Both are checked against torch's
``scaled_dot_product_attention`` in float64 (a library routine, not the oracle's loop).
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle


def _mask_from_parents(parents):
    n = len(parents)
    m = np.zeros((n, 1), np.uint64)
    for i in range(n):
        j = i
        w = 0
        while j >= 0:
            w |= 1 << j
            j = parents[j]
        m[i, 0] = w
    return m


def _inputs(rng, L, B, n, Hq, Hkv, d, S, ctx):
    q = rng.normal(0, 1, (L, B, n, Hq, d)).astype(np.float32)
    kc = rng.normal(0, 1, (L, B, S, Hkv, d)).astype(np.float32)
    vc = rng.normal(0, 1, (L, B, S, Hkv, d)).astype(np.float32)
    kt = rng.normal(0, 1, (L, B, n, Hkv, d)).astype(np.float32)
    vt = rng.normal(0, 1, (L, B, n, Hkv, d)).astype(np.float32)
    return q, kc, vc, np.asarray(ctx, np.int32), kt, vt


def _sdpa(q, k, v, allowed, scale):
    """q [Hq, nq, d], k/v [Hq, nk, d] float64, allowed [nq, nk] bool."""
    return F.scaled_dot_product_attention(torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v),
                                          attn_mask=torch.from_numpy(allowed), scale=scale).numpy()


@pytest.mark.parametrize("G", [1, 2, 4])
def test_chain_equals_causal(G):
    """A chain tree (parent of i is i-1) makes the tree part lower-triangular: the result must be
    causal attention over [context, chain]."""
    rng = np.random.default_rng(10 + G)
    L, B, n, Hkv, d, S = 2, 2, 7, 2, 16, 12
    Hq = Hkv * G
    ctx = [9, 12]
    q, kc, vc, cl, kt, vt = _inputs(rng, L, B, n, Hq, Hkv, d, S, ctx)
    parents = [-1] + list(range(n - 1))
    mask = np.stack([_mask_from_parents(parents)] * B)
    scale = 0.3
    out = oracle.tree_attention(q, kc, vc, cl, kt, vt, mask, scale=scale)
    for l in range(L):
        for b in range(B):
            c = ctx[b]
            k_all = np.concatenate([kc[l, b, :c], kt[l, b]], 0).astype(np.float64)  # [c+n, Hkv, d]
            v_all = np.concatenate([vc[l, b, :c], vt[l, b]], 0).astype(np.float64)
            kh = np.repeat(k_all.transpose(1, 0, 2), G, axis=0)
            vh = np.repeat(v_all.transpose(1, 0, 2), G, axis=0)
            qh = q[l, b].astype(np.float64).transpose(1, 0, 2)
            allowed = np.ones((n, c + n), bool)
            allowed[:, c:] = np.tril(np.ones((n, n), bool))
            ref = _sdpa(qh, kh, vh, allowed, scale).transpose(1, 0, 2)
            np.testing.assert_allclose(out[l, b], ref, rtol=1e-11, atol=1e-12)


def _random_tree(rng, n):
    return [-1] + [int(rng.integers(0, i)) for i in range(1, n)]


@pytest.mark.parametrize("seed", range(6))
def test_each_path_runs_alone(seed):
    """Node i's output equals running its root -> i path alone as a causal sequence after the
    context (brute force per node, tiny trees)."""
    rng = np.random.default_rng(100 + seed)
    L, B, Hkv, G, d, S = 1, 2, 2, 2, 8, 6
    n = int(rng.integers(1, 12))
    Hq = Hkv * G
    ctx = [int(rng.integers(0, S + 1)) for _ in range(B)]
    q, kc, vc, cl, kt, vt = _inputs(rng, L, B, n, Hq, Hkv, d, S, ctx)
    parents = [_random_tree(rng, n) for _ in range(B)]
    mask = np.stack([_mask_from_parents(p) for p in parents])
    out = oracle.tree_attention(q, kc, vc, cl, kt, vt, mask)
    scale = 1.0 / np.sqrt(d)
    for b in range(B):
        c = ctx[b]
        for i in range(n):
            path = []
            j = i
            while j >= 0:
                path.append(j)
                j = parents[b][j]
            path = path[::-1]
            k_seq = np.concatenate([kc[0, b, :c], kt[0, b, path]], 0).astype(np.float64)
            v_seq = np.concatenate([vc[0, b, :c], vt[0, b, path]], 0).astype(np.float64)
            qh = q[0, b, i].astype(np.float64)[:, None, :]  # [Hq, 1, d], last position of the path
            kh = np.repeat(k_seq.transpose(1, 0, 2), G, axis=0)
            vh = np.repeat(v_seq.transpose(1, 0, 2), G, axis=0)
            allowed = np.ones((1, k_seq.shape[0]), bool)
            ref = _sdpa(qh, kh, vh, allowed, scale)[:, 0, :]
            np.testing.assert_allclose(out[0, b, i], ref, rtol=1e-11, atol=1e-12)


def test_root_with_empty_context_is_its_own_value():
    """With no context the root sees only itself: its output is exactly its own V row."""
    rng = np.random.default_rng(5)
    q, kc, vc, cl, kt, vt = _inputs(rng, 1, 1, 3, 4, 2, 8, 4, [0])
    mask = _mask_from_parents([-1, 0, 0])[None]
    out = oracle.tree_attention(q, kc, vc, cl, kt, vt, mask)
    for h in range(4):
        np.testing.assert_array_equal(out[0, 0, 0, h], vt[0, 0, 0, h // 2].astype(np.float64))


def test_bf16_bits_and_rows_api():
    """bf16 inputs (uint16 bit patterns) decode to the same values torch gives; the selected-rows
    entry point agrees with the full one."""
    rng = np.random.default_rng(9)
    L, B, n, Hq, Hkv, d, S = 2, 1, 5, 4, 1, 16, 10
    f = [torch.from_numpy(a).to(torch.bfloat16) for a in _inputs(rng, L, B, n, Hq, Hkv, d, S, [7])[:6] if a.dtype == np.float32]
    bits = [t.view(torch.int16).numpy().view(np.uint16) for t in f]
    wide = [t.to(torch.float32).numpy() for t in f]
    ctx = np.array([7], np.int32)
    mask = _mask_from_parents([-1, 0, 1, 0, 3])[None]
    a = oracle.tree_attention(bits[0], bits[1], bits[2], ctx, bits[3], bits[4], mask)
    b = oracle.tree_attention(wide[0], wide[1], wide[2], ctx, wide[3], wide[4], mask)
    np.testing.assert_array_equal(a, b)
    rows = np.array([[1, 0, 4, 3], [0, 0, 0, 0], [1, 0, 2, 1]], np.int32)
    r = oracle.tree_attention_rows(rows, bits[0], bits[1], bits[2], ctx, bits[3], bits[4], mask)
    for j, (l, bb, i, h) in enumerate(rows):
        np.testing.assert_array_equal(r[j], a[l, bb, i, h])


def test_layer_range_and_bad_context():
    rng = np.random.default_rng(2)
    q, kc, vc, cl, kt, vt = _inputs(rng, 3, 1, 2, 2, 1, 8, 4, [4])
    mask = _mask_from_parents([-1, 0])[None]
    full = oracle.tree_attention(q, kc, vc, cl, kt, vt, mask)
    part = oracle.tree_attention(q, kc, vc, cl, kt, vt, mask, layers=(1, 2))
    np.testing.assert_array_equal(part[1], full[1])
    assert not part[0].any() and not part[2].any()
    with pytest.raises(oracle.OracleError):
        oracle.tree_attention(q, kc, vc, np.array([5], np.int32), kt, vt, mask)  # ctx > S_max
