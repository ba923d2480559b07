"""GPU parity of eagle_kv_commit against the oracle: every byte of both caches at small sizes
(committed paths from real oracle rounds, refused sequences, nothing committed), and sampled
(layer, sequence) slices at the 8B shape, each checked by the oracle on its own slice."""
import numpy as np
import pytest
import torch

import eagle_draft_tree_gb300 as eg
import oracle
from tests.gpu_parity import np_

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _bits(t):
    """The stored bytes of a tensor as numpy (bf16 -> uint16 bits, f32 as is)."""
    return np_(t)


def _commit_case(seed, L, B, n, Hkv, d, S, D, k, dtype):
    rng = np.random.default_rng(seed)
    V, m = 300, n - 1
    R = 1 + (D - 1) * k
    draft = rng.normal(0, 2, (B, R, V)).astype(np.float32)
    tree = oracle.build_tree(draft, rng.integers(0, V, B).astype(np.int32), D, k, m)
    target = (draft[np.arange(B)[:, None], np.maximum(tree["node_row"], 0)] +
              rng.normal(0, 0.3, (B, n, V))).astype(np.float32)
    ver = oracle.tree_verify(target, draft, tree["tokens"], tree["parents"], tree["node_row"],
                             rng.random((B, n)).astype(np.float32), 1.0, D + 1)
    g = torch.Generator().manual_seed(seed)
    mk = lambda *s: torch.randn(*s, generator=g).to(dtype).to(DEV)  # noqa: E731
    kt, vt, kc, vc = mk(L, B, n, Hkv, d), mk(L, B, n, Hkv, d), mk(L, B, S, Hkv, d), mk(L, B, S, Hkv, d)
    ctx = torch.from_numpy(rng.integers(0, S - D - 1, B).astype(np.int32)).to(DEV)
    return ver, kt, vt, kc, vc, ctx


def _check(ver, kt, vt, kc, vc, ctx, path=None, ln=None, expect_ok=True):
    path = ver["out_path"] if path is None else path
    ln = ver["out_len"] if ln is None else ln
    ref_k, ref_v, ref_ctx, ok = oracle.kv_commit(_bits(kt), _bits(vt), path, ln, np_(ctx), _bits(kc), _bits(vc))
    ws = eg.Workspace(device=DEV)
    new_ctx = eg.kv_commit(kt, vt, torch.from_numpy(np.ascontiguousarray(path, np.int32)).to(DEV),
                           torch.from_numpy(np.ascontiguousarray(ln, np.int32)).to(DEV), ctx, kc, vc, ws=ws)
    status = ws.status()
    assert ok == expect_ok
    assert status == (eg.EAGLE_OK if expect_ok else eg.EAGLE_ERR_DEVICE_INPUT)
    assert np.array_equal(np_(new_ctx), ref_ctx)
    assert np.array_equal(_bits(kc), ref_k) and np.array_equal(_bits(vc), ref_v)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("shape", [(2, 3, 10, 2, 128, 40, 3, 3), (3, 5, 21, 4, 64, 64, 5, 4),
                                   (1, 2, 61, 8, 128, 80, 8, 10)])
def test_commit_matches_oracle(shape, dtype):
    L, B, n, Hkv, d, S, D, k = shape
    for seed in (1, 2):
        ver, kt, vt, kc, vc, ctx = _commit_case(seed, L, B, n, Hkv, d, S, D, k, dtype)
        _check(ver, kt, vt, kc, vc, ctx)


def test_refused_and_empty_commits():
    L, B, n, Hkv, d, S, D, k = 2, 4, 10, 2, 64, 24, 3, 3
    ver, kt, vt, kc, vc, ctx = _commit_case(5, L, B, n, Hkv, d, S, D, k, torch.bfloat16)
    path = np.array(ver["out_path"], np.int32)
    ln = np.array(ver["out_len"], np.int32)
    ln[0] = 0                       # nothing committed: a no-op
    ln[1] = D + 2                   # more than D + 1 tokens: refused
    path[2, 0], ln[2] = n, max(ln[2], 2)  # a node id outside [1, n): refused
    ctx[3] = S - 1                  # no room for the root and one more row: refused
    ln[3] = 2
    path[3, 0] = 1
    _check(ver, kt, vt, kc, vc, ctx, path, ln, expect_ok=False)


def test_commit_at_the_8b_shape_sampled():
    """The bench's shape (32 layers, 8 KV heads of 128, 61 nodes), a cache with room for the
    round; sampled (layer, sequence) slices checked by the oracle one by one."""
    L, B, n, Hkv, d, D, k, ctx0 = 32, 2, 61, 8, 128, 8, 10, 2048
    S = ctx0 + D + 8
    ver, kt, vt, kc, vc, _ = _commit_case(9, L, B, n, Hkv, d, S, D, k, torch.bfloat16)
    ctx = torch.full((B,), ctx0, dtype=torch.int32, device=DEV)
    ctx[1] = ctx0 - 5
    before_k, before_v = kc.clone(), vc.clone()
    ws = eg.Workspace(device=DEV)
    path_t = torch.from_numpy(np.ascontiguousarray(ver["out_path"], np.int32)).to(DEV)
    ln_t = torch.from_numpy(np.ascontiguousarray(ver["out_len"], np.int32)).to(DEV)
    new_ctx = eg.kv_commit(kt, vt, path_t, ln_t, ctx, kc, vc, ws=ws)
    assert ws.status() == eg.EAGLE_OK
    rng = np.random.default_rng(0)
    for l, b in {(0, 0), (L - 1, B - 1), *((int(rng.integers(L)), int(rng.integers(B))) for _ in range(6))}:
        sl = (slice(l, l + 1), slice(b, b + 1))
        ref_k, ref_v, ref_ctx, ok = oracle.kv_commit(
            _bits(kt[sl]), _bits(vt[sl]), ver["out_path"][b:b + 1], ver["out_len"][b:b + 1], np_(ctx[b:b + 1]),
            _bits(before_k[sl]), _bits(before_v[sl]))
        assert ok and int(new_ctx[b]) == int(ref_ctx[0])
        assert np.array_equal(_bits(kc[sl]), ref_k) and np.array_equal(_bits(vc[sl]), ref_v)
