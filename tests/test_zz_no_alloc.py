"""eagle_tree_verify_static, the verify entry point that uses the library's static device scratch
instead of a caller workspace: it must agree with eagle_tree_verify (the same kernels run, so the
outputs are identical) over two consecutive calls, and reject configurations larger than its
scratch on the host.  This file sorts last so the static scratch is also exercised after every
other test has run."""
import ctypes

import numpy as np
import pytest
import torch

import datagen
import eagle_draft_tree_gb300 as eg

DEV = "cuda"


def test_static_verify_rejects_configs_beyond_its_scratch():
    lib = eg.load()
    # 120 sequences of 64 nodes need more than the 256 KB scratch (113 of 64 fit)
    big = eg.VerifyCfg(120, 1000, 8, 8, 63, 1.0)
    assert lib.eagle_tree_verify_workspace_size(ctypes.byref(big)) > (256 << 10)
    st = lib.eagle_tree_verify_static(ctypes.byref(big), *([None] * 10), None)
    assert st == eg.EAGLE_ERR_UNSUPPORTED
    # an invalid configuration is reported as by eagle_tree_verify
    bad = eg.VerifyCfg(0, 1000, 8, 8, 60, 1.0)
    assert lib.eagle_tree_verify_static(ctypes.byref(bad), *([None] * 10), None) == eg.EAGLE_ERR_INVALID_ARG


def _inputs(wl, seed):
    draft = datagen.draft_logits(wl.batch, wl.rows, wl.vocab, seed, DEV)
    root = datagen.root_tokens(wl.batch, wl.vocab, seed, DEV)
    tree = eg.build_tree(draft, root, depth=wl.depth, topk=wl.topk, keep=wl.keep)
    target = datagen.target_logits(draft, tree["node_row"], datagen.noise_sigmas(wl, seed), seed)
    u = datagen.uniforms(wl.batch, wl.nodes, seed, DEV)
    return draft, tree, target, u


@pytest.mark.gpu
@pytest.mark.parametrize("name,T", [("llama31_8b", 1.0), ("serving_b64", 0.7), ("vicuna_13b", 0.0)])
def test_static_verify_matches_workspace_verify(name, T):
    wl = datagen.WORKLOADS[name].with_(temperature=T)
    draft, tree, target, u = _inputs(wl, seed=3)
    ref = eg.tree_verify(target, draft, tree, u, temperature=T, depth=wl.depth, topk=wl.topk)
    torch.cuda.synchronize()
    ref = {k: v.cpu().numpy() for k, v in ref.items()}
    for call in range(2):  # two consecutive calls: nothing carries over in the static scratch
        got = eg.tree_verify_static(target, draft, tree, u, temperature=T, depth=wl.depth, topk=wl.topk)
        torch.cuda.synchronize()
        got = {k: v.cpu().numpy() for k, v in got.items()}
        for k in ("out_tokens", "out_len", "out_path"):
            assert np.array_equal(got[k], ref[k]), (call, k)
        fin = np.isfinite(ref["out_ratio"])
        assert np.array_equal(np.isnan(got["out_ratio"]), np.isnan(ref["out_ratio"]))
        np.testing.assert_allclose(got["out_ratio"][fin], ref["out_ratio"][fin], rtol=1e-6, atol=0)


@pytest.mark.gpu
def test_static_verify_after_a_different_round():
    """A round of another shape in between leaves no trace in the static scratch."""
    wl = datagen.WORKLOADS["llama31_8b"]
    d1, t1, g1, u1 = _inputs(wl, seed=5)
    first = eg.tree_verify_static(g1, d1, t1, u1, temperature=1.0, depth=wl.depth, topk=wl.topk)
    other = datagen.WORKLOADS["serving_b64"]
    d2, t2, g2, u2 = _inputs(other, seed=6)
    eg.tree_verify_static(g2, d2, t2, u2, temperature=0.7, depth=other.depth, topk=other.topk)
    again = eg.tree_verify_static(g1, d1, t1, u1, temperature=1.0, depth=wl.depth, topk=wl.topk)
    torch.cuda.synchronize()
    for k in ("out_tokens", "out_len", "out_path"):
        assert torch.equal(first[k], again[k]), k


@pytest.mark.gpu
def test_static_verify_reports_a_malformed_tree_through_out_len():
    """This entry point never reads the device status word, so a device-side error has to show in
    its outputs: a sequence whose tree names a parent after its child commits nothing
    (out_len = 0), while the other sequences of the call commit what eagle_tree_verify commits."""
    wl = datagen.WORKLOADS["serving_b64"].with_(batch=4)
    draft, tree, target, u = _inputs(wl, seed=7)
    ref = eg.tree_verify(target, draft, tree, u, temperature=0.7, depth=wl.depth, topk=wl.topk)
    bad = {k: v.clone() for k, v in tree.items()}
    bad["parents"][2, 5] = 9  # node 5's parent after it: not a tree in creation order
    for _ in range(2):
        got = eg.tree_verify_static(target, draft, bad, u, temperature=0.7, depth=wl.depth, topk=wl.topk)
        torch.cuda.synchronize()
        assert int(got["out_len"][2]) == 0
        for b in (0, 1, 3):
            assert int(got["out_len"][b]) == int(ref["out_len"][b])
            assert torch.equal(got["out_tokens"][b], ref["out_tokens"][b])
