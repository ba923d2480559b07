"""The C-ABI library builds, loads without a GPU, exports every symbol include/eagle.h declares,
and rejects bad arguments on the host before touching the device (no compute call here)."""
import ctypes
import os
import re

import pytest

import eagle_draft_tree_gb300 as eg

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "eagle.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(eagle_[a-z0-9_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    lib = eg.load()
    names = declared_functions()
    assert len(names) >= 10
    for name in names:
        assert hasattr(lib, name), name
    # the binding knows every declared symbol's signature
    assert set(names) == set(eg._SIGS)


def test_status_strings():
    lib = eg.load()
    for s in range(6):
        assert lib.eagle_status_string(s).decode()
    assert lib.eagle_status_string(99).decode() == "unknown status"


def _tree(**kw):
    base = dict(batch=1, vocab=1000, depth=3, topk=4, keep=10, tree_temp=1.0)
    base.update(kw)
    return eg.TreeCfg(**base)


@pytest.mark.parametrize("kw,code", [
    (dict(), None),
    (dict(batch=0), eg.EAGLE_ERR_INVALID_ARG),
    (dict(topk=17), eg.EAGLE_ERR_UNSUPPORTED),
    (dict(depth=8, topk=10, keep=64), eg.EAGLE_ERR_UNSUPPORTED),
    (dict(keep=1000), eg.EAGLE_ERR_INVALID_ARG),
    (dict(tree_temp=0.0), eg.EAGLE_ERR_INVALID_ARG),
    (dict(topk=5, vocab=4), eg.EAGLE_ERR_INVALID_ARG),
    (dict(depth=40, topk=16, keep=60), eg.EAGLE_ERR_UNSUPPORTED),
])
def test_build_tree_host_validation(kw, code):
    lib = eg.load()
    cfg = _tree(**kw)
    size = lib.eagle_build_tree_workspace_size(ctypes.byref(cfg))
    if code is None:
        assert size >= 256
        # null pointers are caught before any launch
        st = lib.eagle_build_tree(ctypes.byref(cfg), None, None, None, None, None, None, None, None, None, 0, None)
        assert st == eg.EAGLE_ERR_INVALID_ARG
    else:
        assert size == 0
        st = lib.eagle_build_tree(ctypes.byref(cfg), *([None] * 9), 0, None)
        assert st == code


@pytest.mark.parametrize("kw,code", [
    (dict(), None),
    (dict(heads_q=6, heads_kv=4), eg.EAGLE_ERR_UNSUPPORTED),
    (dict(head_dim=96), eg.EAGLE_ERR_UNSUPPORTED),
    (dict(nodes=65), eg.EAGLE_ERR_UNSUPPORTED),
    (dict(dtype=7), eg.EAGLE_ERR_INVALID_ARG),
    (dict(max_seq=-1), eg.EAGLE_ERR_INVALID_ARG),
])
def test_attention_host_validation(kw, code):
    lib = eg.load()
    base = dict(batch=1, layers=2, nodes=11, heads_q=4, heads_kv=2, head_dim=64, max_seq=128, dtype=1, scale=0.0)
    base.update(kw)
    cfg = eg.AttnCfg(**base)
    size = lib.eagle_tree_attention_workspace_size(ctypes.byref(cfg))
    st = lib.eagle_tree_attention(ctypes.byref(cfg), *([None] * 9), 0, None)
    if code is None:
        assert size >= 256 and st == eg.EAGLE_ERR_INVALID_ARG
    else:
        assert size == 0 and st == code


@pytest.mark.parametrize("kw,code", [
    (dict(), None),
    (dict(temperature=-1.0), eg.EAGLE_ERR_INVALID_ARG),
    (dict(keep=70), eg.EAGLE_ERR_UNSUPPORTED),
    (dict(vocab=10_000_000), eg.EAGLE_ERR_UNSUPPORTED),
])
def test_verify_host_validation(kw, code):
    lib = eg.load()
    base = dict(batch=2, vocab=1000, depth=3, topk=4, keep=10, temperature=1.0)
    base.update(kw)
    cfg = eg.VerifyCfg(**base)
    size = lib.eagle_tree_verify_workspace_size(ctypes.byref(cfg))
    st = lib.eagle_tree_verify(ctypes.byref(cfg), *([None] * 11), 0, None)
    if code is None:
        assert size >= 256 and st == eg.EAGLE_ERR_INVALID_ARG
    else:
        assert size == 0 and st == code


def test_workspace_too_small_rejected():
    lib = eg.load()
    cfg = _tree()
    fake = ctypes.c_void_p(256 * 1024)  # never dereferenced: the size check fails first
    st = lib.eagle_build_tree(ctypes.byref(cfg), fake, fake, fake, fake, fake, fake, fake, None, fake, 16, None)
    assert st == eg.EAGLE_ERR_INVALID_ARG


def test_binding_refuses_cpu_tensors():
    import torch
    x = torch.zeros((1, 9, 1000), dtype=torch.float32)
    r = torch.zeros((1,), dtype=torch.int32)
    with pytest.raises((ValueError, RuntimeError, AssertionError)):
        eg.build_tree(x, r, depth=3, topk=4, keep=10, ws=object())


def test_context_split_is_planned_only_for_small_unit_counts():
    lib = eg.load()
    small = eg.AttnCfg(1, 1, 61, 32, 8, 128, 2048, eg.EAGLE_DTYPE_BF16, 0.0)   # 8 units: split
    full = eg.AttnCfg(1, 32, 61, 32, 8, 128, 2048, eg.EAGLE_DTYPE_BF16, 0.0)   # 256 units: none
    assert lib.eagle_tree_attention_workspace_size(ctypes.byref(small)) > 256
    assert lib.eagle_tree_attention_workspace_size(ctypes.byref(full)) == 256


@pytest.mark.parametrize("parents,code", [
    ([-1, 0, 0, 1], None),
    ([0, 0], eg.EAGLE_ERR_INVALID_ARG),           # the root has a parent
    ([-1, 0, 3, 1], eg.EAGLE_ERR_INVALID_ARG),    # a parent after its child
    ([-1] + [0] * 17, eg.EAGLE_ERR_UNSUPPORTED),  # 17 children of one node
])
def test_static_tree_host_validation(parents, code):
    lib = eg.load()
    cfg = eg.static_tree_cfg(2, 1000, parents, 1.0)
    size = lib.eagle_build_static_tree_workspace_size(ctypes.byref(cfg))
    st = lib.eagle_build_static_tree(ctypes.byref(cfg), *([None] * 9), 0, None)
    if code is None:
        assert size >= 256 and st == eg.EAGLE_ERR_INVALID_ARG  # valid template, null buffers
    else:
        assert size == 0 and st == code


def test_sampled_and_stepwise_host_validation():
    lib = eg.load()
    cfg = _tree()
    fake = ctypes.c_void_p(256 * 1024)  # never dereferenced: a host check fails first
    P = [fake] * 7
    # sampled build: the uniforms are required; vocabularies above 2^21 are not supported
    st = lib.eagle_build_tree_sampled(ctypes.byref(cfg), fake, None, *P, fake, 1 << 30, None)
    assert st == eg.EAGLE_ERR_INVALID_ARG
    big = _tree(vocab=(1 << 21) + 4)
    assert lib.eagle_build_tree_sampled(ctypes.byref(big), *([fake] * 9), fake, 1 << 30, None) == eg.EAGLE_ERR_UNSUPPORTED
    scfg = eg.static_tree_cfg(2, 1000, [-1, 0, 0, 1], 1.0)
    st = lib.eagle_build_static_tree_sampled(ctypes.byref(scfg), fake, None, *P, fake, 1 << 30, None)
    assert st == eg.EAGLE_ERR_INVALID_ARG
    # stepwise: frontier outputs are required while a deeper frontier remains; depth in 1..D-1
    assert lib.eagle_build_begin(ctypes.byref(cfg), fake, None, fake, 1 << 30, None, None, None) == \
        eg.EAGLE_ERR_INVALID_ARG
    for d in (0, 3):
        assert lib.eagle_build_expand(ctypes.byref(cfg), d, fake, None, fake, 1 << 30, fake, fake, None) == \
            eg.EAGLE_ERR_INVALID_ARG
    assert lib.eagle_build_expand(ctypes.byref(cfg), 1, fake, None, fake, 1 << 30, None, fake, None) == \
        eg.EAGLE_ERR_INVALID_ARG
    # too small a workspace (the stepwise state lives in it)
    assert lib.eagle_build_expand(ctypes.byref(cfg), 2, fake, None, fake, 16, None, None, None) == \
        eg.EAGLE_ERR_INVALID_ARG
    assert lib.eagle_build_finalize(ctypes.byref(cfg), fake, fake, 1 << 30, None, *([fake] * 5), None) == \
        eg.EAGLE_ERR_INVALID_ARG
    assert lib.eagle_build_finalize(ctypes.byref(_tree(batch=0)), fake, fake, 1 << 30, *([fake] * 6), None) == \
        eg.EAGLE_ERR_INVALID_ARG
