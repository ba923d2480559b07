"""fp64 CPU oracle for the EAGLE draft-tree verify round.

TEST INFRASTRUCTURE ONLY: this package checks the CUDA library; it is not part of it.  Only
``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import it.
It shares no code with the CUDA path and never imports it.

The arithmetic lives in ``eagle_oracle.c`` (plain C, double precision, one element at a time);
this module compiles it with gcc on first use and wraps it with numpy arrays.  Every function
cites the page passage it restates; the readings taken where the pages are silent are listed at
the top of the C file.

Parity pins: every function here is pinned by ``tests/test_oracle_*.py`` (invariants the pages
fix, brute force on tiny inputs, library special cases, and hand-worked fixtures under
``tests/golden/``).  No function is unpinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "eagle_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

ORC_OK, ORC_BAD_ARG, ORC_NOT_CLOSED, ORC_BAD_TREE = 0, 1, 2, 3
DT_F32, DT_BF16 = 0, 1


class OracleError(RuntimeError):
    pass


def compile_source(src: str, out: str) -> str:
    """Compile one C source file into a shared library (gcc, OpenMP when available)."""
    tmp = out + ".%d.tmp" % os.getpid()
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-o", tmp, src, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile ``eagle_oracle.c`` into ``liboracle.so`` next to it."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    return compile_source(_SRC, _LIB)


def _bind(path: str):
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    I = ctypes.c_int
    D = ctypes.c_double
    lib.orc_build_tree.argtypes = [I, I, I, I, I, D, P, P, P, P, P, P, P, P, P, I]
    lib.orc_tree_attention.argtypes = [I, I, I, I, I, I, I, I, D, P, P, P, P, P, P, P, P, I, I, I]
    lib.orc_tree_attention_rows.argtypes = [I, I, I, I, I, I, I, I, D, P, P, P, P, P, P, P, P, I, P, I]
    lib.orc_tree_verify.argtypes = [I, I, I, I, I, D, P, P, P, P, P, P, P, P, P, P, P, I]
    lib.orc_kv_commit.argtypes = [I, I, I, I, I, I, I, I, P, P, P, P, P, P, P, P]
    lib.orc_build_static_tree.argtypes = [I, I, I, P, D, P, P, P, P, P, P, P, P]
    lib.orc_build_tree_ex.argtypes = [I, I, I, I, I, D, P, P, P, P, P, P, P, P, P, P, P, P, P, I]
    lib.orc_build_static_tree_ex.argtypes = [I, I, I, P, D, P, P, P, P, P, P, P, P, P, P]
    lib.orc_row_children.argtypes = [I, I, I, D, P, P, P, P, P]
    for f in (lib.orc_build_tree, lib.orc_tree_attention, lib.orc_tree_attention_rows, lib.orc_tree_verify,
              lib.orc_kv_commit, lib.orc_build_static_tree, lib.orc_build_tree_ex, lib.orc_build_static_tree_ex, lib.orc_row_children):
        f.restype = I
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(build())
    return _lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _check(status: int, what: str) -> None:
    if status != ORC_OK:
        raise OracleError(f"{what}: oracle status {status}")


def _threads(nthreads):
    return int(nthreads) if nthreads else 0


class Oracle:
    """The oracle bound to one compiled library (the default one, or a variant a test compiled)."""

    def __init__(self, path: str | None = None):
        self._path = path

    def _lib(self):
        if self._path is None:
            return _load()
        if not hasattr(self, "_handle"):
            self._handle = _bind(self._path)
        return self._handle

    def build_tree(self, *a, **kw):
        return build_tree(*a, _lib=self._lib(), **kw)

    def tree_attention(self, *a, **kw):
        return tree_attention(*a, _lib=self._lib(), **kw)

    def tree_attention_rows(self, *a, **kw):
        return tree_attention_rows(*a, _lib=self._lib(), **kw)

    def tree_verify(self, *a, **kw):
        return tree_verify(*a, _lib=self._lib(), **kw)

    def kv_commit(self, *a, **kw):
        return kv_commit(*a, _lib=self._lib(), **kw)

    def build_static_tree(self, *a, **kw):
        return build_static_tree(*a, _lib=self._lib(), **kw)

    def row_children(self, *a, **kw):
        return row_children(*a, _lib=self._lib(), **kw)


def build_tree(draft_logits, root_token, depth: int, topk: int, keep: int, tree_temp: float = 1.0,
               nthreads: int | None = None, child_u=None, frontier: bool = False, _lib=None):
    """EAGLE-2 dynamic draft tree ([EAGLE-2 notes] Expanding / Rerank / Tree Attention Mask).

    draft_logits: float32 [B, R, V], R = 1 + (depth-1)*topk.  root_token: int32 [B].
    child_u: None for top-k children (greedy), else float32 [B, R, topk] uniforms: the children of
    row r are topk inverse-CDF draws from softmax(x_r / tree_temp) ([EAGLE-1 notes] A.1,
    non-greedy), in draw order.
    Returns dict of tokens/parents/depths/node_row int32 [B, n], mask uint64 [B, n, W],
    node_logv float64 [B, n], margin float64 [B] (smallest relative key gap at a selection),
    draw_gap float64 [B] (smallest distance of a uniform to the CDF step deciding its draw; inf
    without draws) and, with ``frontier``, front_tok/front_par int32 [B, depth-1, topk]: the
    frontier of depths 1..depth-1 in slot order and each node's parent slot (-1 at depth 1).
    """
    x = _c(draft_logits, np.float32)
    B, R, V = x.shape
    assert R == 1 + (depth - 1) * topk, "draft rows must be 1 + (D-1)k"
    root = _c(root_token, np.int32).reshape(B)
    u = None if child_u is None else _c(child_u, np.float32).reshape(B, R, topk)
    n = keep + 1
    W = (n + 63) // 64
    out = dict(
        tokens=np.zeros((B, n), np.int32), parents=np.zeros((B, n), np.int32),
        depths=np.zeros((B, n), np.int32), node_row=np.zeros((B, n), np.int32),
        mask=np.zeros((B, n, W), np.uint64), node_logv=np.zeros((B, n), np.float64),
        margin=np.zeros(B, np.float64), draw_gap=np.zeros(B, np.float64))
    ft = fp = None
    if frontier:
        ft = np.zeros((B, max(depth - 1, 1), topk), np.int32)
        fp = np.zeros_like(ft)
    st = (_lib or _load()).orc_build_tree_ex(B, V, depth, topk, keep, float(tree_temp), _ptr(x), _ptr(u),
                                             _ptr(root), _ptr(out["tokens"]), _ptr(out["parents"]),
                                             _ptr(out["depths"]), _ptr(out["node_row"]), _ptr(out["mask"]),
                                             _ptr(out["node_logv"]), _ptr(out["margin"]), _ptr(out["draw_gap"]),
                                             _ptr(ft), _ptr(fp), _threads(nthreads))
    _check(st, "build_tree")
    if frontier:
        out["front_tok"] = ft[:, :depth - 1]
        out["front_par"] = fp[:, :depth - 1]
    return out


def _attn_common(q, k_cache, v_cache, ctx_len, k_tree, v_tree, mask):
    dt = np.dtype(q.dtype)
    if dt == np.float32:
        dtype = DT_F32
    elif dt == np.uint16:  # bf16 bit patterns
        dtype = DT_BF16
    else:
        raise TypeError("q/k/v must be float32 or uint16 (bf16 bits)")
    arrs = [_c(a, dt) for a in (q, k_cache, v_cache, k_tree, v_tree)]
    return dtype, arrs, _c(ctx_len, np.int32), _c(mask, np.uint64)


def tree_attention(q, k_cache, v_cache, ctx_len, k_tree, v_tree, mask, scale: float | None = None,
                   layers: tuple[int, int] | None = None, nthreads: int | None = None, _lib=None):
    """Tree-masked GQA attention, literal fp64 softmax ([EAGLE-3 blog] section 5;
    [EAGLE-2 notes] Tree Attention Mask).

    q [L,B,n,Hq,d]; k_cache/v_cache [L,B,S_max,Hkv,d]; k_tree/v_tree [L,B,n,Hkv,d]; ctx_len [B];
    mask uint64 [B,n,W].  Float arrays are float32 or uint16 holding bf16 bits.
    Returns float64 [L,B,n,Hq,d] (layers outside ``layers`` are zero).
    """
    dtype, (q, kc, vc, kt, vt), ctx, msk = _attn_common(q, k_cache, v_cache, ctx_len, k_tree, v_tree, mask)
    L, B, n, Hq, d = q.shape
    S_max, Hkv = kc.shape[2], kc.shape[3]
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    l0, l1 = layers if layers is not None else (0, L)
    out = np.zeros((L, B, n, Hq, d), np.float64)
    st = (_lib or _load()).orc_tree_attention(L, B, n, Hq, Hkv, d, S_max, dtype, float(scale), _ptr(q), _ptr(kc), _ptr(vc),
                                    _ptr(ctx), _ptr(kt), _ptr(vt), _ptr(msk), _ptr(out), l0, l1,
                                    _threads(nthreads))
    _check(st, "tree_attention")
    return out


def tree_attention_rows(rows, q, k_cache, v_cache, ctx_len, k_tree, v_tree, mask, scale: float | None = None,
                        nthreads: int | None = None, _lib=None):
    """Same as :func:`tree_attention` for selected query rows only; rows int [count, 4] of
    (layer, seq, node, head).  Returns float64 [count, d]."""
    dtype, (q, kc, vc, kt, vt), ctx, msk = _attn_common(q, k_cache, v_cache, ctx_len, k_tree, v_tree, mask)
    L, B, n, Hq, d = q.shape
    S_max, Hkv = kc.shape[2], kc.shape[3]
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    r = _c(rows, np.int32).reshape(-1, 4)
    out = np.zeros((r.shape[0], d), np.float64)
    st = (_lib or _load()).orc_tree_attention_rows(L, B, n, Hq, Hkv, d, S_max, dtype, float(scale), _ptr(q), _ptr(kc),
                                         _ptr(vc), _ptr(ctx), _ptr(kt), _ptr(vt), _ptr(msk), _ptr(r),
                                         r.shape[0], _ptr(out), _threads(nthreads))
    _check(st, "tree_attention_rows")
    return out


def tree_verify(target_logits, draft_logits, tokens, parents, node_row, uniforms, temperature: float,
                max_commit: int, nthreads: int | None = None, _lib=None):
    """Multi-round tree speculative sampling ([EAGLE-1 notes] A3, 3.3, A.2; [EAGLE-3 blog] 1, 2).

    target_logits float32 [B,n,V]; draft_logits float32 [B,R,V]; tokens/parents/node_row int32
    [B,n]; uniforms float32 [B,n]; temperature 0 means greedy.  max_commit = D + 1.
    Returns dict out_tokens [B,max_commit] (-1 padded), out_len [B], out_path [B,max_commit-1]
    (accepted node ids, -1 padded), out_ratio float64 [B,n] (NaN for the root and at T = 0),
    margin float64 [B] (smallest |u - decision value| met on the walk).
    """
    tgt = _c(target_logits, np.float32)
    dft = _c(draft_logits, np.float32)
    B, n, V = tgt.shape
    R = dft.shape[1]
    assert dft.shape[0] == B and dft.shape[2] == V
    tok, par, row = (_c(a, np.int32).reshape(B, n) for a in (tokens, parents, node_row))
    u = _c(uniforms, np.float32).reshape(B, n)
    w = max(max_commit - 1, 1)
    out = dict(out_tokens=np.full((B, max_commit), -1, np.int32), out_len=np.zeros(B, np.int32),
               out_path=np.full((B, w), -1, np.int32), out_ratio=np.zeros((B, n), np.float64),
               margin=np.zeros(B, np.float64))
    st = (_lib or _load()).orc_tree_verify(B, V, R, n, max_commit, float(temperature), _ptr(tgt), _ptr(dft), _ptr(tok),
                                 _ptr(par), _ptr(row), _ptr(u), _ptr(out["out_tokens"]), _ptr(out["out_len"]),
                                 _ptr(out["out_path"]), _ptr(out["out_ratio"]), _ptr(out["margin"]),
                                 _threads(nthreads))
    _check(st, "tree_verify")
    return out


def kv_commit(k_tree, v_tree, out_path, out_len, ctx_len, k_cache, v_cache, _lib=None):
    """Append each sequence's root and accepted path to its KV cache ([EAGLE-3 blog] sections 1
    and 5; the reading is at ``orc_kv_commit`` in the C file).

    k_tree/v_tree [L,B,n,Hkv,d] and k_cache/v_cache [L,B,S_max,Hkv,d]: float32, or uint16 holding
    bf16 bits (the bytes are copied); out_path int32 [B,D]; out_len, ctx_len int32 [B].  The
    input caches are not modified.  Returns (k_cache', v_cache', new_ctx_len int32 [B], ok): ok
    is False when some sequence's commit was refused (that sequence is left as it was)."""
    kt, vt = np.ascontiguousarray(k_tree), np.ascontiguousarray(v_tree)
    kc, vc = np.array(k_cache, copy=True, order="C"), np.array(v_cache, copy=True, order="C")
    assert kt.dtype == vt.dtype == kc.dtype == vc.dtype and kt.dtype in (np.float32, np.uint16)
    L, B, n, Hkv, d = kt.shape
    S_max = kc.shape[2]
    assert kc.shape == (L, B, S_max, Hkv, d) and vc.shape == kc.shape and vt.shape == kt.shape
    path = _c(out_path, np.int32).reshape(B, -1)
    D = path.shape[1]
    ln, ctx = _c(out_len, np.int32).reshape(B), _c(ctx_len, np.int32).reshape(B)
    new_ctx = np.zeros(B, np.int32)
    st = (_lib or _load()).orc_kv_commit(L, B, n, Hkv, d, S_max, D, kt.dtype.itemsize, _ptr(kt), _ptr(vt),
                                         _ptr(path), _ptr(ln), _ptr(ctx), _ptr(kc), _ptr(vc), _ptr(new_ctx))
    if st not in (ORC_OK, ORC_BAD_ARG):
        _check(st, "kv_commit")
    return kc, vc, new_ctx, st == ORC_OK


def build_static_tree(draft_logits, root_token, template_parents, tree_temp: float = 1.0, child_u=None,
                      _lib=None):
    """Static tree or chain from a template ([EAGLE-1 notes] A.1, 4.3.1; the reading is at
    ``orc_build_static_tree`` in the C file).  draft_logits float32 [B, R, V] with R = the template
    nodes that have children; root_token int32 [B].  child_u: None (top-k children) or float32
    [B, R, kmax] uniforms, kmax = the most children of one template node (sampled children,
    [EAGLE-1 notes] A.1 non-greedy).  Returns tokens/parents/depths/node_row int32 [B, n], mask
    uint64 [B, n, 1], node_logv float64 [B, n], draw_gap float64 [B]."""
    x = _c(draft_logits, np.float32)
    B, R, V = x.shape
    tmpl = np.ascontiguousarray(template_parents, np.int32)
    n = tmpl.shape[0]
    root = _c(root_token, np.int32).reshape(B)
    out = {k: np.zeros((B, n), np.int32) for k in ("tokens", "parents", "depths", "node_row")}
    out["mask"] = np.zeros((B, n, 1), np.uint64)
    out["node_logv"] = np.zeros((B, n), np.float64)
    out["draw_gap"] = np.zeros(B, np.float64)
    internal = len(set(int(p) for p in tmpl[1:]))
    if R != internal:
        raise OracleError(f"build_static_tree: {R} draft rows for {internal} template nodes with children")
    u = None
    if child_u is not None:
        kmax = int(np.bincount(tmpl[1:], minlength=n).max()) if n > 1 else 1
        u = _c(child_u, np.float32).reshape(B, R, kmax)
    st = (_lib or _load()).orc_build_static_tree_ex(B, V, n, _ptr(tmpl), float(tree_temp), _ptr(x), _ptr(u),
                                                    _ptr(root), _ptr(out["tokens"]), _ptr(out["parents"]),
                                                    _ptr(out["depths"]), _ptr(out["node_row"]), _ptr(out["mask"]),
                                                    _ptr(out["node_logv"]), _ptr(out["draw_gap"]))
    _check(st, "build_static_tree")
    return out


def row_children(rows, topk: int, tree_temp: float = 1.0, child_u=None, _lib=None):
    """The children of independent draft rows ([EAGLE-1 notes] A.1: top-k when greedy, k draws
    from softmax(x / T) when not).  rows float32 [N, V]; child_u None or float32 [N, topk].
    Returns tok int32 [N, topk], lc float64 [N, topk] (log-confidences) and gap float64 [N, topk]
    (each draw's distance to the CDF step that decided it; inf for top-k children)."""
    x = _c(rows, np.float32)
    N, V = x.shape
    u = None if child_u is None else _c(child_u, np.float32).reshape(N, topk)
    tok = np.zeros((N, topk), np.int32)
    lc = np.zeros((N, topk), np.float64)
    gap = np.full((N, topk), np.inf, np.float64)
    st = (_lib or _load()).orc_row_children(N, V, topk, float(tree_temp), _ptr(x), _ptr(u), _ptr(tok), _ptr(lc),
                                            _ptr(gap))
    _check(st, "row_children")
    return dict(tok=tok, lc=lc, gap=gap)
