"""eagle_draft_tree_gb300 -- the EAGLE draft-tree verify round on GB300 (sm_103a).

A thin ctypes binding over ``libeagle.so`` (C ABI declared in ``include/eagle.h``).  Functions
here only marshal arguments (shape, dtype, device and contiguity checks, pointer extraction);
every step of the round runs in the library's CUDA kernels.  There is no CPU fallback: if the
library cannot be built or loaded, or a tensor is not on a CUDA device, the call raises.

    ws = Workspace()                       # grows as needed; zeroed once
    tree = build_tree(draft_logits, root_token, depth=D, topk=k, keep=m, ws=ws)
    out = tree_attention(q, k_cache, v_cache, ctx_len, k_tree, v_tree, tree["mask"], ws=ws)
    res = tree_verify(target_logits, draft_logits, tree, uniforms, temperature=T, depth=D,
                      topk=k, ws=ws)
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

__all__ = [
    "EagleError", "Workspace", "load", "library_path", "build_tree", "tree_attention", "tree_verify",
    "device_status", "last_launch_count", "selftest_wait_timeout", "kv_commit", "build_static_tree",
    "StaticTreeCfg", "static_tree_cfg", "chain_template", "TreeCfg", "AttnCfg", "VerifyCfg",
]

EAGLE_OK, EAGLE_ERR_INVALID_ARG, EAGLE_ERR_UNSUPPORTED, EAGLE_ERR_CUDA, EAGLE_ERR_TIMEOUT, EAGLE_ERR_DEVICE_INPUT = range(6)
EAGLE_DTYPE_F32, EAGLE_DTYPE_BF16 = 0, 1


class EagleError(RuntimeError):
    def __init__(self, what: str, status: int):
        super().__init__(f"{what}: {_status_string(status)} (status {status})")
        self.status = status


class TreeCfg(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("vocab", ctypes.c_int32), ("depth", ctypes.c_int32),
                ("topk", ctypes.c_int32), ("keep", ctypes.c_int32), ("tree_temp", ctypes.c_float)]


class AttnCfg(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("layers", ctypes.c_int32), ("nodes", ctypes.c_int32),
                ("heads_q", ctypes.c_int32), ("heads_kv", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("max_seq", ctypes.c_int32), ("dtype", ctypes.c_int32), ("scale", ctypes.c_float)]


class VerifyCfg(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("vocab", ctypes.c_int32), ("depth", ctypes.c_int32),
                ("topk", ctypes.c_int32), ("keep", ctypes.c_int32), ("temperature", ctypes.c_float)]


class StaticTreeCfg(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("vocab", ctypes.c_int32), ("nodes", ctypes.c_int32),
                ("tree_temp", ctypes.c_float), ("parents", ctypes.c_int8 * 64)]


def static_tree_cfg(batch: int, vocab: int, template_parents, tree_temp: float = 1.0) -> StaticTreeCfg:
    """The C struct for a template of parent indices (parents[0] = -1, parents[i] < i)."""
    tp = [int(x) for x in template_parents]
    if not 1 <= len(tp) <= 64:
        raise ValueError("a template has 1 to 64 nodes")
    arr = (ctypes.c_int8 * 64)(*(tp + [-1] * (64 - len(tp))))
    return StaticTreeCfg(batch, vocab, len(tp), tree_temp, arr)


def chain_template(depth: int) -> list[int]:
    """The chain of `depth` draft tokens below the root: parents -1, 0, 1, ..., depth - 1."""
    return [-1] + list(range(depth))


_lock = threading.Lock()
_lib = None

# every symbol of include/eagle.h with its ctypes signature
_P = ctypes.c_void_p
_SIGS = {
    "eagle_build_tree_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(TreeCfg)]),
    "eagle_build_tree": (ctypes.c_int32, [ctypes.POINTER(TreeCfg)] + [_P] * 9 + [ctypes.c_size_t, _P]),
    "eagle_tree_attention_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(AttnCfg)]),
    "eagle_tree_attention": (ctypes.c_int32, [ctypes.POINTER(AttnCfg)] + [_P] * 9 + [ctypes.c_size_t, _P]),
    "eagle_tree_verify_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(VerifyCfg)]),
    "eagle_tree_verify": (ctypes.c_int32, [ctypes.POINTER(VerifyCfg)] + [_P] * 11 + [ctypes.c_size_t, _P]),
    "eagle_tree_verify_static": (ctypes.c_int32, [ctypes.POINTER(VerifyCfg)] + [_P] * 10 + [_P]),
    "eagle_workspace_init": (ctypes.c_int32, [_P, ctypes.c_size_t, _P]),
    "eagle_get_device_status": (ctypes.c_int32, [_P, _P, ctypes.POINTER(ctypes.c_int32)]),
    "eagle_status_string": (ctypes.c_char_p, [ctypes.c_int32]),
    "eagle_last_launch_count": (ctypes.c_int32, []),
    "eagle_selftest_wait_timeout": (ctypes.c_int32, [_P, _P, _P]),
    "eagle_selftest_exp2_error": (ctypes.c_int32, [_P, _P]),
    "eagle_kv_commit_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(AttnCfg)]),
    "eagle_build_static_tree_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(StaticTreeCfg)]),
    "eagle_build_static_tree": (ctypes.c_int32, [ctypes.POINTER(StaticTreeCfg)] + [_P] * 9 + [ctypes.c_size_t, _P]),
    "eagle_kv_commit": (ctypes.c_int32, [ctypes.POINTER(AttnCfg), ctypes.c_int32] + [_P] * 9 + [ctypes.c_size_t, _P]),
    "eagle_build_tree_sampled": (ctypes.c_int32, [ctypes.POINTER(TreeCfg)] + [_P] * 10 + [ctypes.c_size_t, _P]),
    "eagle_build_static_tree_sampled": (ctypes.c_int32,
                                        [ctypes.POINTER(StaticTreeCfg)] + [_P] * 10 + [ctypes.c_size_t, _P]),
    "eagle_build_begin": (ctypes.c_int32, [ctypes.POINTER(TreeCfg), _P, _P, _P, ctypes.c_size_t, _P, _P, _P]),
    "eagle_build_expand": (ctypes.c_int32,
                           [ctypes.POINTER(TreeCfg), ctypes.c_int32, _P, _P, _P, ctypes.c_size_t, _P, _P, _P]),
    "eagle_build_finalize": (ctypes.c_int32, [ctypes.POINTER(TreeCfg), _P, _P, ctypes.c_size_t] + [_P] * 7),
}


def library_path() -> str:
    return _build.LIB


def load(build_if_needed: bool = True):
    """Load libeagle.so (compiling it first when it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build() if build_if_needed else _build.LIB
            if not os.path.exists(path):
                raise ImportError(f"libeagle.so not found at {path}; run eagle_draft_tree_gb300.build")
            lib = ctypes.CDLL(path)
            for name, (res, args) in _SIGS.items():
                f = getattr(lib, name)
                f.restype = res
                f.argtypes = args
            _lib = lib
    return _lib


def _status_string(s: int) -> str:
    try:
        return load().eagle_status_string(int(s)).decode()
    except Exception:  # pragma: no cover
        return "status"


def last_launch_count() -> int:
    """Kernel launches issued by the most recent entry-point call on this thread."""
    return int(load().eagle_last_launch_count())


def selftest_exp2_error(device="cuda", stream=None) -> float:
    """eagle_selftest_exp2_error: the largest relative error of the SFU's 2^f over |f| <= 1/2."""
    out = torch.zeros(1, dtype=torch.float32, device=device)
    _check(load().eagle_selftest_exp2_error(_ptr(out), _stream(stream)), "eagle_selftest_exp2_error")
    return float(out.cpu()[0])


def selftest_wait_timeout(ws: "Workspace", stream=None) -> tuple[int, list[int]]:
    """eagle_selftest_wait_timeout: a warp and a thread each wait on a barrier nothing completes.
    Returns (the device status read back, [ns the warp waited, ns the thread waited])."""
    ws.reserve(256, stream)
    elapsed = torch.zeros(2, dtype=torch.int64, device=ws.device)
    _check(load().eagle_selftest_wait_timeout(ws.ptr, _ptr(elapsed), _stream(stream)),
           "eagle_selftest_wait_timeout")
    st = ws.status(stream)
    return st, [int(x) for x in elapsed.cpu()]


def _check(status: int, what: str) -> None:
    if status != EAGLE_OK:
        raise EagleError(what, status)


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t: torch.Tensor | None) -> ctypes.c_void_p | None:
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _need(t: torch.Tensor, name: str, dtype: torch.dtype, shape: tuple | None = None) -> torch.Tensor:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor (the library has no CPU path)")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


class Workspace:
    """A device workspace (uint8 tensor, 256-byte aligned) zeroed once when (re)allocated."""

    def __init__(self, nbytes: int = 0, device=None):
        self.device = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
        self.buf = None
        self.nbytes = 0
        if nbytes:
            self.reserve(nbytes)

    def reserve(self, nbytes: int, stream=None) -> "Workspace":
        nbytes = max(int(nbytes), 256)
        if nbytes > self.nbytes:
            self.buf = torch.empty(nbytes + 256, dtype=torch.uint8, device=self.device)
            self.nbytes = nbytes
            _check(load().eagle_workspace_init(self.ptr, ctypes.c_size_t(self.nbytes), _stream(stream)),
                   "eagle_workspace_init")
        return self

    @property
    def ptr(self) -> ctypes.c_void_p:
        base = self.buf.data_ptr()
        return ctypes.c_void_p((base + 255) // 256 * 256)

    def status(self, stream=None) -> int:
        """Read and clear the device status word (synchronises the stream)."""
        out = ctypes.c_int32(0)
        _check(load().eagle_get_device_status(self.ptr, _stream(stream), ctypes.byref(out)),
               "eagle_get_device_status")
        return int(out.value)


def device_status(ws: Workspace, stream=None) -> int:
    return ws.status(stream)


def tree_cfg(batch, vocab, depth, topk, keep, tree_temp=1.0) -> TreeCfg:
    return TreeCfg(batch, vocab, depth, topk, keep, float(tree_temp))


def _tree_out(B: int, n: int, dev, with_logv: bool) -> dict:
    out = {k: torch.empty((B, n), dtype=torch.int32, device=dev) for k in ("tokens", "parents", "depths", "node_row")}
    out["mask"] = torch.empty((B, n), dtype=torch.int64, device=dev)
    out["node_logv"] = torch.empty((B, n), dtype=torch.float32, device=dev) if with_logv else None
    return out


def build_tree(draft_logits: torch.Tensor, root_token: torch.Tensor, depth: int, topk: int, keep: int,
               tree_temp: float = 1.0, ws: Workspace | None = None, out: dict | None = None,
               with_logv: bool = True, stream=None, child_u: torch.Tensor | None = None) -> dict:
    """eagle_build_tree: draft logits f32 [B,R,V], root tokens i32 [B] -> the flattened tree
    (tokens, parents, depths, node_row i32 [B,n]; mask int64 [B,n] holding the u64 bit masks;
    node_logv f32 [B,n]).  With child_u f32 [B,R,topk]: eagle_build_tree_sampled (each row's
    children are topk inverse-CDF draws from softmax(x / tree_temp))."""
    lib = load()
    B, R, V = draft_logits.shape
    cfg = tree_cfg(B, V, depth, topk, keep, tree_temp)
    _need(draft_logits, "draft_logits", torch.float32)
    _need(root_token, "root_token", torch.int32, (B,))
    if child_u is not None:
        _need(child_u, "child_u", torch.float32, (B, R, topk))
    n = keep + 1
    dev = draft_logits.device
    if out is None:
        out = _tree_out(B, n, dev, with_logv)
    ws = ws or Workspace(device=dev)
    need = lib.eagle_build_tree_workspace_size(ctypes.byref(cfg))
    if need == 0:
        _check(EAGLE_ERR_UNSUPPORTED if R == 1 + (depth - 1) * topk else EAGLE_ERR_INVALID_ARG, "eagle_build_tree")
    if R != 1 + (depth - 1) * topk:
        raise ValueError(f"draft_logits must have 1 + (depth-1)*topk = {1 + (depth - 1) * topk} rows, got {R}")
    ws.reserve(need, stream)
    tail = (_ptr(root_token), _ptr(out["tokens"]), _ptr(out["parents"]), _ptr(out["depths"]), _ptr(out["node_row"]),
            _ptr(out["mask"]), _ptr(out.get("node_logv")), ws.ptr, ctypes.c_size_t(ws.nbytes), _stream(stream))
    if child_u is None:
        _check(lib.eagle_build_tree(ctypes.byref(cfg), _ptr(draft_logits), *tail), "eagle_build_tree")
    else:
        _check(lib.eagle_build_tree_sampled(ctypes.byref(cfg), _ptr(draft_logits), _ptr(child_u), *tail),
               "eagle_build_tree_sampled")
    return out


class BuildState:
    """The workspace and configuration of one stepwise build (eagle_build_begin / _expand /
    _finalize); the workspace carries the rows' children and the frontiers between the calls."""

    def __init__(self, batch: int, vocab: int, depth: int, topk: int, keep: int, tree_temp: float = 1.0,
                 ws: Workspace | None = None, device=None, stream=None):
        self.cfg = tree_cfg(batch, vocab, depth, topk, keep, tree_temp)
        self.device = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
        need = load().eagle_build_tree_workspace_size(ctypes.byref(self.cfg))
        if need == 0:
            _check(EAGLE_ERR_UNSUPPORTED, "eagle_build_tree_workspace_size")
        self.ws = (ws or Workspace(device=self.device)).reserve(need, stream)
        self.front_tok = torch.empty((batch, topk), dtype=torch.int32, device=self.device)
        self.front_par = torch.empty((batch, topk), dtype=torch.int32, device=self.device)


def _frontier(state: BuildState, written: bool):
    return (state.front_tok, state.front_par) if written else None


def build_begin(state: BuildState, root_logits: torch.Tensor, child_u: torch.Tensor | None = None, stream=None):
    """eagle_build_begin: the root's draft logits f32 [B,V] (child_u f32 [B,1,topk] for sampled
    children) -> the frontier of depth 1 (front_tok, front_par i32 [B,topk]), or None when
    depth == 1.  The returned tensors belong to ``state`` and are overwritten by the next step."""
    c = state.cfg
    _need(root_logits, "root_logits", torch.float32, (c.batch, c.vocab))
    if child_u is not None:
        _need(child_u, "child_u", torch.float32, (c.batch, 1, c.topk))
    st = load().eagle_build_begin(ctypes.byref(c), _ptr(root_logits), _ptr(child_u), state.ws.ptr,
                                  ctypes.c_size_t(state.ws.nbytes), _ptr(state.front_tok), _ptr(state.front_par),
                                  _stream(stream))
    _check(st, "eagle_build_begin")
    return _frontier(state, c.depth >= 2)


def build_expand(state: BuildState, depth: int, frontier_logits: torch.Tensor, child_u: torch.Tensor | None = None,
                 stream=None):
    """eagle_build_expand: the draft logits f32 [B,topk,V] of the depth-``depth`` frontier (slot
    order; child_u f32 [B,topk,topk] for sampled children) -> the frontier of depth + 1, or None
    when depth + 1 is the last depth."""
    c = state.cfg
    _need(frontier_logits, "frontier_logits", torch.float32, (c.batch, c.topk, c.vocab))
    if child_u is not None:
        _need(child_u, "child_u", torch.float32, (c.batch, c.topk, c.topk))
    st = load().eagle_build_expand(ctypes.byref(c), int(depth), _ptr(frontier_logits), _ptr(child_u), state.ws.ptr,
                                   ctypes.c_size_t(state.ws.nbytes), _ptr(state.front_tok), _ptr(state.front_par),
                                   _stream(stream))
    _check(st, "eagle_build_expand")
    return _frontier(state, depth + 1 <= c.depth - 1)


def build_finalize(state: BuildState, root_token: torch.Tensor, out: dict | None = None, with_logv: bool = True,
                   stream=None) -> dict:
    """eagle_build_finalize: the rerank, flatten and masks of the stepwise build -> the same dict
    as build_tree."""
    c = state.cfg
    _need(root_token, "root_token", torch.int32, (c.batch,))
    if out is None:
        out = _tree_out(c.batch, c.keep + 1, state.device, with_logv)
    st = load().eagle_build_finalize(ctypes.byref(c), _ptr(root_token), state.ws.ptr, ctypes.c_size_t(state.ws.nbytes),
                                     _ptr(out["tokens"]), _ptr(out["parents"]), _ptr(out["depths"]),
                                     _ptr(out["node_row"]), _ptr(out["mask"]), _ptr(out.get("node_logv")),
                                     _stream(stream))
    _check(st, "eagle_build_finalize")
    return out


def tree_attention(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, ctx_len: torch.Tensor,
                   k_tree: torch.Tensor, v_tree: torch.Tensor, mask: torch.Tensor, scale: float = 0.0,
                   ws: Workspace | None = None, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """eagle_tree_attention over every layer: q [L,B,n,Hq,d]; k/v_cache [L,B,S_max,Hkv,d];
    k/v_tree [L,B,n,Hkv,d]; ctx_len i32 [B]; mask int64 [B,n] -> out [L,B,n,Hq,d] (dtype of q)."""
    lib = load()
    L, B, n, Hq, d = q.shape
    S_max, Hkv = k_cache.shape[2], k_cache.shape[3]
    dt = q.dtype
    if dt not in (torch.bfloat16, torch.float32):
        raise TypeError("q/K/V must be bfloat16 or float32")
    _need(q, "q", dt)
    _need(k_cache, "k_cache", dt, (L, B, S_max, Hkv, d))
    _need(v_cache, "v_cache", dt, (L, B, S_max, Hkv, d))
    _need(k_tree, "k_tree", dt, (L, B, n, Hkv, d))
    _need(v_tree, "v_tree", dt, (L, B, n, Hkv, d))
    _need(ctx_len, "ctx_len", torch.int32, (B,))
    _need(mask, "mask", torch.int64, (B, n))
    cfg = AttnCfg(B, L, n, Hq, Hkv, d, S_max, EAGLE_DTYPE_BF16 if dt == torch.bfloat16 else EAGLE_DTYPE_F32,
                  float(scale))
    if out is None:
        out = torch.empty_like(q)
    else:
        _need(out, "out", dt, tuple(q.shape))
    ws = ws or Workspace(device=q.device)
    need = lib.eagle_tree_attention_workspace_size(ctypes.byref(cfg))
    if need == 0:
        _check(EAGLE_ERR_UNSUPPORTED, "eagle_tree_attention")
    ws.reserve(need, stream)
    st = lib.eagle_tree_attention(ctypes.byref(cfg), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(ctx_len),
                                  _ptr(k_tree), _ptr(v_tree), _ptr(mask), _ptr(out), ws.ptr,
                                  ctypes.c_size_t(ws.nbytes), _stream(stream))
    _check(st, "eagle_tree_attention")
    return out


def build_static_tree(draft_logits: torch.Tensor, root_token: torch.Tensor, template_parents, tree_temp: float = 1.0,
                      ws: Workspace | None = None, out: dict | None = None, with_logv: bool = True,
                      stream=None, child_u: torch.Tensor | None = None) -> dict:
    """eagle_build_static_tree: a static tree (EAGLE-1) or chain from a template of parent
    indices.  draft_logits f32 [B,R,V] (R = template nodes with children, in index order), root
    tokens i32 [B] -> the same dict as build_tree (n = len(template_parents)).  With child_u f32
    [B,R,kmax] (kmax = the most children of one node): eagle_build_static_tree_sampled."""
    lib = load()
    B, R, V = draft_logits.shape
    cfg = static_tree_cfg(B, V, template_parents, tree_temp)
    n = cfg.nodes
    internal = len({int(p) for p in template_parents[1:]})
    if R != internal:
        raise ValueError(f"draft_logits must have one row per template node with children ({internal}), got {R}")
    _need(draft_logits, "draft_logits", torch.float32)
    _need(root_token, "root_token", torch.int32, (B,))
    if child_u is not None:
        kmax = max([sum(1 for q in template_parents[1:] if int(q) == p) for p in range(n)] + [1])
        _need(child_u, "child_u", torch.float32, (B, R, kmax))
    dev = draft_logits.device
    if out is None:
        out = _tree_out(B, n, dev, with_logv)
    ws = ws or Workspace(device=dev)
    need = lib.eagle_build_static_tree_workspace_size(ctypes.byref(cfg))
    if need == 0:
        _check(EAGLE_ERR_UNSUPPORTED, "eagle_build_static_tree")
    ws.reserve(need, stream)
    tail = (_ptr(root_token), _ptr(out["tokens"]), _ptr(out["parents"]), _ptr(out["depths"]), _ptr(out["node_row"]),
            _ptr(out["mask"]), _ptr(out.get("node_logv")), ws.ptr, ctypes.c_size_t(ws.nbytes), _stream(stream))
    if child_u is None:
        _check(lib.eagle_build_static_tree(ctypes.byref(cfg), _ptr(draft_logits), *tail), "eagle_build_static_tree")
    else:
        _check(lib.eagle_build_static_tree_sampled(ctypes.byref(cfg), _ptr(draft_logits), _ptr(child_u), *tail),
               "eagle_build_static_tree_sampled")
    return out


def kv_commit(k_tree: torch.Tensor, v_tree: torch.Tensor, out_path: torch.Tensor, out_len: torch.Tensor,
              ctx_len: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
              new_ctx_len: torch.Tensor | None = None, ws: Workspace | None = None, stream=None) -> torch.Tensor:
    """eagle_kv_commit: append each sequence's root and accepted path (out_path [B,D], out_len [B]
    from tree_verify) from k/v_tree [L,B,n,Hkv,d] to k/v_cache [L,B,S_max,Hkv,d] in place at
    positions ctx_len[b] ...; returns new_ctx_len i32 [B] = ctx_len + out_len."""
    lib = load()
    L, B, n, Hkv, d = k_tree.shape
    S_max = k_cache.shape[2]
    dt = k_tree.dtype
    if dt not in (torch.bfloat16, torch.float32):
        raise TypeError("K/V must be bfloat16 or float32")
    _need(k_tree, "k_tree", dt)
    _need(v_tree, "v_tree", dt, (L, B, n, Hkv, d))
    _need(k_cache, "k_cache", dt, (L, B, S_max, Hkv, d))
    _need(v_cache, "v_cache", dt, (L, B, S_max, Hkv, d))
    _need(out_path, "out_path", torch.int32)
    _need(out_len, "out_len", torch.int32, (B,))
    _need(ctx_len, "ctx_len", torch.int32, (B,))
    D = out_path.shape[1]
    if out_path.shape != (B, D):
        raise ValueError("out_path must be [B, D]")
    cfg = AttnCfg(B, L, n, Hkv, Hkv, d, S_max, EAGLE_DTYPE_BF16 if dt == torch.bfloat16 else EAGLE_DTYPE_F32, 0.0)
    if new_ctx_len is None:
        new_ctx_len = torch.empty_like(ctx_len)
    else:
        _need(new_ctx_len, "new_ctx_len", torch.int32, (B,))
    ws = ws or Workspace(device=k_tree.device)
    need = lib.eagle_kv_commit_workspace_size(ctypes.byref(cfg))
    if need == 0:
        _check(EAGLE_ERR_UNSUPPORTED, "eagle_kv_commit")
    ws.reserve(need, stream)
    st = lib.eagle_kv_commit(ctypes.byref(cfg), D, _ptr(k_tree), _ptr(v_tree), _ptr(out_path), _ptr(out_len),
                             _ptr(ctx_len), _ptr(k_cache), _ptr(v_cache), _ptr(new_ctx_len), ws.ptr,
                             ctypes.c_size_t(ws.nbytes), _stream(stream))
    _check(st, "eagle_kv_commit")
    return new_ctx_len


def tree_verify(target_logits: torch.Tensor, draft_logits: torch.Tensor, tree: dict, uniforms: torch.Tensor,
                temperature: float, depth: int, topk: int, ws: Workspace | None = None, out: dict | None = None,
                with_ratio: bool = True, stream=None) -> dict:
    """eagle_tree_verify: target f32 [B,n,V], draft f32 [B,R,V], the tree (tokens/parents/node_row
    i32 [B,n]), uniforms f32 [B,n] -> out_tokens i32 [B,D+1], out_len i32 [B], out_path i32 [B,D],
    out_ratio f32 [B,n]."""
    lib = load()
    B, n, V = target_logits.shape
    R = draft_logits.shape[1]
    _need(target_logits, "target_logits", torch.float32)
    _need(draft_logits, "draft_logits", torch.float32, (B, 1 + (depth - 1) * topk, V))
    for key in ("tokens", "parents", "node_row"):
        _need(tree[key], key, torch.int32, (B, n))
    _need(uniforms, "uniforms", torch.float32, (B, n))
    cfg = VerifyCfg(B, V, depth, topk, n - 1, float(temperature))
    dev = target_logits.device
    if out is None:
        out = dict(out_tokens=torch.empty((B, depth + 1), dtype=torch.int32, device=dev),
                   out_len=torch.empty((B,), dtype=torch.int32, device=dev),
                   out_path=torch.empty((B, depth), dtype=torch.int32, device=dev),
                   out_ratio=torch.empty((B, n), dtype=torch.float32, device=dev) if with_ratio else None)
    ws = ws or Workspace(device=dev)
    need = lib.eagle_tree_verify_workspace_size(ctypes.byref(cfg))
    if need == 0:
        _check(EAGLE_ERR_UNSUPPORTED, "eagle_tree_verify")
    ws.reserve(need, stream)
    del R
    st = lib.eagle_tree_verify(ctypes.byref(cfg), _ptr(target_logits), _ptr(draft_logits), _ptr(tree["tokens"]),
                               _ptr(tree["parents"]), _ptr(tree["node_row"]), _ptr(uniforms),
                               _ptr(out["out_tokens"]), _ptr(out["out_len"]), _ptr(out["out_path"]),
                               _ptr(out.get("out_ratio")), ws.ptr, ctypes.c_size_t(ws.nbytes), _stream(stream))
    _check(st, "eagle_tree_verify")
    return out


def tree_verify_static(target_logits: torch.Tensor, draft_logits: torch.Tensor, tree: dict, uniforms: torch.Tensor,
                       temperature: float, depth: int, topk: int, out: dict | None = None, with_ratio: bool = True,
                       stream=None) -> dict:
    """eagle_tree_verify_static: tree_verify with the library's static device scratch instead of a
    caller workspace (same arguments and outputs; up to 256 KB of scratch, e.g. 113 x 64 nodes)."""
    lib = load()
    B, n, V = target_logits.shape
    _need(target_logits, "target_logits", torch.float32)
    _need(draft_logits, "draft_logits", torch.float32, (B, 1 + (depth - 1) * topk, V))
    for key in ("tokens", "parents", "node_row"):
        _need(tree[key], key, torch.int32, (B, n))
    _need(uniforms, "uniforms", torch.float32, (B, n))
    cfg = VerifyCfg(B, V, depth, topk, n - 1, float(temperature))
    dev = target_logits.device
    if out is None:
        out = dict(out_tokens=torch.empty((B, depth + 1), dtype=torch.int32, device=dev),
                   out_len=torch.empty((B,), dtype=torch.int32, device=dev),
                   out_path=torch.empty((B, depth), dtype=torch.int32, device=dev),
                   out_ratio=torch.empty((B, n), dtype=torch.float32, device=dev) if with_ratio else None)
    st = lib.eagle_tree_verify_static(ctypes.byref(cfg), _ptr(target_logits), _ptr(draft_logits),
                                      _ptr(tree["tokens"]), _ptr(tree["parents"]), _ptr(tree["node_row"]),
                                      _ptr(uniforms), _ptr(out["out_tokens"]), _ptr(out["out_len"]),
                                      _ptr(out["out_path"]), _ptr(out.get("out_ratio")), _stream(stream))
    _check(st, "eagle_tree_verify_static")
    return out
