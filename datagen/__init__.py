"""Seeded synthetic inputs for the EAGLE draft-tree verify round.

This module is the one thing the CUDA path and the fp64 oracle share: both consume the bytes it
makes.  It holds none of the method's arithmetic (no softmax, no selection, no attention); it
only draws random numbers with ``torch.Generator`` and lays them out in the library's row-major
layouts.  Tensors are drawn on the device they are asked for (CPU for small cases, the GPU for
the multi-GB workloads) and the oracle always receives a CPU copy of the very same bytes.

Workload recipe (each value below is a reading of the workload descriptions, stated once here):
  * draft logits  ~ N(0, 2^2) per entry, then one uniformly drawn token per row gets +6;
  * target row of tree node i = draft row node_row[i] (a fresh draft-like row when the node was
    never expanded) + N(0, sigma^2) noise, sigma per workload (per sequence for the serving mix);
  * q, K, V (cache and tree) ~ N(0, 1), rounded once to the stored dtype;
  * uniforms ~ U(0, 1) in float32 (verify tests and sampled-children draws, separate streams);
    root tokens uniform over the vocabulary;
  * context lengths fixed per workload, or uniform integers in [512, 8192] for the serving mix.
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    batch: int          # B
    vocab: int          # V
    depth: int          # D
    topk: int           # k
    keep: int           # m (kept draft tokens; the root is extra)
    layers: int         # L
    heads_q: int        # Hq
    heads_kv: int       # Hkv
    head_dim: int       # d
    ctx: int            # fixed context length, or the upper bound of the ragged draw
    ctx_min: int        # lower bound of the ragged draw (== ctx for fixed contexts)
    kv_dtype: str       # "f32" or "bf16"
    temperature: float  # verify temperature (0 = greedy)
    noise: float        # target-logit noise sigma (upper bound when noise_min is set)
    noise_min: float | None = None  # per-sequence sigma ~ U(noise_min, noise)

    @property
    def rows(self) -> int:  # R = 1 + (D-1)k draft rows per sequence
        return 1 + (self.depth - 1) * self.topk

    @property
    def pool(self) -> int:  # P = k + (D-1)k^2 candidates per sequence
        return self.topk + (self.depth - 1) * self.topk * self.topk

    @property
    def nodes(self) -> int:  # n = m + 1 (root first)
        return self.keep + 1

    @property
    def group(self) -> int:  # G = Hq / Hkv
        return self.heads_q // self.heads_kv

    @property
    def max_seq(self) -> int:  # S_max of the cache layout
        return self.ctx

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads (sizes as the workload descriptions give them).
WORKLOADS = {
    "tiny_f32": Workload("tiny_f32", 1, 1000, 3, 4, 10, 1, 4, 2, 64, 128, 128, "f32", 1.0, 0.5),
    "llama31_8b": Workload("llama31_8b", 1, 128256, 8, 10, 60, 32, 32, 8, 128, 2048, 2048, "bf16", 1.0, 0.5),
    "vicuna_13b": Workload("vicuna_13b", 1, 32000, 6, 10, 50, 40, 40, 40, 128, 4096, 4096, "bf16", 1.0, 1.0),
    "llama2_70b_b4": Workload("llama2_70b_b4", 4, 32000, 6, 10, 48, 80, 64, 8, 128, 8192, 8192, "bf16", 1.0, 0.5),
    "serving_b64": Workload("serving_b64", 64, 128256, 8, 10, 60, 32, 32, 8, 128, 8192, 512, "bf16", 0.7, 1.5, 0.2),
}
WORKLOAD_ORDER = ["tiny_f32", "llama31_8b", "vicuna_13b", "llama2_70b_b4", "serving_b64"]

# Per-tensor stream offsets so every tensor of a seed has its own generator stream.
_S_DRAFT, _S_PLANT, _S_ROOT, _S_TGT, _S_TPLANT, _S_TNOISE, _S_SIG = 11, 12, 13, 21, 22, 23, 24
_S_Q, _S_KC, _S_VC, _S_KT, _S_VT, _S_CTX, _S_U = 31, 32, 33, 34, 35, 36, 41
_S_CU = 43


def _gen(seed: int, stream: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((int(seed) * 1_000_003 + stream * 7919) % (2**63 - 1))
    return g


def _dev(device) -> torch.device:
    return torch.device(device)


def draft_logits(batch: int, rows: int, vocab: int, seed: int, device="cpu", sigma: float = 2.0,
                 plant: float = 6.0) -> torch.Tensor:
    """float32 [B, R, V]: N(0, sigma^2) with +plant added to one uniformly drawn token per row."""
    dev = _dev(device)
    x = torch.randn((batch, rows, vocab), generator=_gen(seed, _S_DRAFT, dev), device=dev, dtype=torch.float32)
    x.mul_(sigma)
    tok = torch.randint(0, vocab, (batch, rows, 1), generator=_gen(seed, _S_PLANT, dev), device=dev)
    x.scatter_add_(2, tok, torch.full((batch, rows, 1), plant, device=dev, dtype=torch.float32))
    return x


def root_tokens(batch: int, vocab: int, seed: int, device="cpu") -> torch.Tensor:
    dev = _dev(device)
    return torch.randint(0, vocab, (batch,), generator=_gen(seed, _S_ROOT, dev), device=dev, dtype=torch.int32)


def noise_sigmas(wl: Workload, seed: int) -> torch.Tensor:
    """float64 [B] per-sequence target noise sigma (constant unless the workload draws it)."""
    if wl.noise_min is None:
        return torch.full((wl.batch,), float(wl.noise), dtype=torch.float64)
    u = torch.rand((wl.batch,), generator=_gen(seed, _S_SIG, torch.device("cpu")), dtype=torch.float64)
    return wl.noise_min + (wl.noise - wl.noise_min) * u


def target_logits(draft: torch.Tensor, node_row: torch.Tensor, sigmas, seed: int, sigma: float = 2.0,
                  plant: float = 6.0) -> torch.Tensor:
    """float32 [B, n, V]: target row i = draft row node_row[i] + N(0, sigma_b^2); a node with no draft
    row (node_row = -1) starts from a fresh draft-like row.  ``node_row`` is the tree's own output,
    so this is called once the tree of the round is known (outside any timed region)."""
    dev = draft.device
    B, R, V = draft.shape
    rows = node_row.to(device=dev, dtype=torch.int64)
    n = rows.shape[1]
    fresh = torch.randn((B, n, V), generator=_gen(seed, _S_TGT, dev), device=dev, dtype=torch.float32).mul_(sigma)
    ptok = torch.randint(0, V, (B, n, 1), generator=_gen(seed, _S_TPLANT, dev), device=dev)
    fresh.scatter_add_(2, ptok, torch.full((B, n, 1), plant, device=dev, dtype=torch.float32))
    base = torch.gather(draft, 1, rows.clamp(min=0).unsqueeze(-1).expand(B, n, V))
    use_draft = (rows >= 0).unsqueeze(-1)
    out = torch.where(use_draft, base, fresh)
    del fresh, base
    noise = torch.randn((B, n, V), generator=_gen(seed, _S_TNOISE, dev), device=dev, dtype=torch.float32)
    sig = torch.as_tensor(sigmas, dtype=torch.float32, device=dev).reshape(-1, 1, 1).expand(B, 1, 1)
    out.addcmul_(noise, sig)
    return out


def uniforms(batch: int, nodes: int, seed: int, device="cpu") -> torch.Tensor:
    """float32 [B, n] in [0, 1): u[:, 0] draws the final token, u[:, i] tests node i."""
    dev = _dev(device)
    return torch.rand((batch, nodes), generator=_gen(seed, _S_U, dev), device=dev, dtype=torch.float32)


def child_uniforms(batch: int, rows: int, topk: int, seed: int, device="cpu") -> torch.Tensor:
    """float32 [B, R, k] in [0, 1): the draws of sampled children, one per (row, child)."""
    dev = _dev(device)
    return torch.rand((batch, rows, topk), generator=_gen(seed, _S_CU, dev), device=dev, dtype=torch.float32)


def ctx_lens(wl: Workload, seed: int) -> torch.Tensor:
    """int32 [B] context lengths (CPU)."""
    if wl.ctx_min == wl.ctx:
        return torch.full((wl.batch,), wl.ctx, dtype=torch.int32)
    g = _gen(seed, _S_CTX, torch.device("cpu"))
    return torch.randint(wl.ctx_min, wl.ctx + 1, (wl.batch,), generator=g, dtype=torch.int32)


def attention_inputs(wl: Workload, seed: int, device="cpu", layers: int | None = None) -> dict:
    """q [L,B,n,Hq,d]; k_cache, v_cache [L,B,S_max,Hkv,d]; k_tree, v_tree [L,B,n,Hkv,d]; all N(0,1)
    in the workload's dtype.  Positions at or beyond a sequence's context length are drawn too
    (they must never be read)."""
    dev = _dev(device)
    L = wl.layers if layers is None else layers
    dt = torch.float32 if wl.kv_dtype == "f32" else torch.bfloat16
    B, n, Hq, Hkv, d, S = wl.batch, wl.nodes, wl.heads_q, wl.heads_kv, wl.head_dim, wl.max_seq

    def rn(shape, stream):
        return torch.randn(shape, generator=_gen(seed, stream, dev), device=dev, dtype=dt)

    return dict(
        q=rn((L, B, n, Hq, d), _S_Q),
        k_cache=rn((L, B, S, Hkv, d), _S_KC),
        v_cache=rn((L, B, S, Hkv, d), _S_VC),
        k_tree=rn((L, B, n, Hkv, d), _S_KT),
        v_tree=rn((L, B, n, Hkv, d), _S_VT),
        ctx_len=ctx_lens(wl, seed).to(dev),
    )


def to_numpy(t: torch.Tensor):
    """CPU numpy view of a tensor; bf16 becomes its uint16 bit pattern."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view("uint16")
    return t.numpy()


def bytes_of(wl: Workload, ctx_total: int | None = None) -> dict:
    """Algorithmic HBM bytes of one round (each input read once, each output written once)."""
    es = 4 if wl.kv_dtype == "f32" else 2
    B, n, L, Hq, Hkv, d, V, R = wl.batch, wl.nodes, wl.layers, wl.heads_q, wl.heads_kv, wl.head_dim, wl.vocab, wl.rows
    if ctx_total is None:
        ctx_total = B * (wl.ctx if wl.ctx_min == wl.ctx else (wl.ctx + wl.ctx_min) / 2)
    kv = 2 * L * ctx_total * Hkv * d * es
    tree_kv = 2 * L * B * n * Hkv * d * es
    qo = 2 * L * B * n * Hq * d * es
    logits = B * (n + R) * V * 4
    metric = kv + 2 * B * wl.keep * V * 4
    return dict(kv=kv, tree_kv=tree_kv, q_out=qo, logits=logits, attention=kv + tree_kv + qo,
                exact=kv + tree_kv + qo + logits, metric=metric)


def attention_flops(wl: Workload, ctx_total: float | None = None) -> float:
    """2 flops per multiply-add of QK^T and PV over the context keys (tree keys are negligible)."""
    if ctx_total is None:
        ctx_total = wl.batch * (wl.ctx if wl.ctx_min == wl.ctx else (wl.ctx + wl.ctx_min) / 2)
    return 4.0 * wl.layers * wl.heads_q * wl.nodes * wl.head_dim * ctx_total


def scale_of(wl: Workload) -> float:
    return 1.0 / math.sqrt(wl.head_dim)
