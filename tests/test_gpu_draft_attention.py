"""Tree attention at a draft model's shape: one decoder layer, one sequence, the tree growing by
k nodes per draft step (n = 1, 1 + k, 1 + 2k, ...).  These shapes fill only a few SMs per unit,
so the tensor-core kernel shares each unit's context among several CTAs and merges their
partial results; every output element is compared with the oracle."""
import numpy as np
import pytest
import torch

import datagen
import eagle_draft_tree_gb300 as eg
import oracle
from tests.gpu_parity import ATTN_TOL, np_

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _chain_of_steps_mask(n, k, rng):
    """Ancestor-or-self masks of a tree grown by k children of an earlier node per step."""
    parents = [-1]
    while len(parents) < n:
        base = len(parents)
        for _ in range(min(k, n - base)):
            parents.append(int(rng.integers(0, base)))
    masks = np.zeros(n, np.uint64)
    for i in range(n):
        m, j = 0, i
        while j >= 0:
            m |= 1 << j
            j = parents[j]
        masks[i] = np.uint64(m)
    return masks


@pytest.mark.parametrize("n", [1, 11, 21, 41, 61])
@pytest.mark.parametrize("ctx,S", [(0, 2112), (5, 2112), (300, 364), (1000, 1064), (2048, 2112)],
                         ids=["ctx0-empty-splits", "ctx5-empty-splits", "ctx300-unsplit", "ctx1000", "ctx2048"])
def test_draft_shape_attention_matches_oracle(n, ctx, S):
    """S_max sets the split count; a context much shorter than S_max leaves splits with no tile."""
    Hq, Hkv, d, k = 32, 8, 128, 10
    rng = np.random.default_rng(n * 1000 + ctx)
    g = torch.Generator().manual_seed(n * 7 + ctx)
    mk = lambda *s: torch.randn(*s, generator=g).to(torch.bfloat16).to(DEV)  # noqa: E731
    q, kc, vc = mk(1, 1, n, Hq, d), mk(1, 1, S, Hkv, d), mk(1, 1, S, Hkv, d)
    kt, vt = mk(1, 1, n, Hkv, d), mk(1, 1, n, Hkv, d)
    ctx_t = torch.tensor([ctx], dtype=torch.int32, device=DEV)
    masks = _chain_of_steps_mask(n, k, rng)
    mask_t = torch.from_numpy(masks.view(np.int64).reshape(1, n)).to(DEV)
    ws = eg.Workspace(device=DEV)
    out = eg.tree_attention(q, kc, vc, ctx_t, kt, vt, mask_t, ws=ws)
    assert ws.status() == eg.EAGLE_OK
    ref = oracle.tree_attention(np_(q), np_(kc), np_(vc), np_(ctx_t), np_(kt), np_(vt), masks.reshape(1, n, 1))
    got = out.float().cpu().numpy().astype(np.float64)
    assert np.abs(got - ref).max() <= ATTN_TOL["bf16"]
