"""Device waits are bounded in time: a wait on a barrier that nothing completes gives up after
about a second, reports EAGLE_ERR_TIMEOUT through the workspace status word, and leaves the
context usable (no fault, trap or hang is involved)."""
import numpy as np
import pytest
import torch

import eagle_draft_tree_gb300 as eg
import oracle
from tests.gpu_parity import ATTN_TOL, np_

pytestmark = pytest.mark.gpu


def test_wait_on_a_barrier_nothing_completes_times_out():
    ws = eg.Workspace(device="cuda")
    status, elapsed = eg.selftest_wait_timeout(ws)
    assert status == eg.EAGLE_ERR_TIMEOUT
    assert eg.last_launch_count() == 1
    for ns in elapsed:  # the warp-wide and the single-thread wait
        assert 0.9e9 <= ns <= 5e9, elapsed
    # the context still works: a small attention call matches the oracle and reports no error
    g = torch.Generator().manual_seed(3)
    L, B, n, Hq, Hkv, d, S = 1, 2, 5, 4, 2, 128, 40
    mk = lambda *s: (torch.randn(*s, generator=g) * 0.5).to(torch.bfloat16).cuda()
    q, kc, vc = mk(L, B, n, Hq, d), mk(L, B, S, Hkv, d), mk(L, B, S, Hkv, d)
    kt, vt = mk(L, B, n, Hkv, d), mk(L, B, n, Hkv, d)
    ctx = torch.tensor([40, 17], dtype=torch.int32, device="cuda")
    mask = torch.tensor([[(1 << (i + 1)) - 1 for i in range(n)]] * B, dtype=torch.int64, device="cuda")
    out = eg.tree_attention(q, kc, vc, ctx, kt, vt, mask, ws=ws)
    assert ws.status() == eg.EAGLE_OK
    ref = oracle.tree_attention(np_(q), np_(kc), np_(vc), np_(ctx), np_(kt), np_(vt),
                                mask.cpu().numpy().view(np.uint64).reshape(B, n, 1))
    assert np.abs(out.float().cpu().numpy().astype(np.float64) - ref).max() <= ATTN_TOL["bf16"]
