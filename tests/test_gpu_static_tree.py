"""GPU parity of eagle_build_static_tree against the oracle: chains, random templates (up to 64
nodes, up to 16 children a node), a wide root, the root alone; indices bit-exact, log V to 1e-5
relative; a root token out of range is flagged on the device."""
import numpy as np
import pytest
import torch

import datagen
import eagle_draft_tree_gb300 as eg
import oracle
from tests.gpu_parity import np_
from tests.test_oracle_static_tree import random_template

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _compare(template, B, V, T, seed):
    internal = len(set(template[1:]))
    draft = datagen.draft_logits(B, max(internal, 1), V, seed, DEV)[:, :internal].contiguous()
    root = datagen.root_tokens(B, V, seed, DEV)
    ws = eg.Workspace(device=DEV)
    g = eg.build_static_tree(draft, root, template, T, ws=ws)
    assert ws.status() == eg.EAGLE_OK
    o = oracle.build_static_tree(np_(draft), np_(root), template, T)
    for k in ("tokens", "parents", "depths", "node_row"):
        assert np.array_equal(np_(g[k]), o[k]), k
    assert np.array_equal(np_(g["mask"]).view(np.uint64), o["mask"][:, :, 0])
    np.testing.assert_allclose(np_(g["node_logv"]).astype(np.float64), o["node_logv"], rtol=1e-5, atol=1e-6)


@pytest.mark.parametrize("D", [1, 5, 8])
@pytest.mark.parametrize("T", [1.0, 0.7])
def test_chain_matches_oracle(D, T):
    _compare(eg.chain_template(D), 3, 128256, T, 10 + D)


@pytest.mark.parametrize("seed", range(6))
def test_random_templates_match_oracle(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(2, 65))
    _compare(random_template(rng, n), int(rng.integers(1, 5)), int(rng.choice([100, 5000, 32000])), 1.0, seed)


def test_wide_root_and_root_alone():
    _compare([-1] + [0] * 16, 2, 1000, 1.0, 3)  # 16 children of the root
    _compare([-1], 2, 1000, 1.0, 4)             # no draft row at all


def test_bad_root_token_sets_status():
    draft = datagen.draft_logits(2, 1, 100, 1, DEV)
    root = torch.tensor([5, 100], dtype=torch.int32, device=DEV)
    ws = eg.Workspace(device=DEV)
    eg.build_static_tree(draft, root, [-1, 0, 0], 1.0, ws=ws)
    assert ws.status() == eg.EAGLE_ERR_DEVICE_INPUT
