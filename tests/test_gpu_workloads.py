"""The five workloads at full size, through the C ABI in the benchmark's launch configuration:
every tree index and committed token against the oracle, attention on sampled rows (each row's
oracle value computed from its own slice of the inputs) and on whole (layer, sequence, KV head)
units: every node and query head of the unit against its own fp64 evaluation."""
import numpy as np
import pytest
import torch

import datagen
import eagle_draft_tree_gb300 as eg
import oracle
from tests.gpu_parity import (ATTN_TOL, attention_sample_rows, compare_build, compare_verify, gpu_build, np_,
                              oracle_attention_rows, oracle_attention_unit, oracle_tree_tensors, whole_units)

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("name", datagen.WORKLOAD_ORDER)
def test_workload_round(name):
    wl = datagen.WORKLOADS[name]
    seed = datagen.WORKLOAD_ORDER.index(name)
    ws = eg.Workspace()
    draft = datagen.draft_logits(wl.batch, wl.rows, wl.vocab, seed, DEV)
    root = datagen.root_tokens(wl.batch, wl.vocab, seed, DEV)

    # build: bit-exact trees
    g = gpu_build(draft, root, wl, ws)
    draft_np = np_(draft)
    o_tree = oracle.build_tree(draft_np, np_(root), wl.depth, wl.topk, wl.keep)
    log = []
    compare_build(g, o_tree, log)
    assert len(log) <= max(1, wl.batch // 16), log
    assert ws.status() == eg.EAGLE_OK

    # verify at the workload's temperature (and greedy for the 8B shape)
    target = datagen.target_logits(draft, torch.from_numpy(o_tree["node_row"]).to(DEV),
                                   datagen.noise_sigmas(wl, seed), seed)
    u = datagen.uniforms(wl.batch, wl.nodes, seed, DEV)
    tree = oracle_tree_tensors(o_tree, DEV)
    target_np, u_np = np_(target), np_(u)
    # (with every ratio requested, and without, as the benchmark calls it)
    for T in ([wl.temperature, 0.0] if name == "llama31_8b" else [wl.temperature]):
        ov = oracle.tree_verify(target_np, draft_np, o_tree["tokens"], o_tree["parents"], o_tree["node_row"], u_np,
                                T, wl.depth + 1)
        ov["parents"] = o_tree["parents"]
        for with_ratio in (True, False):
            gv = eg.tree_verify(target, draft, tree, u, temperature=T, depth=wl.depth, topk=wl.topk, ws=ws,
                                with_ratio=with_ratio)
            torch.cuda.synchronize()
            gv = {k: np_(v) for k, v in gv.items() if v is not None}
            vlog = []
            compare_verify(gv, ov, vlog)
            assert len(vlog) <= max(1, wl.batch // 16), vlog
            assert ws.status() == eg.EAGLE_OK
    del target, target_np

    # attention over every layer at full size; oracle on sampled rows
    inp = datagen.attention_inputs(wl, seed, DEV)
    out = eg.tree_attention(inp["q"], inp["k_cache"], inp["v_cache"], inp["ctx_len"], inp["k_tree"],
                            inp["v_tree"], tree["mask"], ws=ws)
    torch.cuda.synchronize()
    assert ws.status() == eg.EAGLE_OK
    rng = np.random.default_rng(seed)
    rows = attention_sample_rows(wl, rng, 40)
    inp["ctx_len"] = inp["ctx_len"].cpu()
    ref = oracle_attention_rows(inp, o_tree["mask"], rows, wl.group, datagen.scale_of(wl))
    got = np.stack([out[l, b, i, h].double().cpu().numpy() for (l, b, i, h) in rows])
    err = np.abs(got - ref).max()
    assert err <= ATTN_TOL[wl.kv_dtype], err
    assert torch.isfinite(out).all()
    # whole units, element by element
    G = wl.group
    for (l, b, g) in whole_units(wl, inp["ctx_len"]):
        ref_u = oracle_attention_unit(inp, o_tree["mask"], l, b, g, G, datagen.scale_of(wl))
        got_u = out[l, b, :, g * G:(g + 1) * G].double().cpu().numpy()
        err_u = np.abs(got_u - ref_u).max()
        assert err_u <= ATTN_TOL[wl.kv_dtype], ((l, b, g), err_u)
