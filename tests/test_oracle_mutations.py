"""The pins have teeth: plant a plausible mistake in a private copy of the oracle's C source,
compile it, and check that a pin rejects the mutant.  The real oracle is never modified."""
import os
import tempfile

import numpy as np
import pytest
from scipy.special import softmax
from scipy.stats import chisquare

import oracle
from tests.test_oracle_attention import _inputs, _mask_from_parents, _sdpa
from tests.test_oracle_build import _brute_force_tree
from tests.test_oracle_kv_commit import commit_matches_golden
from tests.test_oracle_sampled_children import frontier_consistent, sampled_matches_golden
from tests.test_oracle_static_tree import static_invariants_hold, static_matches_golden
from tests.test_oracle_verify import _iid_trials, _logits

SRC = os.path.join(os.path.dirname(oracle.__file__), "eagle_oracle.c")


def _mutant(old: str, new: str, tmpdir: str) -> oracle.Oracle:
    text = open(SRC).read()
    assert text.count(old) == 1, f"mutation anchor not unique: {old!r}"
    src = os.path.join(tmpdir, "mutant.c")
    with open(src, "w") as f:
        f.write(text.replace(old, new))
    return oracle.Oracle(oracle.compile_source(src, os.path.join(tmpdir, "libmutant.so")))


def _chi_square_pvalue(orc):
    V, trials = 16, 200_000
    rng = np.random.default_rng(77)
    p, q = rng.dirichlet(np.ones(V)), rng.dirichlet(np.ones(V))
    p2 = rng.dirichlet(np.ones(V), size=V)
    first, _, _ = _iid_trials(rng, p, q, p2, 2, trials, orc=orc)
    pe = softmax(_logits(p).astype(np.float64))
    obs = np.bincount(first, minlength=V)
    return chisquare(obs, pe * obs.sum()).pvalue


def _build_matches_brute_force(orc):
    for seed in range(8):
        rng = np.random.default_rng(seed)
        D, k, V = 3, 3, 8
        m = 7
        x = rng.normal(0, 2, (1, 1 + (D - 1) * k, V)).astype(np.float32)
        try:
            o = orc.build_tree(x, [0], D, k, m)
        except oracle.OracleError:  # the ancestor-closure check fired
            return False
        _, kept = _brute_force_tree(x[0], D, k, m)
        got = set()
        for i in range(1, m + 1):
            path, j = [], i
            while j > 0:
                path.append(int(o["tokens"][0, j]))
                j = o["parents"][0, j]
            got.add(tuple(reversed(path)))
        if got != {c["path"] for c in kept}:
            return False
        # V = product of softmax confidences along the path
        probs = {r: softmax(x[0, r].astype(np.float64)) for r in range(x.shape[1])}
        for i in range(1, m + 1):
            prod, j = 1.0, i
            while j > 0:
                prod *= probs[o["node_row"][0, o["parents"][0, j]]][o["tokens"][0, j]]
                j = o["parents"][0, j]
            if not np.isclose(np.exp(o["node_logv"][0, i]), prod, rtol=1e-10):
                return False
    return True


def _chain_matches_causal(orc):
    rng = np.random.default_rng(3)
    L, B, n, Hkv, G, d, S = 1, 1, 5, 2, 2, 8, 6
    Hq = Hkv * G
    q, kc, vc, cl, kt, vt = _inputs(rng, L, B, n, Hq, Hkv, d, S, [6])
    mask = _mask_from_parents([-1, 0, 1, 2, 3])[None]
    out = orc.tree_attention(q, kc, vc, cl, kt, vt, mask, scale=0.25)
    k_all = np.concatenate([kc[0, 0], kt[0, 0]], 0).astype(np.float64)
    v_all = np.concatenate([vc[0, 0], vt[0, 0]], 0).astype(np.float64)
    allowed = np.ones((n, S + n), bool)
    allowed[:, S:] = np.tril(np.ones((n, n), bool))
    ref = _sdpa(q[0, 0].astype(np.float64).transpose(1, 0, 2), np.repeat(k_all.transpose(1, 0, 2), G, 0),
                np.repeat(v_all.transpose(1, 0, 2), G, 0), allowed, 0.25).transpose(1, 0, 2)
    return np.allclose(out[0, 0], ref, rtol=1e-10, atol=1e-12)


MUTANTS = {
    # verification: resample from p itself instead of the residual after a rejection
    "residual_not_adjusted": ("tmp[t] = p[t] - q[t] > 0.0 ? p[t] - q[t] : 0.0;", "tmp[t] = p[t];", "verify"),
    # verification: the adjusted distribution also removes q's mass where p < q (no clipping)
    "residual_not_clipped": ("tmp[t] = p[t] - q[t] > 0.0 ? p[t] - q[t] : 0.0;", "tmp[t] = fabs(p[t] - q[t]);", "verify"),
    # verification: ratio inverted
    "ratio_inverted": ("if (q[t] > 0.0) return p[t] / q[t];", "if (p[t] > 0.0) return q[t] / p[t];", "verify"),
    # build: frontier slots read the draft rows in reverse order
    "frontier_rows_reversed": ("par->row = 1 + (f - 1) * k + s;", "par->row = 1 + (f - 1) * k + (nf - 1 - s);", "build"),
    # build: value of a child forgets its parent's value
    "value_not_cumulative": ("c->logv = par->logv + ((double)row[kids[r]] / Tt - lse);",
                             "c->logv = ((double)row[kids[r]] / Tt - lse);", "build"),
    # build: confidence without normalisation (raw logit)
    "confidence_unnormalised": ("c->logv = par->logv + ((double)row[kids[r]] / Tt - lse);",
                                "c->logv = par->logv + ((double)row[kids[r]] / Tt);", "build"),
    # attention: GQA head mapping wrong (interleaved instead of grouped)
    "gqa_interleaved": ("const int g = h / G;", "const int g = h % a->Hkv;", "attention"),
    # attention: a node does not see itself
    "no_self": ("if (!((mrow[j / 64] >> (j % 64)) & 1ull)) continue;\n        size_t koff",
                "if (!((mrow[j / 64] >> (j % 64)) & 1ull) || j == i) continue;\n        size_t koff", "attention"),
    # static tree: siblings take the ranks in reverse order
    "static_rank_reversed": ("tok[i] = top[p][rank];", "tok[i] = top[p][kids[p] - 1 - rank];", "static"),
    # static tree: a child reads its own row instead of its parent's
    "static_own_row": ("const float *row = draft + ((size_t)b * R + row_of[p]) * V;\n            tok[i]",
                       "const float *row = draft + ((size_t)b * R + (row_of[i] >= 0 ? row_of[i] : row_of[p])) * V;\n            tok[i]",
                       "static"),
    # static tree: log V not cumulative along the path
    "static_value_not_cumulative": ("lv[i] = lv[p] + ((double)row[tok[i]] / tree_temp - lse[p]);",
                                    "lv[i] = ((double)row[tok[i]] / tree_temp - lse[p]);", "static"),
    # KV commit: the root is not appended (the path starts at position ctx)
    "commit_skips_root": ("const int node = i == 0 ? 0 : out_path[(size_t)b * D + i - 1];",
                          "const int node = i == len - 1 ? 0 : out_path[(size_t)b * D + i];", "commit"),
    # KV commit: rows written one position late
    "commit_position_shifted": ("const size_t dst = (((size_t)l * B + b) * S_max + ctx + i) * row;",
                                "const size_t dst = (((size_t)l * B + b) * S_max + ctx + i + 1) * row;", "commit"),
    # KV commit: the new length leaves out the root
    "commit_length_short": ("new_ctx_len[b] = ctx + len;", "new_ctx_len[b] = ctx + len - 1;", "commit"),
    # KV commit: keys taken from the tree's values
    "commit_k_from_v": ("memcpy((char *)k_cache + dst, (const char *)k_tree + src, row);",
                        "memcpy((char *)k_cache + dst, (const char *)v_tree + src, row);", "commit"),
    # sampled children: q formed without the tree temperature
    "sample_ignores_temperature": ("q_buf[t] = exp((double)x[t] / T - lse);", "q_buf[t] = exp((double)x[t] - lse);",
                                   "sampled"),
    # sampled children: draws take the uniforms in reverse order
    "sample_draw_order_reversed": ("out[j] = inverse_cdf(q_buf, V, (double)u[j], &g);",
                                   "out[j] = inverse_cdf(q_buf, V, (double)u[k - 1 - j], &g);", "sampled"),
    # sampled children: a drawn token cannot come up again (without replacement, unnormalised)
    "sample_without_replacement": ("        if (g < *gap) *gap = g;\n    }\n}\n\n/* A row's k children",
                                   "        if (g < *gap) *gap = g;\n        q_buf[out[j]] = 0.0;\n    }\n}\n\n/* A row's k children",
                                   "sampled"),
    # sampled children: the CDF walked from the top (1 - u)
    "sample_cdf_from_top": ("out[j] = inverse_cdf(q_buf, V, (double)u[j], &g);",
                            "out[j] = inverse_cdf(q_buf, V, 1.0 - (double)u[j], &g);", "sampled"),
    # frontier outputs: parent slot off by one
    "frontier_parent_slot_shifted": ("pool[order[s]->parent].row - 1 - (f - 2) * k;",
                                     "pool[order[s]->parent].row - (f - 2) * k;", "sampled"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_mutant(name):
    old, new, part = MUTANTS[name]
    with tempfile.TemporaryDirectory() as td:
        orc = _mutant(old, new, td)
        if part == "verify":
            assert _chi_square_pvalue(orc) < 1e-6
        elif part == "build":
            assert not _build_matches_brute_force(orc)
        elif part == "commit":
            assert not commit_matches_golden(orc)
        elif part == "sampled":
            assert not (sampled_matches_golden(orc) and frontier_consistent(orc))
        elif part == "static":
            assert not (static_matches_golden(orc) and static_invariants_hold(orc))
        else:
            assert not _chain_matches_causal(orc)


def test_pins_accept_real_oracle():
    assert _chi_square_pvalue(oracle) > 1e-3
    assert _build_matches_brute_force(oracle)
    assert _chain_matches_causal(oracle)
    assert commit_matches_golden(oracle)
    assert static_matches_golden(oracle) and static_invariants_hold(oracle)
    assert sampled_matches_golden(oracle) and frontier_consistent(oracle)
