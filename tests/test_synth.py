"""The seeded input recipe: workload shapes, paged K/V layout, tree and token
generators.  These are the properties the benchmark's and the parity tests'
inputs are stated to have; the tests keep them from drifting."""
import numpy as np
import torch

from eagle_speculative_decoding_gb300 import synth


def test_workload_shapes():
    c = synth.CONFIGS
    for name in ("llama8b", "serve64", "long4", "chain3"):
        assert (c[name]["d"], c[name]["Hq"], c[name]["Hkv"], c[name]["D"], c[name]["V"]) == (4096, 32, 8, 128, 128256)
    assert (c["llama70b"]["d"], c["llama70b"]["Hq"], c["llama70b"]["Hkv"]) == (8192, 64, 8)
    assert c["llama8b"]["B"] == 1 and c["llama8b"]["N"] == 60 and c["llama8b"]["ctx"] == (2048, 2048)
    assert c["serve64"]["B"] == 64 and c["serve64"]["ctx"] == (1024, 4096)
    assert c["long4"]["B"] == 4 and c["long4"]["ctx"] == (32768, 32768)
    assert c["chain3"]["topk"] == 1 and c["chain3"]["width"] == 1 and c["chain3"]["N"] == 3
    for name, cfg in c.items():
        # a tree of N nodes fits the u64 ancestry mask with the root
        assert cfg["N"] + 1 <= 64, name
        # the budget is reachable: enough candidates are drafted
        assert synth.n_candidates(cfg) >= cfg["N"], name
    assert synth.FFN_WIDTH[4096] == 14336 and synth.FFN_WIDTH[8192] == 28672


def test_context_lengths_fixed_or_uniform_in_range():
    g = synth.generator(3)
    fixed = synth.ctx_lengths(synth.CONFIGS["long4"], g)
    assert fixed.tolist() == [32768] * 4
    ctx = synth.ctx_lengths(dict(synth.CONFIGS["serve64"], B=4096), g)
    assert int(ctx.min()) >= 1024 and int(ctx.max()) <= 4096
    # roughly uniform: both quarters of the range are populated
    assert int((ctx < 1024 + 768).sum()) > 600 and int((ctx > 4096 - 768).sum()) > 600


def test_paged_kv_table_is_a_scattered_permutation():
    g = synth.generator(5)
    ctx = [37, 16, 100, 1]
    kc, vc, table = synth.paged_kv(ctx, 2, 8, 16, torch.float32, g)
    npages = [(c + 15) // 16 for c in ctx]
    P = sum(npages) + 3
    assert kc.shape == vc.shape == (P, 16, 2, 8)
    assert table.shape == (4, max(npages))
    used = []
    for b, n in enumerate(npages):
        row = table[b].tolist()
        assert all(0 <= p < P for p in row[:n])
        assert all(p == -1 for p in row[n:])
        used += row[:n]
    assert len(set(used)) == len(used) == sum(npages)  # no page shared
    assert used != sorted(used)  # logical pages are scattered over the pool


def test_tree_generators():
    g = synth.generator(7)
    parent, depth = synth.random_tree(40, 3, g)
    assert int(parent[0]) == -1 and depth[0] == 0
    for i in range(1, 40):
        p = int(parent[i])
        assert 0 <= p < i and depth[i] == depth[p] + 1 and depth[i] <= 4
    assert synth.chain_tree(5).tolist() == [-1, 0, 1, 2, 3]
    tok = synth.distinct_sibling_tokens(parent, 50, g)
    for p in set(parent.tolist()):
        sib = [int(tok[i]) for i in range(40) if int(parent[i]) == p]
        assert len(sib) == len(set(sib))
    t = synth.random_tokens((1000,), 17, g)
    assert int(t.min()) >= 0 and int(t.max()) < 17


def test_logits_and_candidates():
    g = synth.generator(9)
    z = synth.target_logits((50, 300), g, min_top2_gap=1e-2)
    top2 = torch.topk(z, 2, dim=1).values
    assert bool(((top2[:, 0] - top2[:, 1]) > 1e-2).all())
    assert abs(float(z.std()) - synth.LOGIT_STD) < 0.1
    ids, lps = synth.draft_candidates(6, 5, 200, g)
    for j in range(6):
        assert len(set(ids[j].tolist())) == 5
        assert bool((lps[j][:-1] >= lps[j][1:]).all())  # sorted descending
        assert float(torch.logsumexp(lps[j], 0)) <= 1e-6  # a sub-distribution
    w = synth.normal((400, 400), synth.WEIGHT_STD, torch.float32, g)
    assert abs(float(w.std()) - 0.02) < 1e-3
    assert np.isclose(float(synth.normal((10,), 1.0, torch.bfloat16, synth.generator(1)).float()[0]),
                      float(synth.normal((10,), 1.0, torch.bfloat16, synth.generator(1)).float()[0]))
