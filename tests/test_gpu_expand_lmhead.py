"""GPU parity of eagle_tree_expand_lmhead: the EAGLE-2 expansion step fed
straight from the LM head's per-CTA partial results ("M7.5" 0x06A, 0x06B;
"EAGLE" "Tree-Structured Draft Generation").

Each depth runs, on the same drafter rows and LM-head weights:
  fused    eagle_lmhead_topk_partial -> eagle_tree_expand_lmhead
  unfused  eagle_lmhead_topk (partial + merge) -> eagle_tree_expand
  oracle   tree_expand_step on the unfused path's candidate lists
The fused tree state must equal the unfused one bit for bit after every
depth, and both the oracle's; the unfused lists themselves must equal the
oracle's LM head (ids exact away from near-ties, log-probs to 1e-3).
"""
import numpy as np
import pytest
import torch

import oracle
from eagle_speculative_decoding_gb300 import synth
from gpu_helpers import check_topk, need_gpu

pytestmark = pytest.mark.gpu


def _state(b, B, width, max_nodes, roots):
    z = lambda *s, dt=torch.int32: torch.zeros(s, dtype=dt, device="cuda")
    return dict(parent=z(B, max_nodes), token=z(B, max_nodes), logv=z(B, max_nodes, dt=torch.float32),
                depth=z(B, max_nodes), count=z(B), frontier=z(B, width), nf=z(B), root=roots.cuda(), status=z(1))


@pytest.mark.parametrize("cfg,V,d", [("llama8b", 128256, 4096), ("serve64", 128256, 4096),
                                     ("long4", 32000, 4096), ("toy", 1024, 256)])
def test_fused_expansion_matches_unfused_and_oracle(cfg, V, d):
    b = need_gpu()
    c = synth.CONFIGS[cfg]
    B, k, width, depth = c["B"], c["topk"], c["width"], c["depth"]
    dt = synth.torch_dtype(c["dtype"])
    code = b.EAGLE_BF16 if dt == torch.bfloat16 else b.EAGLE_FP32
    gen = synth.generator(sum(map(ord, cfg)) + V)
    w = synth.normal((V, d), synth.WEIGHT_STD, dt, gen)
    wd, wf = w.cuda(), w.float().numpy()
    roots = synth.random_tokens((B,), V, gen)
    max_nodes = 1 + synth.n_candidates(c)
    fused, unfused = _state(b, B, width, max_nodes, roots), _state(b, B, width, max_nodes, roots)
    sts = [oracle.tree_expand_init(int(roots[i])) for i in range(B)]
    P_max = width
    ws = b.workspace(b.eagle_lmhead_topk_workspace_size(B * P_max, d, V, k, code), "cuda")
    ws_u = b.workspace(b.eagle_lmhead_topk_workspace_size(B * P_max, d, V, k, code), "cuda")
    near_total = positions = 0
    for s in range(depth):
        P = 1 if s == 0 else width
        x = synth.normal((B * P, d), 1.0, dt, gen)
        xd = x.cuda()
        # unfused: merged lists, then the expansion
        ids = torch.empty((B * P, k), dtype=torch.int32, device="cuda")
        lps = torch.empty((B * P, k), dtype=torch.float32, device="cuda")
        b.eagle_lmhead_topk(xd, wd, k, ids, lps, ws=ws_u, status=unfused["status"])
        u = unfused
        b.eagle_tree_expand(s, width, ids.view(B, P, k), lps.view(B, P, k), u["root"], u["parent"], u["token"],
                            u["logv"], u["depth"], u["count"], u["frontier"], u["nf"], status=u["status"])
        # fused: partials, then the expansion that merges them
        f = fused
        b.eagle_lmhead_topk_partial(xd, wd, k, ws, status=f["status"])
        b.eagle_tree_expand_lmhead(s, width, k, ws, d, V, f["root"], f["parent"], f["token"], f["logv"],
                                   f["depth"], f["count"], f["frontier"], f["nf"], dtype=code,
                                   status=f["status"])
        torch.cuda.synchronize()
        for key in ("parent", "token", "logv", "depth", "count", "frontier", "nf", "status"):
            assert torch.equal(f[key], u[key]), (s, key)
        assert int(f["status"].item()) == 0
        # the merged lists against the oracle's LM head
        ids_h, lps_h = ids.cpu().numpy(), lps.cpu().numpy()
        ref = oracle.lmhead_topk(x.float().numpy(), wf, k)
        lse = ref["row_max"] + np.log(ref["row_sumexp"])
        near_total += check_topk(ids_h, lps_h, ref["z"], lambda i, v: ref["z"][i, v] - lse[i], k, 1e-4)
        positions += ids_h.size
        # the oracle's expansion of the same lists
        for i in range(B):
            n = len(sts[i]["frontier"])
            oracle.tree_expand_step(sts[i], ids_h[i * P:i * P + n], lps_h[i * P:i * P + n], width)
        nf, fr = f["nf"].cpu().numpy(), f["frontier"].cpu().numpy()
        for i in range(B):
            assert nf[i] == len(sts[i]["frontier"])
            assert fr[i, :nf[i]].tolist() == sts[i]["frontier"]
    parent, token, logv = (f[key].cpu().numpy() for key in ("parent", "token", "logv"))
    for i in range(B):
        nn = len(sts[i]["logv"])
        assert parent[i, :nn].tolist() == sts[i]["parent"]
        assert token[i, :nn].tolist() == sts[i]["token"]
        assert np.array_equal(logv[i, :nn], np.array(sts[i]["logv"], np.float32))
    print(f"{cfg}: {near_total} of {positions} list positions in near-tie groups")
    assert near_total <= positions // 100


def test_host_checks():
    b = need_gpu()
    L = b.lib()
    z = torch.zeros(64, dtype=torch.int32, device="cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    # a workspace smaller than the LM head's: refused before anything launches
    rc = L.eagle_tree_expand_lmhead(1, 0, 2, 2, 16, ws.data_ptr(), ws.numel(), 256, 1024, 1.0, 1, z.data_ptr(),
                                    *([z.data_ptr()] * 7), None, None)
    assert rc == 3
    # M = B * width above the LM head's row limit
    rc = L.eagle_tree_expand_lmhead(64, 1, 64, 2, 2048, ws.data_ptr(), ws.numel(), 256, 1024, 1.0, 1,
                                    z.data_ptr(), *([z.data_ptr()] * 7), None, None)
    assert rc == 2
