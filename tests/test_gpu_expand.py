"""GPU parity of eagle_tree_expand / eagle_tree_expand_finalize (bit-exact)."""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from eagle_speculative_decoding_gb300 import synth
from gpu_helpers import need_gpu

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "eagle2_numeric_tree.txt")


class GpuTree:
    def __init__(self, b, B, width, k, max_nodes, R, root_tokens):
        d = "cuda"
        self.b, self.B, self.width, self.k, self.R = b, B, width, k, R
        z = lambda *s, dt=torch.int32: torch.zeros(s, dtype=dt, device=d)
        self.parent, self.token = z(B, max_nodes), z(B, max_nodes)
        self.logv, self.depth = z(B, max_nodes, dt=torch.float32), z(B, max_nodes)
        self.count, self.frontier, self.nf = z(B), z(B, width), z(B)
        self.root = root_tokens.to(d)
        self.status = z(1)

    def step(self, s, ids, lps):
        self.b.eagle_tree_expand(s, self.width, ids.cuda(), lps.cuda(), self.root, self.parent,
                                 self.token, self.logv, self.depth, self.count, self.frontier,
                                 self.nf, status=self.status)

    def finalize(self, budget, ctx):
        d = "cuda"
        R, B = self.R, self.B
        out = {n: torch.zeros((B, R), dtype=torch.int32, device=d)
               for n in ("token", "parent_row", "depth", "node_id", "position")}
        out["mask"] = torch.zeros((B, R), dtype=torch.int64, device=d)
        out["n_rows"] = torch.zeros(B, dtype=torch.int32, device=d)
        self.b.eagle_tree_expand_finalize(budget, self.parent, self.token, self.logv, self.depth,
                                          self.count, ctx.cuda(), out["token"], out["parent_row"],
                                          out["depth"], out["mask"], out["node_id"],
                                          out["position"], out["n_rows"], status=self.status)
        torch.cuda.synchronize()
        return {k: v.cpu().numpy() for k, v in out.items()}


def test_numeric_example_on_gpu():
    b = need_gpu()
    # A=.60, B=.40 under the seed; A1=.80, A2=.20 under A; B1=.95 under B
    lp = lambda c: math.log(c)
    g = GpuTree(b, 1, 2, 2, 16, 5, torch.tensor([1], dtype=torch.int32))
    g.step(0, torch.tensor([[[10, 11]]], dtype=torch.int32),
           torch.tensor([[[lp(.6), lp(.4)]]], dtype=torch.float32))
    torch.cuda.synchronize()
    assert g.frontier.cpu().tolist() == [[1, 2]]
    g.step(1, torch.tensor([[[12, 13], [14, -1]]], dtype=torch.int32),
           torch.tensor([[[lp(.8), lp(.2)], [lp(.95), -np.inf]]], dtype=torch.float32))
    flat = g.finalize(4, torch.tensor([100], dtype=torch.int32))
    # rows: A (token 10), A1 (12), B (11), B1 (14)
    assert flat["token"][0].tolist() == [1, 10, 12, 11, 14]
    assert flat["parent_row"][0].tolist() == [-1, 0, 1, 0, 3]
    assert flat["mask"][0].tolist() == [1, 3, 7, 9, 25]
    assert flat["position"][0].tolist() == [100, 101, 102, 101, 102]
    assert int(g.status.item()) == 0


@pytest.mark.parametrize("cfg", ["toy", "llama8b", "serve64", "long4", "chain3"])
def test_random_trees_bit_exact(cfg):
    b = need_gpu()
    c = synth.CONFIGS[cfg]
    B, k, width, depth, N = c["B"], c["topk"], c["width"], c["depth"], c["N"]
    V = 5000
    gen = synth.generator(sum(map(ord, cfg)))
    max_nodes = 1 + synth.n_candidates(c)
    R = N + 1
    roots = synth.random_tokens((B,), V, gen)
    g = GpuTree(b, B, width, k, max_nodes, R, roots)
    sts = [oracle.tree_expand_init(int(roots[i])) for i in range(B)]
    for s in range(depth):
        P = 1 if s == 0 else width
        ids = torch.full((B, P, k), -1, dtype=torch.int32)
        lps = torch.full((B, P, k), -np.inf, dtype=torch.float32)
        for i in range(B):
            n = len(sts[i]["frontier"])
            a, l = synth.draft_candidates(n, k, V, gen)
            ids[i, :n], lps[i, :n] = a, l
            oracle.tree_expand_step(sts[i], a.numpy(), l.numpy(), width)
        g.step(s, ids, lps)
        torch.cuda.synchronize()
        fr = g.frontier.cpu().numpy()
        nf = g.nf.cpu().numpy()
        for i in range(B):
            assert nf[i] == len(sts[i]["frontier"])
            assert fr[i, :nf[i]].tolist() == sts[i]["frontier"]
    ctx = synth.ctx_lengths(c, gen)
    flat = g.finalize(N, ctx)
    assert int(g.status.item()) == 0
    logv = g.logv.cpu().numpy()
    for i in range(B):
        ref = oracle.tree_expand_finalize(sts[i], N, int(ctx[i]), R_out=R)
        assert flat["n_rows"][i] == ref["n_rows"]
        for key in ("token", "parent_row", "depth", "node_id", "position"):
            assert np.array_equal(flat[key][i], ref[key]), key
        assert np.array_equal(flat["mask"][i].astype(np.uint64), ref["mask"])
        nn = len(sts[i]["logv"])
        assert np.array_equal(logv[i, :nn], np.array(sts[i]["logv"], np.float32))


def test_device_validation_duplicate_and_nan():
    b = need_gpu()
    g = GpuTree(b, 2, 2, 2, 16, 4, torch.tensor([1, 1], dtype=torch.int32))
    ids = torch.tensor([[[3, 3]], [[4, 5]]], dtype=torch.int32)
    lps = torch.tensor([[[-1.0, -2.0]], [[-1.0, -2.0]]])
    g.step(0, ids, lps)
    torch.cuda.synchronize()
    assert int(g.status.item()) == 5  # duplicate under one parent
    assert g.nf.cpu().tolist() == [0, 2]
    g2 = GpuTree(b, 1, 2, 2, 16, 4, torch.tensor([1], dtype=torch.int32))
    g2.step(0, torch.tensor([[[3, 4]]], dtype=torch.int32), torch.tensor([[[-1.0, float("nan")]]]))
    torch.cuda.synchronize()
    assert int(g2.status.item()) == 7
    g3 = GpuTree(b, 1, 2, 2, 16, 4, torch.tensor([1], dtype=torch.int32))
    g3.step(0, torch.tensor([[[3, 4]]], dtype=torch.int32), torch.tensor([[[-0.1, -0.2]]]))
    torch.cuda.synchronize()
    assert int(g3.status.item()) == 5  # sibling mass above one


def test_budget_zero_and_host_limits():
    b = need_gpu()
    g = GpuTree(b, 1, 2, 2, 16, 3, torch.tensor([9], dtype=torch.int32))
    g.step(0, torch.tensor([[[3, 4]]], dtype=torch.int32), torch.tensor([[[-1.0, -2.0]]]))
    flat = g.finalize(0, torch.tensor([5], dtype=torch.int32))
    assert flat["n_rows"][0] == 1 and flat["token"][0].tolist() == [9, -1, -1]
    with pytest.raises(b.EagleError):
        g.step(5, torch.zeros((1, 2, 2), dtype=torch.int32), torch.zeros((1, 2, 2)))  # max_nodes too small


@pytest.mark.parametrize("schedule,k,B", [((4, 3, 2, 1), 4, 1), ((4, 3, 2, 1), 4, 3), ((2, 2, 2, 2, 1), 2, 5),
                                          ((1, 1, 1), 1, 2), ((3, 0, 2), 3, 2)])
def test_static_tree_bit_exact(schedule, k, B):
    # a fixed tree grown depth by depth with the same fan-out for every node of
    # a depth; node arrays and the flatten of the whole tree are bit-exact
    b = need_gpu()
    V = 3000
    gen = synth.generator(sum(schedule) * 10 + k + B)
    widths = [1]
    for f in schedule:
        widths.append(widths[-1] * f)
    width = max(max(widths[1:]), 1)
    n_nodes = sum(widths[1:])
    max_nodes = 1 + k + len(schedule) * width * k
    roots = synth.random_tokens((B,), V, gen)
    d = "cuda"
    z = lambda *s, dt=torch.int32: torch.zeros(s, dtype=dt, device=d)
    parent, token, logv, depth = z(B, max_nodes), z(B, max_nodes), z(B, max_nodes, dt=torch.float32), z(B, max_nodes)
    count, frontier, nf, status = z(B), z(B, width), z(B), z(1)
    sts = [oracle.tree_expand_init(int(roots[i])) for i in range(B)]
    for s, f in enumerate(schedule):
        P = 1 if s == 0 else width
        ids = torch.full((B, P, k), -1, dtype=torch.int32)
        lps = torch.full((B, P, k), -math.inf, dtype=torch.float32)
        for i in range(B):
            npar = len(sts[i]["frontier"])
            ci, cl = synth.draft_candidates(npar, k, V, gen)
            ids[i, :npar], lps[i, :npar] = ci, cl
        fan = torch.full((P,), f, dtype=torch.int32, device=d)
        b.eagle_tree_expand_static(s, width, fan, ids.to(d), lps.to(d), roots.to(d), parent, token, logv, depth,
                                   count, frontier, nf, status=status)
        for i in range(B):
            npar = len(sts[i]["frontier"])
            oracle.static_tree_step(sts[i], ids[i, :npar].numpy(), lps[i, :npar].numpy(), [f] * npar)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for i in range(B):
        n = len(sts[i]["parent"])
        assert n == 1 + n_nodes
        assert int(count[i]) == n
        assert parent[i, :n].cpu().tolist() == sts[i]["parent"]
        assert token[i, :n].cpu().tolist() == sts[i]["token"]
        assert np.array_equal(logv[i, :n].cpu().numpy(), np.array(sts[i]["logv"], np.float32))
        assert depth[i, :n].cpu().tolist() == sts[i]["depth"]
        nfi = int(nf[i])
        assert frontier[i, :nfi].cpu().tolist() == sts[i]["frontier"][:width]
    if n_nodes + 1 <= 64:
        R = n_nodes + 1
        ctx = torch.randint(0, 500, (B,), generator=gen, dtype=torch.int32)
        out = {n: torch.zeros((B, R), dtype=torch.int32, device=d)
               for n in ("token", "parent_row", "depth", "node_id", "position")}
        out["mask"] = torch.zeros((B, R), dtype=torch.int64, device=d)
        out["n_rows"] = torch.zeros(B, dtype=torch.int32, device=d)
        b.eagle_tree_expand_finalize(n_nodes, parent, token, logv, depth, count, ctx.to(d), out["token"],
                                     out["parent_row"], out["depth"], out["mask"], out["node_id"],
                                     out["position"], out["n_rows"], status=status)
        torch.cuda.synchronize()
        for i in range(B):
            ref = oracle.tree_expand_finalize(sts[i], n_nodes, int(ctx[i]), R_out=R)
            for key in ("token", "parent_row", "depth", "node_id", "position"):
                assert np.array_equal(out[key][i].cpu().numpy(), ref[key]), key
            assert np.array_equal(out["mask"][i].cpu().numpy().view(np.uint64), ref["mask"])


def test_static_tree_bad_fanout_flags():
    b = need_gpu()
    d = "cuda"
    z = lambda *s, dt=torch.int32: torch.zeros(s, dtype=dt, device=d)
    parent, token, logv, depth = z(1, 64), z(1, 64), z(1, 64, dt=torch.float32), z(1, 64)
    count, frontier, nf, status = z(1), z(1, 4), z(1), z(1)
    ids = torch.tensor([[[5, 6, 7]]], dtype=torch.int32, device=d)
    lps = torch.log(torch.tensor([[[0.5, 0.2, 0.1]]], device=d))
    fan = torch.tensor([4], dtype=torch.int32, device=d)  # more than k = 3
    b.eagle_tree_expand_static(0, 4, fan, ids, lps, torch.tensor([1], dtype=torch.int32, device=d), parent,
                               token, logv, depth, count, frontier, nf, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 5
