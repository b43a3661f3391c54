"""A whole EAGLE draft round on the GPU, checked stage by stage.

Per depth: eagle_draft_rows (bookkeeping) -> eagle_draft_input (input FC with
the token embedding) -> eagle_draft_layer (the drafter's decoder layer over
its own KV) -> eagle_lmhead_topk -> eagle_tree_expand.  Every stage is
compared with the oracle on the inputs the GPU had at that depth: integer
bookkeeping and the expansion bit-exact, features within the float
tolerances, top-k ids exact outside near-ties of the oracle's logits.
"""
import numpy as np
import pytest
import torch

import oracle
from eagle_speculative_decoding_gb300 import synth
from gpu_helpers import REL_TOL, check_topk, need_gpu, rel_err

pytestmark = pytest.mark.gpu


def _bf16_store(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(torch.bfloat16).double().numpy()


class Round:
    """Model, drafter state and tree store of one draft round (toy shape)."""

    def __init__(self, b, dtype, seed, B=2, d=256, Hq=4, Hkv=2, D=64, I=512, V=1024, k=4, width=4, depth=3):
        self.b, self.dtype = b, dtype
        self.B, self.d, self.Hq, self.Hkv, self.D, self.I, self.V = B, d, Hq, Hkv, D, I, V
        self.k, self.width, self.depth = k, width, depth
        self.Rmax = 1 + (depth - 1) * width
        gen = synth.generator(seed)
        dt = self.dt = synth.torch_dtype(dtype)
        std = 0.05
        nrm = lambda shape, s=std: synth.normal(shape, s, dt, gen)
        self.w = dict(norm1=(1 + 0.1 * torch.randn(d, generator=gen)).to(dt), qkv=nrm(((Hq + 2 * Hkv) * D, d)),
                      o=nrm((d, Hq * D)), norm2=(1 + 0.1 * torch.randn(d, generator=gen)).to(dt),
                      gu=nrm((2 * I, d)), down=nrm((d, I)))
        self.w_in = nrm((d, 2 * d))
        self.E = nrm((V, d), 1.0)
        self.w_lm = nrm((V, d), 0.2)
        self.g = nrm((B, d), 1.0)
        self.ctx = torch.randint(30, 90, (B,), generator=gen, dtype=torch.int32)
        self.kc, self.vc, self.table = synth.paged_kv(self.ctx.tolist(), Hkv, D, 16, dt, gen)
        self.root = synth.random_tokens((B,), V, gen)
        self.max_nodes = 1 + k + depth * width * k
        dv = "cuda"
        z = lambda *s, t=torch.int32: torch.zeros(s, dtype=t, device=dv)
        self.parent, self.token = z(B, self.max_nodes), z(B, self.max_nodes)
        self.logv, self.ndepth = z(B, self.max_nodes, t=torch.float32), z(B, self.max_nodes)
        self.count, self.frontier, self.nf = z(B), z(B, width), z(B)
        self.node_row, self.row_mask = z(B, self.max_nodes), z(B, self.Rmax, t=torch.int64)
        self.q_tree = torch.zeros((B, self.Rmax, Hq, D), dtype=dt, device=dv)
        self.k_tree = torch.zeros((B, self.Rmax, Hkv, D), dtype=dt, device=dv)
        self.v_tree = torch.zeros((B, self.Rmax, Hkv, D), dtype=dt, device=dv)
        self.status = z(1)
        self.dev = {n: getattr(self, n).to(dv) for n in ("g", "E", "w_in", "w_lm", "kc", "vc", "table", "ctx", "root")}
        self.wd = {n: t.to(dv) for n, t in self.w.items()}
        self.sts = [oracle.tree_expand_init(int(self.root[i])) for i in range(B)]
        self.node_row_ref = [dict() for _ in range(B)]
        self.row_mask_ref = [dict() for _ in range(B)]

    def f64(self, t):
        return t.double().cpu().numpy()

    def tol(self):
        return 1e-4 if self.dtype == "fp32" else REL_TOL

    def pass_(self, s, a_prev):
        """One drafter pass + LM head + expansion at depth s, each stage
        checked; returns the layer output (the next pass's parent features)."""
        b, B, d, width, k = self.b, self.B, self.d, self.width, self.k
        dv = "cuda"
        W = 1 if s == 0 else width
        prev = self.dev["g"] if s == 0 else a_prev
        r_in = torch.empty((B * W, d), dtype=self.dt, device=dv)
        tokens = torch.empty(B * W, dtype=torch.int32, device=dv)
        pos = torch.empty((B, W), dtype=torch.int32, device=dv)
        b.eagle_draft_rows(s, width, self.dev["ctx"], self.node_row, self.row_mask, prev, r_in, tokens, pos,
                           root_token=self.dev["root"], frontier=self.frontier, n_frontier=self.nf,
                           node_parent=self.parent, node_token=self.token, node_depth=self.ndepth,
                           status=self.status)
        torch.cuda.synchronize()
        # -- bookkeeping: exact
        prev64 = self.f64(prev)
        W_prev = 1 if s <= 1 else width
        rm = self.row_mask.cpu().numpy().view(np.uint64)
        n_of = []
        for i in range(B):
            src = prev64[i:i + 1] if s == 0 else prev64[i * W_prev:(i + 1) * W_prev]
            rows, toks, ps, feats = oracle.draft_rows(s, width, self.sts[i] if s else None, self.node_row_ref[i],
                                                      self.row_mask_ref[i], int(self.ctx[i]), src,
                                                      root_token=int(self.root[i]))
            n = len(rows)
            n_of.append(n)
            assert tokens[i * W:i * W + n].cpu().tolist() == toks
            assert pos[i, :n].cpu().tolist() == ps
            assert np.array_equal(self.f64(r_in[i * W:i * W + n]), feats)
            assert [int(rm[i, r]) for r in rows] == [int(self.row_mask_ref[i][r]) for r in rows]
            assert np.all(self.f64(r_in[i * W + n:(i + 1) * W]) == 0)
        # -- input FC
        u = torch.empty((B * W, d), dtype=self.dt, device=dv)
        b.eagle_draft_input(r_in, tokens, self.dev["E"], self.dev["w_in"], u, status=self.status)
        torch.cuda.synchronize()
        u_ref = oracle.draft_input(self.f64(r_in), tokens.cpu().numpy(), self.f64(self.E), self.f64(self.w_in))
        assert rel_err(self.f64(u), u_ref) < self.tol()
        # -- decoder layer over the drafter's own KV
        r0 = 0 if s == 0 else 1 + (s - 1) * width
        kt0, vt0 = self.f64(self.k_tree), self.f64(self.v_tree)
        a = torch.empty((B * W, d), dtype=self.dt, device=dv)
        b.eagle_draft_layer(u, self.wd, pos, self.dev["kc"], self.dev["vc"], self.dev["table"], self.dev["ctx"],
                            self.q_tree, self.k_tree, self.v_tree, self.row_mask, r0, a, status=self.status)
        torch.cuda.synchronize()
        a_ref, k_ref, _ = oracle.draft_layer(
            self.f64(u), {n: self.f64(t) for n, t in self.w.items()}, pos.cpu().numpy(), self.f64(self.kc),
            self.f64(self.vc), self.table.numpy(), self.ctx.numpy(), kt0, vt0, rm, r0, self.Hq, self.Hkv,
            store=_bf16_store if self.dtype == "bf16" else None)
        assert rel_err(self.f64(a), a_ref) < self.tol()
        assert rel_err(self.f64(self.k_tree)[:, r0:r0 + W], k_ref) < self.tol()
        # -- LM head top-k of the drafter outputs
        ids = torch.empty((B * W, k), dtype=torch.int32, device=dv)
        lps = torch.empty((B * W, k), dtype=torch.float32, device=dv)
        b.eagle_lmhead_topk(a, self.dev["w_lm"], k, ids, lps, status=self.status)
        torch.cuda.synchronize()
        ref = oracle.lmhead_topk(self.f64(a), self.f64(self.w_lm), k)
        z = ref["z"]
        lse = ref["row_max"] + np.log(ref["row_sumexp"])
        live = [i * W + j for i in range(B) for j in range(n_of[i])]
        check_topk(ids.cpu().numpy()[live], lps.cpu().numpy()[live], z[live], lambda i, v: z[live[i], v] - lse[live[i]],
                   k, 1e-4 if self.dtype == "fp32" else 1e-3)
        # -- expansion: bit-exact against the oracle fed the same candidates
        b.eagle_tree_expand(s, width, ids.view(B, W, k), lps.view(B, W, k), self.dev["root"], self.parent,
                            self.token, self.logv, self.ndepth, self.count, self.frontier, self.nf,
                            status=self.status)
        torch.cuda.synchronize()
        ids_np, lps_np = ids.cpu().numpy(), lps.cpu().numpy()
        for i in range(B):
            oracle.tree_expand_step(self.sts[i], ids_np[i * W:i * W + n_of[i]], lps_np[i * W:i * W + n_of[i]], width)
            n = len(self.sts[i]["parent"])
            assert int(self.count[i]) == n
            assert self.parent[i, :n].cpu().tolist() == self.sts[i]["parent"]
            assert self.token[i, :n].cpu().tolist() == self.sts[i]["token"]
            assert self.ndepth[i, :n].cpu().tolist() == self.sts[i]["depth"]
            assert int(self.nf[i]) == len(self.sts[i]["frontier"])
            assert self.frontier[i, :int(self.nf[i])].cpu().tolist() == self.sts[i]["frontier"]
        assert int(self.status.item()) == 0
        return a


@pytest.mark.parametrize("dtype,seed", [("fp32", 1), ("bf16", 2), ("bf16", 3)])
def test_draft_round_chained(dtype, seed):
    b = need_gpu()
    rd = Round(b, dtype, seed)
    a = None
    for s in range(rd.depth):
        a = rd.pass_(s, a)
    # the finished round flattens like any EAGLE-2 tree
    n = len(rd.sts[0]["parent"]) - 1
    assert n == rd.k + (rd.depth - 1) * rd.width * rd.k


def test_draft_rows_rejects_an_unprocessed_parent():
    b = need_gpu()
    rd = Round(b, "fp32", 4)
    a = rd.pass_(0, None)
    # forget that the root was processed: every depth-1 node now lacks its parent's row
    rd.node_row.fill_(-1)
    r_in = torch.empty((rd.B * rd.width, rd.d), dtype=rd.dt, device="cuda")
    tokens = torch.empty(rd.B * rd.width, dtype=torch.int32, device="cuda")
    pos = torch.empty((rd.B, rd.width), dtype=torch.int32, device="cuda")
    b.eagle_draft_rows(1, rd.width, rd.dev["ctx"], rd.node_row, rd.row_mask, a, r_in, tokens, pos,
                       frontier=rd.frontier, n_frontier=rd.nf, node_parent=rd.parent, node_token=rd.token,
                       node_depth=rd.ndepth, status=rd.status)
    torch.cuda.synchronize()
    assert int(rd.status.item()) == 5
    assert float(r_in.abs().max()) == 0.0
