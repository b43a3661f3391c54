"""GPU parity of the stochastic-verification statistics path:
eagle_lmhead_verify_stats (LM head in exponential-race mode + child logits)
and eagle_tree_verify_stats, against oracle.verify_stats / oracle.tree_verify
on the full fp64 logits of the same bf16 (or fp32) inputs."""
import numpy as np
import pytest
import torch

import oracle
from eagle_speculative_decoding_gb300 import synth
from gpu_helpers import need_gpu

pytestmark = pytest.mark.gpu

MARGIN = 1e-4  # fp32 logits and fp32 logs: decisions closer than this are not asserted


def _case(seed, B, R, V, d, depth, dt, lift=1.0):
    gen = synth.generator(seed)
    parents, toks = [], []
    for _ in range(B):
        p, _ = synth.random_tree(R, depth, gen)
        parents.append(p)
        toks.append(synth.distinct_sibling_tokens(p, V, gen))
    parent, tok = torch.stack(parents), torch.stack(toks)
    x = synth.normal((B * R, d), 1.0, torch.float32, gen)
    w = synth.normal((V, d), 0.05, torch.float32, gen)
    # point each child's token row toward its parent's activation so that
    # target probabilities of drafted tokens are large (acceptances happen)
    for b in range(B):
        for c in range(1, R):
            r = int(parent[b, c])
            xr = x[b * R + r]
            w[int(tok[b, c])] += lift * xr / xr.norm() * (2.5 + 0.5 * torch.rand((), generator=gen))
    return parent, tok, x.to(dt), w.to(dt)


def _gpu_stats(b, parent, tok, x, w, T, race_k, seed, offset, n_rows=None):
    d = "cuda"
    B, R = parent.shape
    M = B * R
    out = dict(race_ids=torch.empty((M, race_k), dtype=torch.int32, device=d),
               race_keys=torch.empty((M, race_k), dtype=torch.float32, device=d),
               row_max=torch.empty(M, device=d), row_sumexp=torch.empty(M, device=d),
               child_logit=torch.empty(M, device=d))
    st = torch.zeros(1, dtype=torch.int32, device=d)
    b.eagle_lmhead_verify_stats(x.to(d), w.to(d), parent.to(d), tok.to(d), T, race_k,
                                out["race_ids"], out["race_keys"], out["row_max"],
                                out["row_sumexp"], out["child_logit"],
                                n_rows=None if n_rows is None else n_rows.to(d), seed=seed,
                                offset=offset, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return out


def _race_k(parent):
    B, R = parent.shape
    return max(int((parent[bb, 1:] == r).sum()) for bb in range(B) for r in range(R)) + 1


@pytest.mark.parametrize("dtype,B,R,V,d,T", [
    ("bf16", 3, 13, 4096, 256, 0.8),
    ("bf16", 8, 9, 2048, 128, 1.0),
    ("fp32", 2, 17, 1024, 256, 0.6),
])
def test_statistics_match_oracle(dtype, B, R, V, d, T):
    b = need_gpu()
    T = float(np.float32(T))
    parent, tok, x, w = _case(B * 7 + R, B, R, V, d, 4, synth.torch_dtype(dtype))
    rk = _race_k(parent)
    seed, off = 4242 + B, 17
    g = _gpu_stats(b, parent, tok, x, w, T, rk, seed, off)
    ref = oracle.verify_stats(x.double().numpy(), w.double().numpy(), parent.numpy(), tok.numpy(),
                              T, rk, seed=seed, offset=off)
    tol = 1e-4
    np.testing.assert_allclose(g["row_max"].cpu().numpy(), ref["row_max"], rtol=tol, atol=tol)
    lse_g = g["row_max"].cpu().numpy() + np.log(g["row_sumexp"].cpu().numpy())
    np.testing.assert_allclose(lse_g, ref["row_max"] + np.log(ref["row_sumexp"]), rtol=0, atol=tol)
    np.testing.assert_allclose(g["child_logit"].cpu().numpy(), ref["child_logit"], rtol=tol, atol=tol)
    gi, gk = g["race_ids"].cpu().numpy(), g["race_keys"].cpu().numpy()
    rkeys = ref["race_keys"]
    for row in range(B * R):
        for j in range(rk):
            lo = rkeys[row, j - 1] - rkeys[row, j] if j > 0 else np.inf
            hi = rkeys[row, j] - rkeys[row, j + 1] if j + 1 < rk else np.inf
            if min(lo, hi) > 10 * tol:
                assert gi[row, j] == ref["race_ids"][row, j], (row, j)
            assert abs(gk[row, j] - rkeys[row, j]) < 10 * tol, (row, j)


@pytest.mark.parametrize("B,R,V,d,T", [(6, 13, 4096, 256, 0.8), (16, 9, 2048, 128, 1.0)])
def test_walk_from_statistics_matches_full_logit_walk(B, R, V, d, T):
    b = need_gpu()
    T = float(np.float32(T))
    parent, tok, x, w = _case(B + 3 * R, B, R, V, d, 4, torch.bfloat16)
    rk = _race_k(parent)
    seed, off = 777 + R, 3
    g = _gpu_stats(b, parent, tok, x, w, T, rk, seed, off)
    dev = "cuda"
    depth = 4
    acc = torch.empty(B, dtype=torch.int32, device=dev)
    path = torch.empty((B, depth + 1), dtype=torch.int32, device=dev)
    out = torch.empty((B, depth + 1), dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    b.eagle_tree_verify_stats(parent.to(dev), tok.to(dev), T, depth, g["row_max"], g["row_sumexp"],
                              g["child_logit"], g["race_ids"], acc, path, out, V, seed=seed,
                              offset=off, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    z = (x.double() @ w.double().T).reshape(B, R, V).numpy()
    ref = oracle.tree_verify(parent.numpy(), tok.numpy(), T, depth, target_logits=z, seed=seed,
                             offset=off)
    close = {bb for kind, bb, m in ref["margins"] if m < MARGIN}
    checked = 0
    for bb in range(B):
        if bb in close:
            continue
        checked += 1
        assert acc[bb].item() == ref["accept_len"][bb], bb
        assert path[bb].tolist() == ref["path_rows"][bb].tolist(), bb
        assert out[bb].tolist() == ref["out_tokens"][bb].tolist(), bb
    print(f"B={B} R={R} V={V}: {B - checked} of {B} requests within {MARGIN} of a threshold")
    assert checked == B  # these seeds put no decision within MARGIN of its threshold
    assert ref["accept_len"].max() >= 1


def test_full_size_serve_shape_sampled_rows():
    b = need_gpu()
    c = synth.CONFIGS["serve64"]
    B, R, V, d = c["B"], c["N"] + 1, c["V"], c["d"]
    gen = synth.generator(31)
    parents, toks = [], []
    for _ in range(B):
        p, _ = synth.random_tree(R, c["depth"], gen)
        parents.append(p)
        toks.append(synth.distinct_sibling_tokens(p, V, gen))
    parent, tok = torch.stack(parents), torch.stack(toks)
    x = synth.normal((B * R, d), 1.0, torch.bfloat16, gen)
    w = synth.normal((V, d), synth.WEIGHT_STD, torch.bfloat16, gen)
    rk = c["topk"] + 1
    g = _gpu_stats(b, parent, tok, x, w, 1.0, rk, 5, 0)
    rows = [0, 1, 8, 9, 100, 301, 575]
    ref = oracle.verify_stats(x.double().numpy(), w.double().numpy(), parent.numpy(), tok.numpy(),
                              1.0, rk, seed=5, offset=0, rows=rows)
    for row in rows:
        assert abs(g["row_max"][row].item() - ref["row_max"][row]) < 1e-4
        assert abs(np.log(g["row_sumexp"][row].item()) - np.log(ref["row_sumexp"][row])) < 1e-4
        assert abs(g["child_logit"][row].item() - ref["child_logit"][row]) < 1e-4
        k0 = ref["race_keys"][row]
        if k0[0] - k0[1] > 1e-3:
            assert g["race_ids"][row, 0].item() == ref["race_ids"][row, 0]
        assert abs(g["race_keys"][row, 0].item() - k0[0]) < 1e-3


def test_host_validation():
    b = need_gpu()
    d = "cuda"
    parent = torch.tensor([[-1, 0]], dtype=torch.int32, device=d)
    tok = torch.tensor([[0, 1]], dtype=torch.int32, device=d)
    x = torch.zeros((2, 64), dtype=torch.bfloat16, device=d)
    w = torch.zeros((64, 64), dtype=torch.bfloat16, device=d)
    f = lambda *s, t=torch.float32: torch.empty(s, dtype=t, device=d)
    with pytest.raises(b.EagleError):  # T = 0 is greedy: no statistics path
        b.eagle_lmhead_verify_stats(x, w, parent, tok, 0.0, 2, f(2, 2, t=torch.int32), f(2, 2),
                                    f(2), f(2), f(2))
    with pytest.raises(b.EagleError):  # race_k beyond the register list
        b.eagle_lmhead_verify_stats(x, w, parent, tok, 1.0, 33, f(2, 33, t=torch.int32),
                                    f(2, 33), f(2), f(2), f(2))
