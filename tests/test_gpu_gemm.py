"""GPU parity of eagle_lmhead_topk and eagle_fuse_proj against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from eagle_speculative_decoding_gb300 import synth
from gpu_helpers import NORM_TOL, REL_TOL, need_gpu, norm_err, rel_err, check_topk

pytestmark = pytest.mark.gpu


def _lm_gpu(b, x, w, k, T, bias=None):
    d = "cuda"
    M = x.shape[0]
    ids = torch.empty((M, k), dtype=torch.int32, device=d)
    lp = torch.empty((M, k), dtype=torch.float32, device=d)
    rm = torch.empty(M, dtype=torch.float32, device=d)
    rs = torch.empty(M, dtype=torch.float32, device=d)
    st = torch.zeros(1, dtype=torch.int32, device=d)
    b.eagle_lmhead_topk(x.to(d), w.to(d), k, ids, lp, temperature=T,
                        bias=None if bias is None else bias.to(d), row_max=rm, row_sumexp=rs, status=st)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), lp.cpu().numpy(), rm.cpu().numpy(), rs.cpu().numpy(), int(st.item())


def _lm_check(b, M, d, V, k, T, dtype, seed, rows=None, bias=False):
    gen = synth.generator(seed)
    dt = synth.torch_dtype(dtype)
    x = synth.normal((M, d), 1.0, dt, gen)
    w = synth.normal((V, d), synth.WEIGHT_STD, dt, gen)
    bb = synth.normal((V,), 0.5, torch.float32, gen) if bias else None
    ids, lp, rm, rs, st = _lm_gpu(b, x, w, k, T, bb)
    assert st == 0
    rows = np.arange(M) if rows is None else np.asarray(rows)
    ref = oracle.lmhead_topk(x.float().numpy(), w.float().numpy(), k, temperature=T,
                             bias=None if bb is None else bb.numpy(), rows=rows)
    z = ref["z"]
    lse = ref["row_max"] + np.log(ref["row_sumexp"])
    # fp32 accumulation error of z is ~1e-6 here; closer logits are near ties
    near = check_topk(ids[rows], lp[rows], z, lambda i, v: z[i, v] / T - lse[i], k, 1e-4)
    assert np.abs(rm[rows] - ref["row_max"]).max() < 1e-3
    assert np.abs(np.log(rs[rows]) + rm[rows] - lse).max() < 1e-3
    return near


# ``near``: positions whose oracle logit gap to a neighbour in the sorted list
# is below 1e-4, counted from the oracle on these seeds (they depend on the
# generator only).  Only there may the GPU list a member of the near-tie
# group in place of the oracle's id; everywhere else ids are bit-exact.
@pytest.mark.parametrize("M,d,V,k,T,dtype,near_max", [
    (1, 64, 128, 1, 1.0, "bf16", 0),
    (10, 256, 1024, 4, 1.0, "fp32", 0),     # toy, exact fp32 on the CUDA cores
    (17, 256, 1024, 4, 1.0, "fp32", 1),
    (13, 512, 4096, 10, 0.7, "bf16", 0),    # ragged M, several vocab tiles
    (61, 1024, 8192, 1, 1.0, "bf16", 0),
    (100, 512, 4096, 32, 1.0, "bf16", 72),  # k = 32: bf16 products at d 512 tie often
    (300, 256, 2048, 2, 1.0, "bf16", 0),    # two activation groups
    (300, 256, 65536, 3, 1.0, "bf16", 0),   # three groups, 256-row W_U tiles
])
def test_lmhead_small(M, d, V, k, T, dtype, near_max):
    b = need_gpu()
    near = _lm_check(b, M, d, V, k, T, dtype, seed=M * 7 + k)
    print(f"M={M} d={d} V={V} k={k}: {near} of {M * k} positions in near-tie groups")
    assert near <= near_max


def test_lmhead_bias():
    b = need_gpu()
    _lm_check(b, 9, 256, 2048, 5, 1.0, "bf16", seed=3, bias=True)


@pytest.mark.parametrize("dtype,k", [("bf16", 8), ("bf16", 3), ("fp32", 8)])
def test_lmhead_masked_vocabulary(dtype, k):
    """Degenerate rows: a -inf bias masks all but three ids (spread over the
    CTAs' vocabulary slices), so a top-8 list must end with masked ids.  They
    tie at -inf and are listed by ascending id after the three finite ones,
    with log-prob -inf, as the oracle orders them."""
    b = need_gpu()
    M, d, V = 20, 256, 4096
    gen = synth.generator(41 + k)
    dt = synth.torch_dtype(dtype)
    x = synth.normal((M, d), 1.0, dt, gen)
    w = synth.normal((V, d), synth.WEIGHT_STD, dt, gen)
    bias = torch.full((V,), float("-inf"))
    allowed = [4000, 1234, 77]
    bias[allowed] = 0.0
    ids, lp, rm, rs, st = _lm_gpu(b, x, w, k, 1.0, bias)
    assert st == 0
    ref = oracle.lmhead_topk(x.float().numpy(), w.float().numpy(), k, bias=bias.numpy())
    assert np.array_equal(ids, ref["ids"])
    fin = np.isfinite(ref["logprobs"])
    assert fin.sum(axis=1).tolist() == [min(k, 3)] * M
    assert np.all(np.isneginf(lp[~fin]))
    assert np.abs(lp[fin] - ref["logprobs"][fin]).max() < 1e-3
    assert np.abs(rm - ref["row_max"]).max() < 1e-3


def test_lmhead_nan_logit_sets_status_and_is_never_listed():
    """A NaN logit (here from a NaN bias entry) raises EAGLE_ERR_NONFINITE;
    the NaN id never enters a list, so the ids equal the oracle's with that id
    masked."""
    b = need_gpu()
    M, d, V, k = 12, 256, 4096, 8
    gen = synth.generator(43)
    x = synth.normal((M, d), 1.0, torch.bfloat16, gen)
    w = synth.normal((V, d), synth.WEIGHT_STD, torch.bfloat16, gen)
    ref0 = oracle.lmhead_topk(x.float().numpy(), w.float().numpy(), k)
    bad = int(ref0["ids"][0, 0])  # row 0's best id
    bias = torch.zeros(V)
    bias[bad] = float("nan")
    ids, _, _, _, st = _lm_gpu(b, x, w, k, 1.0, bias)
    assert st == 7  # EAGLE_ERR_NONFINITE
    masked = bias.clone()
    masked[bad] = float("-inf")
    ref = oracle.lmhead_topk(x.float().numpy(), w.float().numpy(), k, bias=masked.numpy())
    assert not np.any(ids == bad)
    check_topk(ids, np.zeros_like(ids, dtype=np.float32), ref["z"], lambda i, v: 0.0, k, 1e-4)


@pytest.mark.parametrize("M,d,V,k,dtype", [(10, 4096, 128256, 10, "bf16"), (300, 256, 4096, 3, "bf16"),
                                           (7, 128, 1024, 4, "fp32")])
def test_lmhead_partial_then_merge_equals_one_call(M, d, V, k, dtype):
    # the two halves launch the same kernels: outputs are bit-identical
    b = need_gpu()
    gen = synth.generator(M + V)
    dt = synth.torch_dtype(dtype)
    x = synth.normal((M, d), 1.0, dt, gen).cuda()
    w = synth.normal((V, d), synth.WEIGHT_STD, dt, gen).cuda()
    code = b.EAGLE_BF16 if dtype == "bf16" else b.EAGLE_FP32
    ws = b.workspace(b.eagle_lmhead_topk_workspace_size(M, d, V, k, code), "cuda")
    outs = []
    for split in (False, True):
        ids = torch.empty((M, k), dtype=torch.int32, device="cuda")
        lps = torch.empty((M, k), dtype=torch.float32, device="cuda")
        mx = torch.empty(M, dtype=torch.float32, device="cuda")
        se = torch.empty(M, dtype=torch.float32, device="cuda")
        if split:
            b.eagle_lmhead_topk_partial(x, w, k, ws, temperature=0.8)
            b.eagle_lmhead_topk_merge(M, d, V, ids, lps, ws, dtype=code, temperature=0.8, row_max=mx, row_sumexp=se)
        else:
            b.eagle_lmhead_topk(x, w, k, ids, lps, temperature=0.8, row_max=mx, row_sumexp=se, ws=ws)
        torch.cuda.synchronize()
        outs.append([t.cpu() for t in (ids, lps, mx, se)])
    for a, c in zip(*outs):
        assert torch.equal(a, c)


@pytest.mark.parametrize("M,d,k,T,rows", [
    (10, 4096, 10, 1.0, None),                  # llama8b draft rows, width 10
    (61, 4096, 1, 1.0, [0, 17, 33, 60]),        # llama8b verify rows
    (576, 4096, 1, 1.0, [0, 191, 192, 383, 384, 575]),  # serve64 verify rows, 3 groups
    (128, 4096, 2, 1.0, [0, 64, 127]),          # serve64 draft rows
    (32, 4096, 8, 0.6, [0, 31]),                # long4 draft rows
    (10, 8192, 10, 1.0, [0, 9]),                # llama70b draft rows
])
def test_lmhead_full_vocab(M, d, k, T, rows):
    b = need_gpu()
    near = _lm_check(b, M, d, 128256, k, T, "bf16", seed=M + d, rows=rows)
    assert near == 0  # every id of these lists is asserted bit-exact


def _margin_rows(M, d, V, gen, w, rows, margin):
    """Activation rows whose checked rows have a top-2 logit gap above
    ``margin`` (oracle logits; rows that miss it are redrawn)."""
    x = synth.normal((M, d), 1.0, torch.bfloat16, gen)
    wf = w.float().numpy()
    for _ in range(20):
        z = oracle.lmhead_topk(x.float().numpy(), wf, 2, rows=rows)["z"]
        top2 = np.sort(z, axis=1)[:, -2:]
        bad = [int(r) for r, g in zip(rows, top2[:, 1] - top2[:, 0]) if g <= margin]
        if not bad:
            return x
        for r in bad:
            x[r] = synth.normal((d,), 1.0, torch.bfloat16, gen)
    raise AssertionError("could not draw rows with the margin")


@pytest.mark.parametrize("M,rows", [(61, None), (576, [0, 1, 100, 191, 192, 383, 384, 500, 575])])
def test_lmhead_greedy_argmax_exact_at_margin(M, rows):
    """Greedy verification reads the LM head's top-1 (k = 1) as the target
    argmax.  With every checked row's top-2 logit gap above 1e-2 (the greedy
    cases' margin) the ids are asserted equal to the oracle's with no
    exemption at all; llama8b's 61 verify rows and serve64's 576."""
    b = need_gpu()
    d, V = 4096, 128256
    gen = synth.generator(900 + M)
    w = synth.normal((V, d), synth.WEIGHT_STD, torch.bfloat16, gen)
    rows = np.arange(M) if rows is None else np.asarray(rows)
    x = _margin_rows(M, d, V, gen, w, rows, 1e-2)
    ids, lp, _, _, st = _lm_gpu(b, x, w, 1, 1.0)
    assert st == 0
    ref = oracle.lmhead_topk(x.float().numpy(), w.float().numpy(), 1, rows=rows)
    assert np.array_equal(ids[rows, 0], ref["ids"][:, 0])
    assert np.abs(lp[rows, 0] - ref["logprobs"][:, 0]).max() < 1e-3


def _fp_check(b, M, d, dtype, seed, rows=None, bias=False):
    gen = synth.generator(seed)
    dt = synth.torch_dtype(dtype)
    hl, hm, hh = (synth.normal((M, d), 1.0, dt, gen) for _ in range(3))
    w = synth.normal((d, 3 * d), synth.WEIGHT_STD, dt, gen)
    bb = synth.normal((d,), 0.1, torch.float32, gen) if bias else None
    dv = "cuda"
    g = torch.empty((M, d), dtype=dt, device=dv)
    st = torch.zeros(1, dtype=torch.int32, device=dv)
    b.eagle_fuse_proj(hl.to(dv), hm.to(dv), hh.to(dv), w.to(dv), g,
                      bias=None if bb is None else bb.to(dv), status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    rows = np.arange(M) if rows is None else np.asarray(rows)
    f = lambda t: t.float().numpy()[rows]
    ref = oracle.fuse_proj(f(hl), f(hm), f(hh), w.float().numpy(), None if bb is None else bb.numpy())
    err = rel_err(g.float().cpu().numpy()[rows], ref)
    nerr = norm_err(g.float().cpu().numpy()[rows], ref)
    print(f"fuse_proj M={M} d={d} {dtype}: rel {err:.2e}, norm-wise {nerr:.2e}")
    assert err < (1e-4 if dtype == "fp32" else REL_TOL), err
    assert nerr < (1e-5 if dtype == "fp32" else NORM_TOL), nerr


@pytest.mark.parametrize("M,d,dtype", [(17, 256, "fp32"), (1, 128, "bf16"), (61, 512, "bf16"),
                                       (300, 256, "bf16"), (5, 1024, "fp32")])
def test_fuse_proj_small(M, d, dtype):
    b = need_gpu()
    _fp_check(b, M, d, dtype, seed=M + d)


def test_fuse_proj_bias():
    b = need_gpu()
    _fp_check(b, 7, 384, "bf16", seed=11, bias=True)


@pytest.mark.parametrize("M,d,rows", [(61, 4096, None), (61, 8192, [0, 30, 60]),
                                      (576, 4096, [0, 200, 575]), (244, 4096, [0, 243])])
def test_fuse_proj_full_size(M, d, rows):
    b = need_gpu()
    _fp_check(b, M, d, "bf16", seed=M * d % 1000, rows=rows)

