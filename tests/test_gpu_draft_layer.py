"""GPU parity of eagle_linear and eagle_draft_layer against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from eagle_speculative_decoding_gb300 import synth
from gpu_helpers import REL_TOL, need_gpu, rel_err

pytestmark = pytest.mark.gpu


def _bf16_store(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(torch.bfloat16).double().numpy()


# One activation group with a host row count runs one cluster of cs CTAs per
# 128-row output tile when the clusters fill at least 4/5 of the SMs (on a
# 152-SM GPU): cs = 4 for the 32 tiles of the down projection, 2 for 64
# tiles, 1 (whole tiles, no split) for 128 tiles over 4 K chunks; the others
# (the drafter's 48-tile QKV among them) take the stream-K split.
@pytest.mark.parametrize("M,n_out,k_in,dtype,bias,res", [
    (1, 128, 64, "bf16", False, False),
    (10, 6144, 4096, "bf16", False, False),     # QKV projection, llama8b drafter: stream-K
    (10, 4096, 14336, "bf16", False, True),     # down projection + residual: clusters of four
    (10, 1536, 4096, "bf16", True, True),       # 12 tiles: stream-K
    (10, 8192, 1024, "bf16", False, True),      # 64 tiles: clusters of two
    (7, 3072, 2048, "bf16", True, False),       # 24 tiles: stream-K
    (20, 16384, 256, "bf16", True, False),      # 128 tiles: one CTA per tile
    (20, 12288, 256, "bf16", True, False),      # 96 tiles, 4 K chunks: stream-K
    (37, 384, 320, "bf16", True, True),
    (300, 256, 192, "bf16", False, True),       # two activation groups (lockstep lanes)
    (1000, 1024, 512, "bf16", True, False),     # four groups
    (2048, 512, 256, "bf16", False, True),      # eight groups
    (512, 4096, 2048, "bf16", True, True),      # two groups of 256 rows over pairs of output tiles
    (700, 4096, 2048, "bf16", False, True),     # three groups of 240 rows, pairs of output tiles
    (17, 256, 128, "fp32", True, True),
])
def test_linear(M, n_out, k_in, dtype, bias, res):
    b = need_gpu()
    gen = synth.generator(M + n_out + k_in)
    dt = synth.torch_dtype(dtype)
    x = synth.normal((M, k_in), 1.0, dt, gen)
    w = synth.normal((n_out, k_in), synth.WEIGHT_STD, dt, gen)
    bb = synth.normal((n_out,), 0.1, torch.float32, gen) if bias else None
    rr = synth.normal((M, n_out), 1.0, dt, gen) if res else None
    y = torch.empty((M, n_out), dtype=dt, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    b.eagle_linear(x.cuda(), w.cuda(), y, bias=None if bb is None else bb.cuda(),
                   residual=None if rr is None else rr.cuda(), status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = oracle.linear(x.double().numpy(), w.double().numpy(), None if bb is None else bb.numpy(),
                        None if rr is None else rr.double().numpy())
    err = rel_err(y.double().cpu().numpy(), ref)
    assert err < (1e-4 if dtype == "fp32" else REL_TOL), err


def test_linear_residual_in_place():
    b = need_gpu()
    gen = synth.generator(3)
    x = synth.normal((8, 256), 1.0, torch.bfloat16, gen).cuda()
    w = synth.normal((256, 256), synth.WEIGHT_STD, torch.bfloat16, gen).cuda()
    y = synth.normal((8, 256), 1.0, torch.bfloat16, gen).cuda()
    ref = oracle.linear(x.double().cpu().numpy(), w.double().cpu().numpy(), residual=y.double().cpu().numpy())
    b.eagle_linear(x, w, y, residual=y)
    torch.cuda.synchronize()
    assert rel_err(y.double().cpu().numpy(), ref) < REL_TOL


def _layer_inputs(B, W, d, Hq, Hkv, D, I, Rmax, r0, ctx_range, dtype, seed):
    gen = synth.generator(seed)
    dt = synth.torch_dtype(dtype)
    std = synth.WEIGHT_STD
    wts = dict(norm1=(1 + 0.1 * torch.randn(d, generator=gen)).to(dt),
               qkv=synth.normal(((Hq + 2 * Hkv) * D, d), std, dt, gen),
               o=synth.normal((d, Hq * D), std, dt, gen),
               norm2=(1 + 0.1 * torch.randn(d, generator=gen)).to(dt),
               gu=synth.normal((2 * I, d), std, dt, gen),
               down=synth.normal((d, I), std, dt, gen))
    x = synth.normal((B * W, d), 1.0, dt, gen)
    ctx = torch.randint(ctx_range[0], ctx_range[1] + 1, (B,), generator=gen, dtype=torch.int32)
    kc, vc, table = synth.paged_kv(ctx.tolist(), Hkv, D, 16, dt, gen)
    kt = synth.normal((B, Rmax, Hkv, D), 1.0, dt, gen)
    vt = synth.normal((B, Rmax, Hkv, D), 1.0, dt, gen)
    # earlier rows: a random tree over rows 0..r0-1; each new row hangs below one of them
    masks = np.zeros((B, Rmax), dtype=np.uint64)
    depth = np.zeros((B, Rmax), dtype=np.int64)
    for b in range(B):
        par = np.full(Rmax, -1)
        for r in range(1, Rmax):
            hi = r if (r < r0 or r0 == 0) else r0
            par[r] = int(torch.randint(0, hi, (1,), generator=gen))
        masks[b] = oracle.ancestor_mask(par, n_rows=r0 + W)
        for r in range(1, Rmax):
            depth[b, r] = depth[b, par[r]] + 1
    pos = np.stack([ctx.numpy()[b] + depth[b, r0:r0 + W] for b in range(B)]).astype(np.int32)
    return wts, x, ctx, kc, vc, table, kt, vt, masks, pos


@pytest.mark.parametrize("B,W,d,Hq,Hkv,D,I,Rmax,r0,ctx_range,dtype", [
    (2, 3, 256, 4, 2, 64, 256, 8, 2, (20, 40), "bf16"),
    (1, 10, 512, 8, 2, 128, 1024, 61, 11, (100, 100), "bf16"),   # depth 2 of a width-10 round
    (3, 4, 256, 4, 4, 64, 128, 16, 0, (0, 33), "bf16"),           # first depth, an empty prefix
    (2, 3, 256, 4, 2, 64, 256, 8, 2, (20, 40), "fp32"),
])
def test_draft_layer_small(B, W, d, Hq, Hkv, D, I, Rmax, r0, ctx_range, dtype):
    b = need_gpu()
    wts, x, ctx, kc, vc, table, kt, vt, masks, pos = _layer_inputs(B, W, d, Hq, Hkv, D, I, Rmax, r0, ctx_range,
                                                                    dtype, seed=B * 100 + W + d)
    dv = "cuda"
    qt_d = torch.zeros((B, Rmax, Hq, D), dtype=x.dtype, device=dv)
    kt_d, vt_d = kt.to(dv), vt.to(dv)
    out = torch.empty_like(x, device=dv)
    st = torch.zeros(1, dtype=torch.int32, device=dv)
    b.eagle_draft_layer(x.to(dv), {k: v.to(dv) for k, v in wts.items()}, torch.from_numpy(pos).to(dv),
                        kc.to(dv), vc.to(dv), table.to(dv), ctx.to(dv), qt_d, kt_d, vt_d,
                        torch.from_numpy(masks.view(np.int64)).to(dv), r0, out, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    store = _bf16_store if dtype == "bf16" else None
    f = lambda t: t.double().numpy()
    ref, knew, vnew = oracle.draft_layer(f(x), {k: f(v) for k, v in wts.items()}, pos, f(kc), f(vc),
                                         table.numpy(), ctx.numpy(), f(kt), f(vt), masks, r0, Hq, Hkv,
                                         store=store)
    tol = 1e-4 if dtype == "fp32" else REL_TOL
    assert rel_err(out.double().cpu().numpy(), ref) < tol
    kt_o, vt_o = kt_d.double().cpu().numpy(), vt_d.double().cpu().numpy()
    assert rel_err(kt_o[:, r0:r0 + W], knew) < tol
    assert rel_err(vt_o[:, r0:r0 + W], vnew) < tol
    # rows outside the new ones are untouched
    keep = [r for r in range(Rmax) if not r0 <= r < r0 + W]
    assert np.array_equal(kt_o[:, keep], f(kt)[:, keep])
    assert np.array_equal(vt_o[:, keep], f(vt)[:, keep])


def test_draft_layer_llama8b_shape():
    # the drafter of the 8B target: d 4096, 32/8 heads x 128, I 14336, a
    # 2048-token prefix, depth 3 of a width-10 round (rows 0..20 earlier)
    b = need_gpu()
    B, W, d, Hq, Hkv, D, I, Rmax, r0 = 1, 10, 4096, 32, 8, 128, 14336, 61, 21
    wts, x, ctx, kc, vc, table, kt, vt, masks, pos = _layer_inputs(B, W, d, Hq, Hkv, D, I, Rmax, r0,
                                                                    (2048, 2048), "bf16", seed=8)
    dv = "cuda"
    qt_d = torch.zeros((B, Rmax, Hq, D), dtype=x.dtype, device=dv)
    kt_d, vt_d = kt.to(dv), vt.to(dv)
    out = torch.empty_like(x, device=dv)
    st = torch.zeros(1, dtype=torch.int32, device=dv)
    b.eagle_draft_layer(x.to(dv), {k: v.to(dv) for k, v in wts.items()}, torch.from_numpy(pos).to(dv),
                        kc.to(dv), vc.to(dv), table.to(dv), ctx.to(dv), qt_d, kt_d, vt_d,
                        torch.from_numpy(masks.view(np.int64)).to(dv), r0, out, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    f = lambda t: t.double().numpy()
    ref, knew, _ = oracle.draft_layer(f(x), {k: f(v) for k, v in wts.items()}, pos, f(kc), f(vc),
                                      table.numpy(), ctx.numpy(), f(kt), f(vt), masks, r0, Hq, Hkv,
                                      store=_bf16_store)
    assert rel_err(out.double().cpu().numpy(), ref) < REL_TOL
    assert rel_err(kt_d.double().cpu().numpy()[:, r0:r0 + W], knew) < REL_TOL
