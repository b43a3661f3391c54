"""GPU parity of eagle_tree_attn against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from eagle_speculative_decoding_gb300 import synth
from gpu_helpers import NORM_TOL, REL_TOL, need_gpu, norm_err, rel_err

pytestmark = pytest.mark.gpu


def _case(seed, B, R, Hq, Hkv, D, ctx_lo, ctx_hi, dtype, depth=6, chain=False):
    gen = synth.generator(seed)
    dt = synth.torch_dtype(dtype)
    ctx = torch.randint(ctx_lo, ctx_hi + 1, (B,), generator=gen, dtype=torch.int32)
    q = synth.normal((B, R, Hq, D), 1.0, dt, gen)
    kt = synth.normal((B, R, Hkv, D), 1.0, dt, gen)
    vt = synth.normal((B, R, Hkv, D), 1.0, dt, gen)
    kc, vc, table = synth.paged_kv(ctx.tolist(), Hkv, D, 16, dt, gen)
    masks = []
    for _ in range(B):
        p = synth.chain_tree(R) if chain else synth.random_tree(R, depth, gen)[0]
        masks.append(oracle.ancestor_mask(p.numpy()).astype(np.int64))
    mask = torch.from_numpy(np.stack(masks))
    return q, kt, vt, kc, vc, table, ctx, mask


def _gpu(b, q, kt, vt, kc, vc, table, ctx, mask, num_splits=0):
    d = "cuda"
    out = torch.empty_like(q, device=d)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=d)
    st = torch.zeros(1, dtype=torch.int32, device=d)
    b.eagle_tree_attn(q.to(d), kt.to(d), vt.to(d), kc.to(d), vc.to(d), table.to(d), ctx.to(d),
                      mask.to(d), out, lse=lse, num_splits=num_splits, status=st)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), lse.cpu().numpy(), int(st.item())


def _ref(q, kt, vt, kc, vc, table, ctx, mask, sample=None):
    f = lambda t: t.float().numpy()
    return oracle.tree_attn(f(q), f(kt), f(vt), f(kc), f(vc), table.numpy(), ctx.numpy(),
                            mask.numpy().astype(np.uint64), sample=sample)


@pytest.mark.parametrize("B,R,Hq,Hkv,D,lo,hi,splits", [
    (1, 17, 4, 2, 64, 128, 128, 0),       # toy shape in bf16
    (2, 13, 8, 2, 128, 1, 300, 0),        # ragged, page tails
    (3, 61, 32, 8, 128, 0, 200, 0),       # empty prefix allowed
    (2, 9, 32, 8, 128, 500, 900, 3),      # forced splits
    (1, 64, 16, 1, 128, 100, 100, 0),     # G = 16, R = 64
    (4, 5, 4, 4, 64, 33, 97, 2),          # MHA, D = 64
    (2, 20, 12, 4, 128, 50, 400, 0),      # G = 3: 42 tree rows x 3 heads per tile
    (3, 33, 10, 2, 64, 0, 260, 0),        # G = 5, rows spill into a second tile
    (1, 61, 32, 8, 128, 2048, 2048, 16),  # many splits, full pages
])
def test_bf16_small_cases(B, R, Hq, Hkv, D, lo, hi, splits):
    b = need_gpu()
    case = _case(B * 31 + R, B, R, Hq, Hkv, D, lo, hi, "bf16")
    out, lse, st = _gpu(b, *case, num_splits=splits)
    ref_o, ref_l = _ref(*case)
    assert st == 0
    err, nerr = rel_err(out, ref_o), norm_err(out, ref_o)
    print(f"B={B} R={R} Hq={Hq} D={D}: rel {err:.2e}, norm-wise {nerr:.2e}")
    assert err < REL_TOL and nerr < NORM_TOL
    assert np.abs(lse - ref_l).max() < 2e-2


@pytest.mark.parametrize("B,R,Hq,Hkv,D,lo,hi", [
    (1, 17, 4, 2, 64, 128, 128),
    (2, 13, 8, 2, 128, 1, 300),
    (3, 61, 32, 8, 128, 0, 200),       # empty prefixes: units of the tree block only
    (1, 64, 16, 1, 128, 100, 100),
    (4, 5, 4, 4, 64, 33, 97),
    (2, 20, 12, 4, 128, 50, 400),
    (3, 33, 10, 2, 64, 0, 260),
    (40, 9, 32, 8, 128, 0, 700),       # many requests: segments cross requests, some empty
    (3, 32, 8, 4, 128, 10, 500),       # two-copy tile of 64 rows per copy, 32-row tree block
    (2, 61, 32, 8, 128, 4000, 5000),   # two query tiles per unit
])
def test_bf16_stream_schedule(B, R, Hq, Hkv, D, lo, hi):
    """The persistent stream schedule (num_splits = -1) on shapes the
    automatic choice gives to the split schedule: units split between CTAs,
    merged pieces, segments crossing requests."""
    b = need_gpu()
    case = _case(B * 37 + R + 1, B, R, Hq, Hkv, D, lo, hi, "bf16")
    out, lse, st = _gpu(b, *case, num_splits=-1)
    ref_o, ref_l = _ref(*case)
    assert st == 0
    err, nerr = rel_err(out, ref_o), norm_err(out, ref_o)
    print(f"stream B={B} R={R} Hq={Hq} D={D}: rel {err:.2e}, norm-wise {nerr:.2e}")
    assert err < REL_TOL and nerr < NORM_TOL
    assert np.abs(lse - ref_l).max() < 2e-2


def test_chain_tree_bf16():
    b = need_gpu()
    case = _case(7, 1, 12, 8, 2, 128, 77, 77, "bf16", chain=True)
    out, lse, st = _gpu(b, *case)
    ref_o = _ref(*case)[0]
    assert rel_err(out, ref_o) < REL_TOL and norm_err(out, ref_o) < NORM_TOL


def test_toy_fp32():
    b = need_gpu()
    c = synth.CONFIGS["toy"]
    case = _case(3, 1, c["N"] + 1, c["Hq"], c["Hkv"], c["D"], 128, 128, "fp32", depth=4)
    out, lse, st = _gpu(b, *case)
    ref_o, ref_l = _ref(*case)
    assert st == 0
    assert rel_err(out, ref_o) < 1e-4
    assert np.abs(lse - ref_l).max() < 1e-4


def test_bad_page_id_reported():
    b = need_gpu()
    q, kt, vt, kc, vc, table, ctx, mask = _case(9, 1, 4, 4, 2, 64, 40, 40, "bf16")
    table[0, 1] = kc.shape[0] + 5
    out, lse, st = _gpu(b, q, kt, vt, kc, vc, table, ctx, mask)
    assert st == 6


@pytest.mark.parametrize("cfg", ["llama8b", "llama70b", "serve64", "long4", "chain3"])
def test_full_size_sampled(cfg):
    b = need_gpu()
    c = synth.CONFIGS[cfg]
    B, R = c["B"], c["N"] + 1
    case = _case(sum(map(ord, cfg)), B, R, c["Hq"], c["Hkv"], c["D"], c["ctx"][0], c["ctx"][1], "bf16",
                 depth=c["depth"])
    out, lse, st = _gpu(b, *case)
    assert st == 0
    rng = np.random.default_rng(0)
    sample = [(int(rng.integers(B)), int(rng.integers(R)), int(rng.integers(c["Hq"]))) for _ in range(24)]
    sample += [(B - 1, R - 1, c["Hq"] - 1), (0, 0, 0)]
    ref = _ref(*case, sample=sample)
    got = np.stack([out[s] for s in sample])
    want = np.stack([ref[s][0] for s in sample])
    err, nerr = rel_err(got, want), norm_err(got, want)
    print(f"{cfg}: rel {err:.2e}, norm-wise {nerr:.2e}")
    assert err < REL_TOL and nerr < NORM_TOL
    assert max(abs(lse[s] - ref[s][1]) for s in sample) < 2e-2
