"""GPU parity of eagle_tree_commit against oracle.tree_commit (bit-exact:
the commit only moves bytes)."""
import numpy as np
import pytest
import torch

import oracle
from eagle_speculative_decoding_gb300 import synth
from gpu_helpers import need_gpu

pytestmark = pytest.mark.gpu


def _case(seed, B, R, Hkv, D, maxd, F, dt):
    gen = synth.generator(seed)
    ctx = torch.randint(0, 200, (B,), generator=gen, dtype=torch.int32)
    ctx[0] = 16  # a page boundary
    kc, vc, table = synth.paged_kv((ctx + maxd + 1).tolist(), Hkv, D, 16, dt, gen)
    kt = synth.normal((B, R, Hkv, D), 1.0, dt, gen)
    vt = synth.normal((B, R, Hkv, D), 1.0, dt, gen)
    feat = synth.normal((B * R, F), 1.0, dt, gen)
    acc = torch.randint(0, maxd + 1, (B,), generator=gen, dtype=torch.int32)
    path = torch.full((B, maxd + 1), -1, dtype=torch.int32)
    for b in range(B):
        rows = [0] + sorted(torch.randperm(R - 1, generator=gen)[:int(acc[b])].add(1).tolist())
        path[b, :len(rows)] = torch.tensor(rows, dtype=torch.int32)
    return kc, vc, table, ctx, kt, vt, feat, path, acc


@pytest.mark.parametrize("dtype,B,R,Hkv,D,maxd,F", [
    ("bf16", 5, 61, 8, 128, 6, 4096),
    ("bf16", 64, 9, 8, 128, 4, 256),
    ("fp32", 3, 17, 2, 64, 4, 64),
])
def test_commit_matches_oracle(dtype, B, R, Hkv, D, maxd, F):
    b = need_gpu()
    dt = synth.torch_dtype(dtype)
    kc, vc, table, ctx, kt, vt, feat, path, acc = _case(B + R, B, R, Hkv, D, maxd, F, dt)
    d = "cuda"
    kc_d, vc_d, ctx_d = kc.to(d), vc.to(d), ctx.to(d)
    fo = torch.full((B, maxd + 1, F), 7.0, dtype=dt, device=d)
    st = torch.zeros(1, dtype=torch.int32, device=d)
    b.eagle_tree_commit(kt.to(d), vt.to(d), path.to(d), acc.to(d), kc_d, vc_d, table.to(d), ctx_d,
                        features=feat.to(d), features_out=fo, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    f32 = lambda t: t.float().numpy()
    ref = oracle.tree_commit(f32(kc), f32(vc), table.numpy(), ctx.numpy(), f32(kt), f32(vt),
                             path.numpy(), acc.numpy(), features=f32(feat))
    assert np.array_equal(kc_d.float().cpu().numpy(), ref["k_cache"])
    assert np.array_equal(vc_d.float().cpu().numpy(), ref["v_cache"])
    assert np.array_equal(ctx_d.cpu().numpy(), ref["ctx_lens"])
    assert np.array_equal(fo.float().cpu().numpy(), ref["features"])


def test_bad_request_left_untouched():
    b = need_gpu()
    kc, vc, table, ctx, kt, vt, feat, path, acc = _case(9, 3, 9, 2, 64, 4, 64, torch.bfloat16)
    path[1, 0] = 50  # row out of range in request 1: nothing of it may be written
    d = "cuda"
    kc_d, vc_d, ctx_d = kc.to(d), vc.to(d), ctx.to(d)
    st = torch.zeros(1, dtype=torch.int32, device=d)
    b.eagle_tree_commit(kt.to(d), vt.to(d), path.to(d), acc.to(d), kc_d, vc_d, table.to(d), ctx_d,
                        status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 5  # EAGLE_ERR_BAD_TREE
    # requests 0 and 2 are committed as the oracle commits them alone (their
    # pages are disjoint from request 1's); request 1 is untouched
    g = [0, 2]
    f32 = lambda t: t.float().numpy()
    ref = oracle.tree_commit(f32(kc), f32(vc), table.numpy()[g], ctx.numpy()[g], f32(kt)[g],
                             f32(vt)[g], path.numpy()[g], acc.numpy()[g])
    assert np.array_equal(kc_d.float().cpu().numpy(), ref["k_cache"])
    assert np.array_equal(vc_d.float().cpu().numpy(), ref["v_cache"])
    got = ctx_d.cpu().numpy()
    assert got[1] == int(ctx[1]) and got[0] == ref["ctx_lens"][0] and got[2] == ref["ctx_lens"][1]
