"""GPU parity of eagle_fuse_proj_accepted (the fusion over the accepted rows
only, "M7.5" 0x05D "Feature And KV Commit") against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from eagle_speculative_decoding_gb300 import synth
from gpu_helpers import NORM_TOL, REL_TOL, need_gpu, norm_err, rel_err

pytestmark = pytest.mark.gpu


def _paths(B, R, depth, rng, accept=None):
    """Per request: accept_len in [0, depth] and a path of distinct rows
    starting at the root row 0 (later slots hold -1)."""
    acc = rng.integers(0, depth + 1, B) if accept is None else np.asarray(accept)
    path = np.full((B, depth + 1), -1, np.int32)
    for b in range(B):
        n = int(acc[b]) + 1
        path[b, :n] = np.concatenate([[0], rng.choice(np.arange(1, R), n - 1, replace=False)])
    return torch.from_numpy(path), torch.from_numpy(acc.astype(np.int32))


def _run(b, hs, w, path, acc, dt, bias=None, ws=None):
    dv = "cuda"
    B, slots = path.shape
    d = hs[0].shape[1]
    g = torch.full((B, slots, d), 7.0, dtype=dt, device=dv)  # stale contents must not survive
    st = torch.zeros(1, dtype=torch.int32, device=dv)
    b.eagle_fuse_proj_accepted(*(h.to(dv) for h in hs), w.to(dv), path.to(dv), acc.to(dv), g,
                               bias=None if bias is None else bias.to(dv), ws=ws, status=st)
    torch.cuda.synchronize()
    return g.float().cpu().numpy(), int(st.item())


def _check(g, hs, w, path, acc, dtype, bias=None, label=""):
    f = lambda t: t.float().numpy()
    ref = oracle.fuse_proj_accepted(f(hs[0]), f(hs[1]), f(hs[2]), f(w), path.numpy(), acc.numpy(),
                                    None if bias is None else bias.numpy())
    B = path.shape[0]
    live = np.zeros(g.shape[:2], bool)
    for bb in range(B):
        live[bb, :int(acc[bb]) + 1] = True
    assert np.all(g[~live] == 0.0)  # slots past the accepted path are zero
    err, nerr = rel_err(g[live], ref[live]), norm_err(g[live], ref[live])
    print(f"{label}: {int(live.sum())} accepted rows, rel {err:.2e}, norm-wise {nerr:.2e}")
    if dtype == "fp32":
        assert err < 1e-4 and nerr < 1e-5
    else:
        assert err < REL_TOL and nerr < NORM_TOL


def _inputs(B, R, d, dtype, seed):
    gen = synth.generator(seed)
    dt = synth.torch_dtype(dtype)
    hs = [synth.normal((B * R, d), 1.0, dt, gen) for _ in range(3)]
    w = synth.normal((d, 3 * d), synth.WEIGHT_STD, dt, gen)
    return hs, w, dt


@pytest.mark.parametrize("B,R,d,depth,dtype", [
    (1, 17, 256, 4, "fp32"),       # toy
    (1, 17, 256, 4, "bf16"),
    (5, 9, 128, 3, "bf16"),        # one output tile: stream-K over K only
    (1, 61, 4096, 6, "bf16"),      # llama8b
    (4, 61, 4096, 8, "bf16"),      # long4
    (64, 9, 4096, 4, "bf16"),      # serve64: 320 slots, two activation groups
    (40, 13, 256, 8, "bf16"),      # 360 slots
])
def test_matches_oracle(B, R, d, depth, dtype):
    b = need_gpu()
    hs, w, dt = _inputs(B, R, d, dtype, seed=B * 13 + d)
    path, acc = _paths(B, R, depth, np.random.default_rng(B + R))
    g, st = _run(b, hs, w, path, acc, dt)
    assert st == 0
    _check(g, hs, w, path, acc, dtype, label=f"B={B} R={R} d={d}")


@pytest.mark.parametrize("d", [4096, 256])
def test_live_rows_cross_the_group_boundary_on_back_to_back_calls(d):
    """Two activation groups of 160 rows (320 slots): calls whose accepted
    rows fill less than one group, exactly one group, both groups, and none,
    one after the other on one workspace (stale packed rows of a previous
    call must not leak)."""
    b = need_gpu()
    B, R, depth = 64, 9, 4
    hs, w, dt = _inputs(B, R, d, "bf16", seed=d)
    ws = b.workspace(b.eagle_fuse_proj_accepted_workspace_size(B, depth, d, b.EAGLE_BF16), "cuda")
    rng = np.random.default_rng(d)
    for accept in (np.zeros(B, int),                           # 64 rows
                   np.array([1] * 32 + [2] * 32),              # 160 rows: one full group
                   np.array([4] * 64),                         # 320 rows: every slot
                   rng.integers(0, 5, B)):
        path, acc = _paths(B, R, depth, rng, accept)
        g, st = _run(b, hs, w, path, acc, dt, ws=ws)
        assert st == 0
        _check(g, hs, w, path, acc, "bf16", label=f"d={d} total={int(acc.sum()) + B}")


def test_bias_and_invalid_request():
    """A request whose accept_len exceeds the slots projects nothing (its
    slots are zero) and raises EAGLE_ERR_BAD_TREE; the others are exact."""
    b = need_gpu()
    B, R, d, depth = 6, 9, 256, 4
    hs, w, dt = _inputs(B, R, d, "bf16", seed=5)
    bias = synth.normal((d,), 0.1, torch.float32, synth.generator(6))
    path, acc = _paths(B, R, depth, np.random.default_rng(3))
    g, st = _run(b, hs, w, path, acc, dt, bias=bias)
    assert st == 0
    _check(g, hs, w, path, acc, "bf16", bias=bias, label="bias")
    bad_acc = acc.clone()
    bad_acc[2] = depth + 1
    g, st = _run(b, hs, w, path, bad_acc, dt, bias=bias)
    assert st == 5  # EAGLE_ERR_BAD_TREE
    assert np.all(g[2] == 0.0)
    keep = [i for i in range(B) if i != 2]
    _check(g[keep], [h.view(B, R, d)[keep].reshape(-1, d) for h in hs], w, path[keep], acc[keep], "bf16",
           bias=bias, label="other requests")
