"""GPU parity of eagle_draft_input (u = W_I [r; e(x)] + b) against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from eagle_speculative_decoding_gb300 import synth
from gpu_helpers import REL_TOL, need_gpu, rel_err

pytestmark = pytest.mark.gpu


def _di_check(b, M, d, V, dtype, seed, rows=None, bias=False, ids=None, expect_status=0):
    gen = synth.generator(seed)
    dt = synth.torch_dtype(dtype)
    r = synth.normal((M, d), 1.0, dt, gen)
    # the table is drawn on the device (128256 x 8192 at full size); the oracle
    # gets the rows it needs, renumbered
    E = synth.normal((V, d), 1.0, dt, synth.generator(seed + 1, "cuda"), device="cuda")
    w = synth.normal((d, 2 * d), synth.WEIGHT_STD, dt, gen)
    bb = synth.normal((d,), 0.1, torch.float32, gen) if bias else None
    if ids is None:
        ids = synth.random_tokens((M,), V, gen)
    ids = torch.as_tensor(ids, dtype=torch.int32)
    dv = "cuda"
    u = torch.empty((M, d), dtype=dt, device=dv)
    st = torch.zeros(1, dtype=torch.int32, device=dv)
    b.eagle_draft_input(r.to(dv), ids.to(dv), E, w.to(dv), u,
                        bias=None if bb is None else bb.to(dv), status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == expect_status
    rows = np.arange(M) if rows is None else np.asarray(rows)
    ids_np = ids.numpy()[rows]
    valid = (ids_np >= 0) & (ids_np < V)
    # an out-of-range id reads as a zero embedding on the device: compare
    # those rows against the oracle with an all-zero table row
    used = np.unique(ids_np[valid])
    sub = E[torch.as_tensor(used, dtype=torch.long, device=dv)].float().cpu().numpy()
    table = np.concatenate([sub, np.zeros((1, d))], axis=0)
    ids_ref = np.where(valid, np.searchsorted(used, ids_np), len(used))
    ref = oracle.draft_input(r.float().numpy()[rows], ids_ref, table, w.float().numpy(),
                             None if bb is None else bb.numpy())
    err = rel_err(u.float().cpu().numpy()[rows], ref)
    assert err < (1e-4 if dtype == "fp32" else REL_TOL), err


@pytest.mark.parametrize("M,d,V,dtype", [
    (1, 128, 50, "bf16"),       # one row, one output tile
    (10, 512, 1000, "bf16"),    # draft rows of one request, ragged bn tail
    (37, 384, 4097, "bf16"),    # odd M, three output tiles
    (300, 256, 3000, "bf16"),   # two activation groups (bn 160)
    (600, 256, 700, "bf16"),    # three activation groups, repeated tokens
    (17, 256, 300, "fp32"),
    (5, 1024, 64, "fp32"),
])
def test_draft_input_small(M, d, V, dtype):
    b = need_gpu()
    _di_check(b, M, d, V, dtype, seed=M * 7 + d)


def test_draft_input_bias_and_edge_tokens():
    b = need_gpu()
    V = 777
    ids = [0, V - 1, 5, 5, 0, V - 1, 400, 3, 2]
    _di_check(b, 9, 384, V, "bf16", seed=5, bias=True, ids=ids)


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_draft_input_bad_token_id(dtype):
    # ids outside [0, vocab) record EAGLE_ERR_BAD_TREE; such a row keeps its
    # feature half, the other rows are unaffected
    b = need_gpu()
    ids = [3, -1, 7, 99, 1, 100000]
    _di_check(b, 6, 256, 99, dtype, seed=9, ids=ids, expect_status=5)


@pytest.mark.parametrize("M,d,rows", [
    (10, 4096, None),                  # llama8b: width-10 frontier of one request
    (128, 4096, [0, 63, 64, 127]),     # serve64: 64 requests x width 2
    (32, 4096, [0, 17, 31]),           # long4: 4 requests x width 8
    (10, 8192, [0, 9]),                # llama70b
    (61, 4096, [0, 30, 60]),           # first draft step over the accepted rows
])
def test_draft_input_full_size(M, d, rows):
    b = need_gpu()
    _di_check(b, M, d, 128256, "bf16", seed=M + d, rows=rows)
