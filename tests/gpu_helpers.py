"""Comparison helpers shared by the GPU parity tests (no method arithmetic)."""
import numpy as np
import pytest
import torch

REL_TOL = 2e-2     # attention / projection outputs, bf16 in, fp32 accumulate
LOGPROB_TOL = 1e-3
# Norm-wise regression bar under the stated 2e-2: a bf16 output vector
# carries rounding of about 2^-9 relative per element (~1e-3 norm-wise), and
# attention adds the bf16 rounding of P; 5e-3 leaves room for both while a
# kernel 5x less accurate than it is now fails.
NORM_TOL = 5e-3


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from eagle_speculative_decoding_gb300 import binding
    binding.lib()  # raises when the library is missing: no silent fallback
    return binding


def rel_err(gpu, ref):
    """Relative error of output vectors (the last axis: one attention head
    output or one projected feature row).  The larger of
      * max over vectors of ||g - o|| / ||o||, and
      * max over elements of |g_i - o_i| / (|o_i| + rms(o of that vector)),
    i.e. elements are measured against their own vector's scale so that
    entries near zero do not turn bf16 rounding into a large ratio."""
    g = np.asarray(gpu, np.float64)
    o = np.asarray(ref, np.float64)
    if o.size == 0:
        return 0.0
    g = g.reshape(-1, o.shape[-1])
    o = o.reshape(-1, o.shape[-1])
    norm = np.linalg.norm(g - o, axis=1) / np.maximum(np.linalg.norm(o, axis=1), 1e-30)
    rms = np.sqrt(np.mean(o * o, axis=1, keepdims=True))
    elem = np.abs(g - o) / (np.abs(o) + rms + 1e-30)
    return float(max(norm.max(), elem.max()))


def norm_err(gpu, ref):
    """max over output vectors (last axis) of ||g - o|| / ||o||."""
    g = np.asarray(gpu, np.float64)
    o = np.asarray(ref, np.float64)
    if o.size == 0:
        return 0.0
    g = g.reshape(-1, o.shape[-1])
    o = o.reshape(-1, o.shape[-1])
    return float((np.linalg.norm(g - o, axis=1) / np.maximum(np.linalg.norm(o, axis=1), 1e-30)).max())


def check_topk(gpu_ids, gpu_lp, z_ref, lp_ref_fn, k, tie_tol):
    """Top-k ids exact wherever the oracle's decision margin exceeds tie_tol;
    inside a near-tie group the GPU id must be a member of the group.  The
    GPU log-prob of the id it returned must match the oracle's for that id.
    Returns the number of positions decided inside a near-tie group."""
    near = 0
    for i in range(gpu_ids.shape[0]):
        z = z_ref[i]
        order = np.lexsort((np.arange(z.shape[0]), -z))[:k + 1]
        zs = z[order]
        for j in range(k):
            gid = int(gpu_ids[i, j])
            lo_gap = zs[j - 1] - zs[j] if j > 0 else np.inf
            hi_gap = zs[j] - zs[j + 1] if j + 1 < len(zs) else np.inf
            if min(lo_gap, hi_gap) >= tie_tol:
                assert gid == int(order[j]), (i, j, gid, int(order[j]))
            else:
                near += 1
                assert abs(z[gid] - zs[j]) < 2 * tie_tol, (i, j, gid)
            assert abs(float(gpu_lp[i, j]) - lp_ref_fn(i, gid)) < LOGPROB_TOL, (i, j)
    return near
