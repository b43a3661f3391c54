"""Pins of the oracle's fusion over the accepted rows (the publish step's
projection: only the verified path's features are fused for the next draft
round, "M7.5" 0x05D "Feature And KV Commit"; "EAGLE-3" "Stage 2:
Verification")."""
import numpy as np
import pytest
import torch

import oracle
from eagle_speculative_decoding_gb300 import synth


def _rand(shape, seed):
    return synth.normal(shape, 1.0, torch.float32, synth.generator(seed)).double().numpy()


def _case(B=3, R=6, d=4, slots=4, seed=0):
    hl, hm, hh = (_rand((B * R, d), seed + i) for i in range(3))
    w = _rand((d, 3 * d), seed + 3)
    path = np.array([[0, 2, 5, -1], [0, -1, -1, -1], [0, 1, 3, 4]])[:B, :slots]
    acc = np.array([2, 0, 3])[:B]
    return hl, hm, hh, w, path, acc


def test_bruteforce_sums_per_accepted_slot():
    hl, hm, hh, w, path, acc = _case()
    B, R, d = 3, 6, 4
    g = oracle.fuse_proj_accepted(hl, hm, hh, w, path, acc)
    assert g.shape == (B, 4, d)
    for b in range(B):
        for j in range(4):
            for o in range(d):
                if j > acc[b]:
                    assert g[b, j, o] == 0.0
                    continue
                r = b * R + path[b, j]
                s = 0.0
                for c in range(d):
                    s += w[o, c] * hl[r, c] + w[o, d + c] * hm[r, c] + w[o, 2 * d + c] * hh[r, c]
                assert abs(g[b, j, o] - s) < 1e-12


def test_equals_the_full_projection_restricted_to_the_path():
    hl, hm, hh, w, path, acc = _case(seed=10)
    R = 6
    full = np.concatenate([hl, hm, hh], axis=1) @ w.T  # every row, then select
    g = oracle.fuse_proj_accepted(hl, hm, hh, w, path, acc)
    for b in range(3):
        for j in range(acc[b] + 1):
            np.testing.assert_allclose(g[b, j], full[b * R + path[b, j]], rtol=1e-13, atol=1e-13)


def test_identity_weight_gathers_h_low_in_path_order():
    hl, hm, hh, _, path, acc = _case(seed=20)
    d, R = 4, 6
    I, Z = np.eye(d), np.zeros((d, d))
    g = oracle.fuse_proj_accepted(hl, hm, hh, np.hstack([I, Z, Z]), path, acc)
    assert np.array_equal(g[0, :3], hl[[0, 2, 5]])
    assert np.array_equal(g[2, :4], hl[[2 * R + 0, 2 * R + 1, 2 * R + 3, 2 * R + 4]])
    assert np.array_equal(g[1, 1:], np.zeros((3, d)))


def test_commit_gather_then_projection_is_the_same_map():
    """The commit's gathered features ([B, Dmax+1, 3d], zeros past the path)
    projected row by row give the same result: gather and projection commute."""
    hl, hm, hh, w, path, acc = _case(seed=30)
    B, R, d = 3, 6, 4
    feats = np.concatenate([hl, hm, hh], axis=1)
    kc = np.zeros((8, 16, 1, 2))
    table = np.arange(6).reshape(3, 2)
    ctx = np.zeros(3, np.int64)
    kt = np.zeros((B, R, 1, 2))
    gathered = oracle.tree_commit(kc, kc, table, ctx, kt, kt, path, acc, features=feats)["features"]
    g = oracle.fuse_proj_accepted(hl, hm, hh, w, path, acc)
    for b in range(B):
        n = acc[b] + 1
        np.testing.assert_allclose(g[b, :n], gathered[b, :n] @ w.T, rtol=1e-13, atol=1e-13)


def test_invalid_paths_raise():
    hl, hm, hh, w, path, acc = _case()
    with pytest.raises(ValueError):
        oracle.fuse_proj_accepted(hl, hm, hh, w, path, np.array([2, 4, 3]))  # beyond the slots
    bad = path.copy()
    bad[0, 1] = 6  # row R does not exist
    with pytest.raises(ValueError):
        oracle.fuse_proj_accepted(hl, hm, hh, w, bad, acc)
