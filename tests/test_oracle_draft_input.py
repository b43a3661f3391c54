"""Pins of the oracle's drafter input FC u = W_I [r; e(x)] (+ b).

Each pin ties the oracle to something other than its own formula: the two
halves of the concatenation recovered with identity blocks, a route through a
pre-projected token table (one-hot algebra instead of a row lookup), pure
Python loops on a tiny case, and the token-id range rule.
"""
import numpy as np
import pytest
import torch

import oracle
from eagle_speculative_decoding_gb300 import synth


def _rand(shape, seed):
    return synth.normal(shape, 1.0, torch.float32, synth.generator(seed)).double().numpy()


def test_identity_blocks_recover_feature_then_embedding():
    # [I | 0] returns r; [0 | I] returns the looked-up embedding rows: the
    # feature comes first in the concatenation, the token second
    M, d, V = 6, 8, 11
    r, E = _rand((M, d), 1), _rand((V, d), 2)
    ids = np.array([3, 0, 10, 3, 7, 1])
    I, Z = np.eye(d), np.zeros((d, d))
    assert np.array_equal(oracle.draft_input(r, ids, E, np.hstack([I, Z])), r)
    assert np.array_equal(oracle.draft_input(r, ids, E, np.hstack([Z, I])), E[ids])


def test_preprojected_token_table_route():
    # W_I [r; E[x]] = W_r r + (E W_e^T)[x]: project the whole table once and
    # pick rows by one-hot products -- no row gather on this side
    M, d, V = 7, 5, 13
    r, E, W, b = _rand((M, d), 3), _rand((V, d), 4), _rand((d, 2 * d), 5), _rand((d,), 6)
    ids = np.array([12, 0, 5, 5, 9, 2, 12])
    table = E @ W[:, d:].T             # [V, d]: every token's embedding half projected
    onehot = np.zeros((M, V))
    onehot[np.arange(M), ids] = 1.0
    expect = r @ W[:, :d].T + onehot @ table + b
    got = oracle.draft_input(r, ids, E, W, b)
    assert np.abs(got - expect).max() < 1e-12


def test_bruteforce_loops_with_bias():
    M, d, V = 3, 4, 6
    r, E, W, b = _rand((M, d), 7), _rand((V, d), 8), _rand((d, 2 * d), 9), _rand((d,), 10)
    ids = [5, 1, 5]
    u = oracle.draft_input(r, ids, E, W, b)
    for i in range(M):
        for o in range(d):
            acc = b[o]
            for c in range(d):
                acc += W[o, c] * r[i, c] + W[o, d + c] * E[ids[i], c]
            assert abs(u[i, o] - acc) < 1e-12


def test_same_token_same_feature_same_output_and_token_only_difference():
    # two rows with equal r and equal token give equal u; rows that differ
    # only in the token differ by W_e (e_a - e_b)
    d, V = 6, 9
    E, W = _rand((V, d), 11), _rand((d, 2 * d), 12)
    r = np.repeat(_rand((1, d), 13), 3, axis=0)
    u = oracle.draft_input(r, [4, 4, 7], E, W)
    assert np.array_equal(u[0], u[1])
    assert np.abs((u[0] - u[2]) - W[:, d:] @ (E[4] - E[7])).max() < 1e-12


def test_token_range_and_shape_errors():
    r, E, W = _rand((2, 4), 14), _rand((5, 4), 15), _rand((4, 8), 16)
    with pytest.raises(ValueError):
        oracle.draft_input(r, [0, 5], E, W)
    with pytest.raises(ValueError):
        oracle.draft_input(r, [-1, 0], E, W)
    with pytest.raises(ValueError):
        oracle.draft_input(r, [0, 1], E, W[:, :6])
    assert oracle.draft_input(r[:0], [], E, W).shape == (0, 4)
