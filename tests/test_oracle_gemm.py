"""Pins of the oracle's fused projection and LM-head top-k."""
import math

import numpy as np
import pytest
import torch

import oracle
from eagle_speculative_decoding_gb300 import synth


def _rand(shape, seed):
    return synth.normal(shape, 1.0, torch.float32, synth.generator(seed)).double().numpy()


def test_fuse_proj_concat_order_low_mid_high():
    M, d = 5, 8
    hl, hm, hh = _rand((M, d), 1), _rand((M, d), 2), _rand((M, d), 3)
    I, Z = np.eye(d), np.zeros((d, d))
    assert np.array_equal(oracle.fuse_proj(hl, hm, hh, np.hstack([I, Z, Z])), hl)
    assert np.array_equal(oracle.fuse_proj(hl, hm, hh, np.hstack([Z, I, Z])), hm)
    assert np.array_equal(oracle.fuse_proj(hl, hm, hh, np.hstack([Z, Z, I])), hh)


def test_fuse_proj_bruteforce_sum_and_bias():
    M, d = 3, 4
    hl, hm, hh = _rand((M, d), 4), _rand((M, d), 5), _rand((M, d), 6)
    w, b = _rand((d, 3 * d), 7), _rand((d,), 8)
    g = oracle.fuse_proj(hl, hm, hh, w, b)
    for i in range(M):
        for o in range(d):
            acc = b[o]
            for c in range(d):
                acc += w[o, c] * hl[i, c] + w[o, d + c] * hm[i, c] + w[o, 2 * d + c] * hh[i, c]
            assert abs(g[i, o] - acc) < 1e-12


def test_lmhead_topk_bruteforce_ranks_and_normaliser():
    M, d, V, k = 3, 6, 40, 5
    x, w = _rand((M, d), 9), _rand((V, d), 10)
    res = oracle.lmhead_topk(x, w, k, temperature=0.7)
    for i in range(M):
        z = [sum(w[v, c] * x[i, c] for c in range(d)) for v in range(V)]
        # rank by pairwise comparison: count ids strictly ahead in (z desc, id asc)
        rank = [sum(1 for u in range(V) if (z[u] > z[v]) or (z[u] == z[v] and u < v)) for v in range(V)]
        expect = sorted(range(V), key=lambda v: rank[v])[:k]
        assert res["ids"][i].tolist() == expect
        lse = math.log(sum(math.exp(zz / 0.7) for zz in z))
        for j, v in enumerate(expect):
            assert abs(res["logprobs"][i, j] - (z[v] / 0.7 - lse)) < 1e-12
        assert abs(res["row_max"][i] - max(z) / 0.7) < 1e-12
        assert abs(res["row_max"][i] + math.log(res["row_sumexp"][i]) - lse) < 1e-12
    # full-vocabulary log-probs sum to one
    full = oracle.lmhead_topk(x, w, V)
    assert np.abs(np.exp(full["logprobs"]).sum(axis=1) - 1).max() < 1e-12


def test_lmhead_ties_to_lower_id_and_one_hot_row():
    d, V = 4, 10
    w = np.zeros((V, d))
    w[7] = [1, 0, 0, 0]
    w[3] = [1, 0, 0, 0]  # exact tie with row 7
    w[5] = [0.5, 0, 0, 0]
    x = np.array([[2.0, 0, 0, 0]])
    res = oracle.lmhead_topk(x, w, 3)
    assert res["ids"][0].tolist() == [3, 7, 5]


def test_lmhead_bias_and_temperature():
    M, d, V = 2, 5, 30
    x, w, b = _rand((M, d), 11), _rand((V, d), 12), _rand((V,), 13)
    r1 = oracle.lmhead_topk(x, w, 4, bias=b)
    z = x @ w.T + b
    assert np.array_equal(r1["ids"], np.argsort(-z, axis=1, kind="stable")[:, :4])
    r2 = oracle.lmhead_topk(x, w, 4, bias=b, temperature=2.0)
    assert np.array_equal(r1["ids"], r2["ids"])  # order independent of T
    # the argmax loses probability as T grows (softmax(z/T) flattens)
    assert np.all(r2["logprobs"][:, 0] <= r1["logprobs"][:, 0] + 1e-12)
    with pytest.raises(ValueError):
        oracle.lmhead_topk(x, w, 0)
    with pytest.raises(ValueError):
        oracle.lmhead_topk(x, w, 2, temperature=0.0)


def test_lmhead_masked_ids_follow_by_ascending_id():
    """A -inf bias removes an id from the softmax: the normaliser is the one
    of the allowed ids alone, and a list longer than the allowed set ends with
    masked ids in ascending order at log-prob -inf (the (z desc, id asc)
    order with z = -inf for all of them)."""
    d, V, k = 6, 24, 6
    x, w = _rand((2, d), 14), _rand((V, d), 15)
    allowed = [19, 4, 11]
    bias = np.full(V, -np.inf)
    bias[allowed] = 0.0
    res = oracle.lmhead_topk(x, w, k, bias=bias)
    for i in range(2):
        z = {v: float(x[i] @ w[v]) for v in allowed}
        fin = sorted(allowed, key=lambda v: (-z[v], v))
        masked = [v for v in range(V) if v not in allowed][:k - len(allowed)]
        assert res["ids"][i].tolist() == fin + masked
        lse = math.log(sum(math.exp(z[v]) for v in allowed))
        for j, v in enumerate(fin):
            assert abs(res["logprobs"][i, j] - (z[v] - lse)) < 1e-12
        assert np.all(np.isneginf(res["logprobs"][i, len(allowed):]))
        assert abs(res["row_max"][i] + math.log(res["row_sumexp"][i]) - lse) < 1e-12
