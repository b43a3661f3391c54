"""Pins of oracle.verify_stats / oracle.tree_verify_stats (the follow-on path
in which stochastic verification reads statistics of the verification LM
head instead of the [B, R, V] target logits)."""
import numpy as np
import pytest
from scipy.special import logsumexp

import oracle
from oracle.philox import race_uniforms


def _case(seed, B, R, V, d, depth, T, lift=True):
    rng = np.random.default_rng(seed)
    x = rng.normal(0, 1, (B * R, d))
    w = rng.normal(0, 0.3, (V, d))
    parent = np.zeros((B, R), np.int64)
    token = np.zeros((B, R), np.int64)
    for b in range(B):
        parent[b, 0] = -1
        depth_of = [0]
        for c in range(1, R):
            cand = [i for i in range(c) if depth_of[i] < depth]
            p = int(rng.choice(cand))
            parent[b, c] = p
            depth_of.append(depth_of[p] + 1)
        for r in range(R):
            ch = [c for c in range(1, R) if parent[b, c] == r]
            toks = rng.choice(V, size=len(ch), replace=False)
            for c, t in zip(ch, toks):
                token[b, c] = t
    if lift:  # make acceptances likely: point each row's top logits at its children
        for b in range(B):
            for c in range(1, R):
                r = parent[b, c]
                w[token[b, c]] += 2.0 * x[b * R + r] / np.linalg.norm(x[b * R + r])
    return x, w, parent, token


def test_row_statistics_are_logsumexp():
    x, w, parent, token = _case(1, 2, 9, 50, 16, 3, 0.7)
    st = oracle.verify_stats(x, w, parent, token, 0.7, race_k=4, seed=3)
    y = (x @ w.T) / 0.7
    np.testing.assert_allclose(st["row_max"] + np.log(st["row_sumexp"]), logsumexp(y, axis=1),
                               rtol=0, atol=1e-12)
    # fp64 dot products in a different summation order than the matrix product
    np.testing.assert_allclose(st["row_max"], y.max(axis=1), rtol=1e-12, atol=1e-12)


def test_child_logits_are_the_dot_products():
    x, w, parent, token = _case(2, 3, 11, 40, 8, 4, 1.0)
    st = oracle.verify_stats(x, w, parent, token, 1.0, race_k=4)
    B, R = parent.shape
    for b in range(B):
        assert st["child_logit"][b * R] == 0.0
        for c in range(1, R):
            want = float(np.dot(x[b * R + parent[b, c]], w[token[b, c]]))
            assert abs(st["child_logit"][b * R + c] - want) < 1e-12


def test_race_winner_matches_full_race_over_log_probabilities():
    # first race candidate = argmax_y log p_y - log(-log u_y) over all ids,
    # computed from the per-request race uniforms and the full distribution
    x, w, parent, token = _case(3, 2, 6, 64, 12, 2, 0.8)
    seed, off = 11, 5
    st = oracle.verify_stats(x, w, parent, token, 0.8, race_k=5, seed=seed, offset=off)
    B, R = parent.shape
    for b in range(B):
        u = race_uniforms(seed, off, b, 64)
        for r in range(R):
            logp = (x[b * R + r] @ w.T) / 0.8
            logp = logp - logsumexp(logp)
            key = logp - np.log(-np.log(u))
            assert st["race_ids"][b * R + r, 0] == int(np.argmax(key))
            # keys sorted descending, ids are the top ones
            ks = st["race_keys"][b * R + r]
            assert np.all(np.diff(ks) <= 0)
            assert set(st["race_ids"][b * R + r]) == set(np.argsort(-key)[:5])


@pytest.mark.parametrize("seed", range(12))
def test_walk_from_statistics_equals_walk_on_full_logits(seed):
    T = [0.6, 1.0, 1.3][seed % 3]
    B, R, V, depth = 3, 13, 48, 4
    x, w, parent, token = _case(100 + seed, B, R, V, 10, depth, T)
    z = (x @ w.T).reshape(B, R, V)
    n_rows = np.array([R, R - 3, 7])
    ref = oracle.tree_verify(parent, token, T, depth, n_rows=n_rows, target_logits=z,
                             seed=seed, offset=2)
    kmax = max(int(np.sum(parent[b, 1:] == r)) for b in range(B) for r in range(R))
    st = oracle.verify_stats(x, w, parent, token, T, race_k=kmax + 1, seed=seed, offset=2,
                             n_rows=n_rows)
    got = oracle.tree_verify_stats(parent, token, T, depth, st["row_max"], st["row_sumexp"],
                                   st["child_logit"], st["race_ids"], n_rows=n_rows, seed=seed,
                                   offset=2)
    for k in ("accept_len", "path_rows", "out_tokens"):
        np.testing.assert_array_equal(got[k], ref[k])
    assert int(ref["accept_len"].max()) >= 1  # the case exercises acceptance


def test_race_k_too_small_is_refused():
    x, w, parent, token = _case(5, 1, 7, 30, 6, 1, 1.0, lift=False)
    # depth-1 tree: every child hangs off the root.  Give one child's token
    # the largest race key and reject every child: with race_k = 1 the only
    # candidate is rejected, which must be refused rather than guessed.
    ru = np.full((1, 30), 0.5)
    ru[0, int(token[0, 1])] = 1.0 - 1e-12
    st = oracle.verify_stats(x, w, parent, token, 1.0, race_k=1, race_u=ru)
    assert int(st["race_ids"][0, 0]) == int(token[0, 1])
    u = np.full((1, 7), 0.999999)
    with pytest.raises(ValueError):
        oracle.tree_verify_stats(parent, token, 1.0, 1, st["row_max"], st["row_sumexp"],
                                 st["child_logit"], st["race_ids"], accept_u=u)
    st2 = oracle.verify_stats(x, w, parent, token, 1.0, race_k=7, race_u=ru)
    out = oracle.tree_verify_stats(parent, token, 1.0, 1, st2["row_max"], st2["row_sumexp"],
                                   st2["child_logit"], st2["race_ids"], accept_u=u)
    assert int(out["out_tokens"][0, 0]) not in set(token[0, 1:].tolist())


def test_validation():
    x, w, parent, token = _case(6, 1, 4, 10, 4, 2, 1.0)
    with pytest.raises(ValueError):
        oracle.verify_stats(x, w, parent, token, 0.0, race_k=2)
    with pytest.raises(ValueError):
        oracle.verify_stats(x, w, parent, token, 1.0, race_k=0)
    with pytest.raises(ValueError):
        oracle.verify_stats(x[:3], w, parent, token, 1.0, race_k=2)


def test_row_subset_matches_full():
    x, w, parent, token = _case(7, 2, 8, 40, 6, 3, 0.9)
    full = oracle.verify_stats(x, w, parent, token, 0.9, race_k=3, seed=4)
    sub = oracle.verify_stats(x, w, parent, token, 0.9, race_k=3, seed=4, rows=[1, 9, 15])
    for r in (1, 9, 15):
        for k in ("row_max", "row_sumexp", "child_logit"):
            assert sub[k][r] == full[k][r]
        np.testing.assert_array_equal(sub["race_ids"][r], full["race_ids"][r])
    assert np.isnan(sub["row_max"][0])
