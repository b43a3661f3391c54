"""Pins of the oracle's tree verification (greedy and stochastic)."""
import itertools
import math
import os

import numpy as np
import pytest
from scipy import stats

import oracle
from eagle_speculative_decoding_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "publication_fixture.txt")


def _softmax(z, T):
    y = np.asarray(z, np.float64) / T
    w = np.exp(y - y.max())
    return w / w.sum()


# ---------------------------------------------------------------- greedy ---

def _children(parent, n, r):
    return [c for c in range(n) if parent[c] == r and c != 0]


@pytest.mark.parametrize("seed", range(8))
def test_greedy_is_longest_matching_path_bruteforce(seed):
    gen = synth.generator(seed)
    R, V = 30, 40
    parent, depth = synth.random_tree(R, 6, gen)
    tok = synth.distinct_sibling_tokens(parent, V, gen).numpy()
    z = synth.target_logits((1, R, V), gen, min_top2_gap=1e-2).numpy()
    # make most rows' argmax one of their children's tokens so paths are long
    rng = np.random.default_rng(seed)
    for r in range(R):
        ch = [c for c in range(1, R) if parent[c] == r]
        if ch and rng.random() < 0.8:
            z[0, r, tok[rng.choice(ch)]] = z[0, r].max() + 1.0
    am = z[0].argmax(axis=1)
    # brute force: every root->node path whose edges all match the parent's argmax
    best = [0]
    for node in range(R):
        path = [node]
        while path[-1] != 0:
            path.append(int(parent[path[-1]]))
        path = path[::-1]
        if all(tok[path[i + 1]] == am[path[i]] for i in range(len(path) - 1)):
            if len(path) > len(best):
                best = path
    res = oracle.tree_verify(parent.numpy()[None], tok[None], 0.0, max_depth=6, target_logits=z)
    a = len(best) - 1
    assert res["accept_len"][0] == a
    assert res["path_rows"][0, :a + 1].tolist() == best
    assert res["out_tokens"][0, :a + 1].tolist() == [int(tok[r]) for r in best[1:]] + [int(am[best[-1]])]
    # the argmax input gives the same result
    res2 = oracle.tree_verify(parent.numpy()[None], tok[None], 0.0, max_depth=6, target_argmax=am[None])
    assert np.array_equal(res2["out_tokens"], res["out_tokens"])


def test_greedy_chain_is_standard_greedy_speculative_decoding():
    R, V = 6, 10
    parent = synth.chain_tree(R).numpy()
    am = np.array([3, 4, 5, 9, 1, 2])
    tok = np.array([0, 3, 4, 6, 1, 2])  # rows 1,2 match; row 3 (6) != argmax of row 2 (5)
    res = oracle.tree_verify(parent[None], tok[None], 0.0, max_depth=5, target_argmax=am[None])
    assert res["accept_len"][0] == 2
    assert res["out_tokens"][0, :3].tolist() == [3, 4, 5]


def test_publication_fixture():
    kv = {}
    for line in open(GOLDEN):
        if line.startswith("#") or not line.strip():
            continue
        f = line.split()
        kv[f[0]] = [int(v) for v in f[1:]]
    res = oracle.tree_verify(np.array([kv["parent_row"]]), np.array([kv["token"]]), 0.0,
                             max_depth=2, target_argmax=np.array([kv["argmax"]]))
    a = int(res["accept_len"][0])
    assert a == kv["accept_len"][0]
    assert res["path_rows"][0, :a + 1].tolist() == kv["accepted_rows"] == kv["kv_rows"]
    assert res["out_tokens"][0, a] == kv["frontier_token"][0]


def test_argmax_ties_go_to_lowest_id():
    z = np.zeros((1, 2, 6), np.float32)
    z[0, 0, [2, 4]] = 5.0
    res = oracle.tree_verify(np.array([[-1, 0]]), np.array([[0, 4]]), 0.0, 1, target_logits=z)
    assert res["accept_len"][0] == 0 and res["out_tokens"][0, 0] == 2


# ------------------------------------------------ exact enumeration (V=8) ---
# Independent restatement of the accepted readings as probability
# computations: each candidate's acceptance probability times the
# probability of reaching it, and the final draw's distribution.

def _level(p, cands, proposals):
    out = np.zeros(len(p))
    acc = np.zeros(len(cands))
    reach, cur = 1.0, p.copy()
    for i, (t, qi) in enumerate(zip(cands, proposals)):
        a = min(1.0, cur[t] / qi[t]) if qi[t] > 0 else 0.0
        acc[i] = reach * a
        reach *= 1 - a
        r = np.maximum(0.0, cur - qi)
        cur = r / r.sum() if r.sum() > 0 else cur
    return acc, reach * cur


def test_enumeration_deterministic_proposals_lossless():
    rng = np.random.default_rng(1)
    V, k = 8, 3
    for _ in range(20):
        p, q = rng.dirichlet(np.ones(V)), rng.dirichlet(np.ones(V))
        cands = list(np.argsort(-q)[:k])
        acc, rest = _level(p, cands, [np.eye(V)[t] for t in cands])
        dist = rest.copy()
        for i, t in enumerate(cands):
            dist[t] += acc[i]
        assert np.abs(dist - p).max() < 1e-12


def test_enumeration_literal_draft_probability_rule_is_not_lossless_for_topk():
    # the reason deterministic top-k children use point-mass proposals
    rng = np.random.default_rng(1)
    V, k = 8, 3
    p, q = rng.dirichlet(np.ones(V)), rng.dirichlet(np.ones(V))
    cands = list(np.argsort(-q)[:k])
    acc, rest = _level(p, cands, [q] * k)
    dist = rest.copy()
    for i, t in enumerate(cands):
        dist[t] += acc[i]
    assert np.abs(dist - p).max() > 0.05


def test_enumeration_sampled_proposals_lossless_algorithm1():
    rng = np.random.default_rng(2)
    V, k = 8, 3
    for _ in range(5):
        p, q = rng.dirichlet(np.ones(V)), rng.dirichlet(np.ones(V))
        tot = np.zeros(V)
        for draw in itertools.product(range(V), repeat=k):
            w = np.prod([q[t] for t in draw])
            acc, rest = _level(p, list(draw), [q] * k)
            d = rest.copy()
            for i, t in enumerate(draw):
                d[t] += acc[i]
            tot += w * d
        assert np.abs(tot - p).max() < 1e-12


def test_enumeration_chain_is_leviathan_rule_two_levels():
    # chain of two sampled drafts: joint of the first two emitted tokens
    rng = np.random.default_rng(3)
    V = 8
    p0, q0, p1, q1 = (rng.dirichlet(np.ones(V)) for _ in range(4))
    joint = np.zeros((V, V))
    first_only = np.zeros(V)
    for t1 in range(V):
        acc, rest = _level(p0, [t1], [q0])
        first_only += q0[t1] * rest  # rejected at level 1: sequence ends after the draw
        # accepted t1: level 2 at the child row (its draft t2 ~ q1)
        for t2 in range(V):
            acc2, rest2 = _level(p1, [t2], [q1])
            d2 = rest2.copy()
            d2[t2] += acc2[0]
            joint[t1] += q0[t1] * acc[0] * q1[t2] * d2
    first = first_only + joint.sum(axis=1)
    assert np.abs(first - p0).max() < 1e-12
    # given an accepted draft t1, the next token follows p1 (the child's row)
    acc_prob = np.array([q0[t] * _level(p0, [t], [q0])[0][0] for t in range(V)])
    for t1 in range(V):
        if acc_prob[t1] > 0:
            assert np.abs(joint[t1] / acc_prob[t1] - p1).max() < 1e-12


# --------------------------------------------- oracle sampler chi-square ---

def _toy_tree(rng, V=8):
    # root with 3 children (rows 1-3), each with 2 children (rows 4-9)
    parent = np.array([-1, 0, 0, 0, 1, 1, 2, 2, 3, 3])
    R = len(parent)
    z = rng.normal(0, 1.5, (R, V)).astype(np.float32)
    zd = (z + rng.normal(0, 0.5, (R, V))).astype(np.float32)
    tok = np.zeros(R, np.int64)
    for r in range(R):
        ch = [c for c in range(1, R) if parent[c] == r]
        order = np.argsort(-zd[r], kind="stable")
        for i, c in enumerate(ch):
            tok[c] = order[i]  # top-k of the parent's draft row
    return parent, tok, z, zd


@pytest.mark.parametrize("T", [1.0, 0.6])
def test_chi_square_deterministic_mode_oracle_samples(T):
    rng = np.random.default_rng(5)
    parent, tok, z, zd = _toy_tree(rng)
    V, R = z.shape[1], len(parent)
    N = 100_000
    ru = oracle.race_uniforms_batch(123, 0, N, V)
    res = oracle.tree_verify(np.broadcast_to(parent, (N, R)), np.broadcast_to(tok, (N, R)), T,
                             max_depth=2, target_logits=np.broadcast_to(z, (N, R, V)),
                             seed=123, offset=0, race_u=lambda b: ru[b])
    out = res["out_tokens"]
    p0 = _softmax(z[0], T)
    child_of = {int(tok[c]): c for c in (1, 2, 3)}
    cats, probs = {}, {}
    for y in range(V):
        if y in child_of:
            c = child_of[y]
            pc = _softmax(z[c], T)
            for y2 in range(V):
                probs[(y, y2)] = p0[y] * pc[y2]
        else:
            probs[(y,)] = p0[y]
    obs = {key: 0 for key in probs}
    for row in out:
        key = (int(row[0]), int(row[1])) if int(row[0]) in child_of else (int(row[0]),)
        obs[key] += 1
    keys = sorted(probs)
    f_obs = np.array([obs[k] for k in keys], float)
    f_exp = np.array([probs[k] for k in keys]) * N
    assert abs(f_exp.sum() - N) < 1e-6 * N
    pval = stats.chisquare(f_obs, f_exp).pvalue
    assert pval > 1e-3


def test_chi_square_sampled_mode_one_level():
    rng = np.random.default_rng(6)
    V, k, N, T = 8, 3, 100_000, 1.0
    z = rng.normal(0, 1.5, (1 + k, V)).astype(np.float32)
    zd = (z + rng.normal(0, 0.5, (1 + k, V))).astype(np.float32)
    q = _softmax(zd[0], T)
    # children tokens are i.i.d. draws from q (the Algorithm 1 premise)
    toks = rng.choice(V, size=(N, k), p=q)
    tok = np.concatenate([np.zeros((N, 1), np.int64), toks], axis=1)
    parent = np.broadcast_to(np.array([-1, 0, 0, 0]), (N, 1 + k))
    ru = oracle.race_uniforms_batch(9, 1, N, V)
    res = oracle.tree_verify(parent, tok, T, max_depth=1, target_logits=np.broadcast_to(z, (N, 1 + k, V)),
                             draft_logits=np.broadcast_to(zd, (N, 1 + k, V)), mode="sampled",
                             seed=9, offset=1, race_u=lambda b: ru[b])
    f_obs = np.bincount(res["out_tokens"][:, 0], minlength=V).astype(float)
    f_exp = _softmax(z[0], T) * N
    assert stats.chisquare(f_obs, f_exp).pvalue > 1e-3


def test_override_uniforms_drive_decisions():
    parent = np.array([[-1, 0, 0, 1]])
    tok = np.array([[0, 1, 2, 3]])
    z = np.zeros((1, 4, 5), np.float32)
    # u = 0 accepts any candidate with p > 0: path 0 -> 1 -> 3
    res = oracle.tree_verify(parent, tok, 1.0, 3, target_logits=z, accept_u=np.zeros((1, 4)))
    assert res["path_rows"][0, :3].tolist() == [0, 1, 3]
    # u -> 1 rejects everything: the bonus is drawn from the root row without 1, 2
    res = oracle.tree_verify(parent, tok, 1.0, 3, target_logits=z, accept_u=np.full((1, 4), 1 - 2 ** -24))
    assert res["accept_len"][0] == 0 and res["out_tokens"][0, 0] not in (1, 2)


def test_validation():
    z = np.zeros((1, 3, 4), np.float32)
    with pytest.raises(ValueError):
        oracle.tree_verify(np.array([[-1, 0, 2]]), np.array([[0, 1, 2]]), 1.0, 2, target_logits=z)
    with pytest.raises(ValueError):
        oracle.tree_verify(np.array([[0, 0, 1]]), np.array([[0, 1, 2]]), 1.0, 2, target_logits=z)
    with pytest.raises(ValueError):
        oracle.tree_verify(np.array([[-1, 0, 1]]), np.array([[0, 1, 2]]), 0.0, 2, target_logits=z,
                           draft_logits=z, mode="sampled")
    with pytest.raises(ValueError, match="deeper"):
        oracle.tree_verify(np.array([[-1, 0, 1]]), np.array([[0, 0, 0]]), 0.0, 1, target_logits=z)
