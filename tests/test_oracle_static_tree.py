"""Pins of the oracle's static (EAGLE-1) tree step: node counts and child
tokens of the 4-3-2-1 schedule, equality with the dynamic expansion when
every node keeps all k children (as sets of root paths with their values),
the greedy chain, the flatten of a whole static tree, and argument errors."""
import math

import numpy as np
import pytest

import oracle

V = 1000


def _cands(parents, k):
    """Deterministic drafter output: parent p's rank-i token and log-prob."""
    ids = np.array([[(p * 7 + i * 13 + 1) % V for i in range(k)] for p in parents], dtype=np.int64)
    lps = np.array([[math.log(0.45 * 0.5 ** i) for i in range(k)] for _ in parents], dtype=np.float32)
    return ids, lps


def _grow_static(schedule, k):
    st = oracle.tree_expand_init(5)
    for f in schedule:
        par = list(st["frontier"])
        ids, lps = _cands(par, k)
        oracle.static_tree_step(st, ids, lps, [f] * len(par))
    return st


def test_schedule_4321_counts_tokens_depths():
    k = 4
    st = _grow_static([4, 3, 2, 1], k)
    assert len(st["parent"]) == 1 + 4 + 12 + 24 + 24
    depth = np.array(st["depth"])
    assert [int((depth == s).sum()) for s in range(5)] == [1, 4, 12, 24, 24]
    # every node's children are its top-f candidates, in rank order
    kids = {}
    for n in range(1, len(st["parent"])):
        kids.setdefault(st["parent"][n], []).append(n)
    fan = {0: 4, 1: 3, 2: 2, 3: 1}
    for p, ch in kids.items():
        f = fan[st["depth"][p]]
        assert len(ch) == f
        ids, _ = _cands([p], k)
        assert [st["token"][c] for c in ch] == list(ids[0, :f])
    assert sorted(st["frontier"]) == [n for n in range(len(depth)) if depth[n] == 4]


def _paths(st):
    out = {}
    for n in range(1, len(st["parent"])):
        path, m = [], n
        while m != 0:
            path.append(st["token"][m])
            m = st["parent"][m]
        out[tuple(reversed(path))] = float(st["logv"][n])
    return out


def test_full_fanout_equals_dynamic_expansion_keeping_everything():
    k, depth = 3, 3
    stat = _grow_static([k] * depth, k)
    # dynamic EAGLE-2 expansion: the drafter's candidates depend only on the
    # parent's (token path), so give it the same function of the path
    stat_paths = _paths(stat)
    path_of = lambda st, n: tuple(reversed([st["token"][m] for m in _walk(st, n)]))

    def draft_fn(st):
        def f(_step, parents):
            rows = [stat_node[path_of(st, p)] if p else 0 for p in parents]
            return _cands(rows, k)
        return f

    stat_node = {(): 0}
    for n in range(1, len(stat["parent"])):
        stat_node[path_of(stat, n)] = n
    dyn = oracle.tree_expand_init(5)
    f = draft_fn(dyn)
    for step in range(depth):
        ids, lps = f(step, list(dyn["frontier"]))
        oracle.tree_expand_step(dyn, ids, lps, 10 ** 6)
    assert _paths(dyn) == stat_paths


def _walk(st, n):
    while n != 0:
        yield n
        n = st["parent"][n]


def test_chain_is_greedy():
    st = _grow_static([1, 1, 1, 1], 3)
    toks, p = [], 0
    for _ in range(4):
        ids, _ = _cands([p], 3)
        toks.append(int(ids[0, 0]))
        p = [n for n in range(1, len(st["parent"])) if st["parent"][n] == p][0]
    assert [st["token"][n] for n in range(1, 5)] == toks


def test_flatten_keeps_a_whole_static_tree_with_siblings_in_rank_order():
    st = _grow_static([3, 2, 1], 3)
    n = len(st["parent"]) - 1
    flat = oracle.tree_expand_finalize(st, n, ctx_len=40)
    assert flat["n_rows"] == n + 1
    assert sorted(flat["node_id"][1:].tolist()) == list(range(1, n + 1))
    assert np.array_equal(flat["mask"], oracle.ancestor_mask(flat["parent_row"]))
    for p in range(n + 1):
        rows = [r for r in range(1, n + 1) if flat["parent_row"][r] == p]
        nodes = [int(flat["node_id"][r]) for r in rows]
        assert nodes == sorted(nodes)  # rank order = creation order under one parent
    assert np.array_equal(flat["position"], 40 + flat["depth"])


def test_fanout_errors():
    st = oracle.tree_expand_init(1)
    ids, lps = _cands([0], 2)
    with pytest.raises(ValueError):
        oracle.static_tree_step(st, ids, lps, [3])
    with pytest.raises(ValueError):
        oracle.static_tree_step(st, ids, lps, [-1])
    with pytest.raises(ValueError):
        oracle.static_tree_step(st, ids, lps, [])
