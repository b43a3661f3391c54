"""Pins of oracle.tree_commit ([M7.5] 0x05D "Feature And KV Commit")."""
import numpy as np
import pytest

import oracle


def _logical(cache, table, b, n):
    """The committed sequence of request b, read position by position."""
    return np.stack([cache[table[b, p // 16], p % 16] for p in range(n)])


def _setup(seed, B=3, R=9, Hkv=2, D=8, maxd=4):
    rng = np.random.default_rng(seed)
    P = 40
    kc = rng.normal(size=(P, 16, Hkv, D))
    vc = rng.normal(size=(P, 16, Hkv, D))
    pages = rng.permutation(P)
    table = pages[:B * 6].reshape(B, 6)
    ctx = np.array([5, 16, 31])[:B]  # a fresh page, an exact page boundary, one slot left
    kt = rng.normal(size=(B, R, Hkv, D))
    vt = rng.normal(size=(B, R, Hkv, D))
    feat = rng.normal(size=(B * R, 5))
    path = np.full((B, maxd + 1), -1)
    acc = np.array([0, 2, 4])[:B]
    for b in range(B):
        rows = [0] + sorted(rng.choice(np.arange(1, R), size=int(acc[b]), replace=False).tolist())
        path[b, :len(rows)] = rows
    return kc, vc, table, ctx, kt, vt, feat, path, acc


def test_committed_sequence_is_prefix_then_accepted_rows():
    kc, vc, table, ctx, kt, vt, feat, path, acc = _setup(1)
    out = oracle.tree_commit(kc, vc, table, ctx, kt, vt, path, acc, features=feat)
    for b in range(3):
        n = int(acc[b]) + 1
        assert out["ctx_lens"][b] == ctx[b] + n
        old = _logical(kc, table, b, int(ctx[b]))
        new = _logical(out["k_cache"], table, b, int(out["ctx_lens"][b]))
        np.testing.assert_array_equal(new[:ctx[b]], old)                 # prefix untouched
        np.testing.assert_array_equal(new[ctx[b]:], kt[b, path[b, :n]])  # rows in path order
        newv = _logical(out["v_cache"], table, b, int(out["ctx_lens"][b]))
        np.testing.assert_array_equal(newv[ctx[b]:], vt[b, path[b, :n]])
        np.testing.assert_array_equal(out["features"][b, :n], feat[b * 9 + path[b, :n]])
        assert not out["features"][b, n:].any()


def test_nothing_else_changes():
    kc, vc, table, ctx, kt, vt, feat, path, acc = _setup(2)
    out = oracle.tree_commit(kc, vc, table, ctx, kt, vt, path, acc)
    touched = set()
    for b in range(3):
        for i in range(int(acc[b]) + 1):
            p = int(ctx[b]) + i
            touched.add((int(table[b, p // 16]), p % 16))
    for pg in range(kc.shape[0]):
        for s in range(16):
            if (pg, s) not in touched:
                assert np.array_equal(out["k_cache"][pg, s], kc[pg, s])
                assert np.array_equal(out["v_cache"][pg, s], vc[pg, s])


def test_rows_by_index_not_token():
    # two accepted rows carrying the same token id must both be committed from
    # their own rows (the commit never looks at token ids)
    kc, vc, table, ctx, kt, vt, feat, path, acc = _setup(3)
    kt[2, path[2, 1]] = 1.0
    kt[2, path[2, 2]] = 2.0
    out = oracle.tree_commit(kc, vc, table, ctx, kt, vt, path, acc)
    new = _logical(out["k_cache"], table, 2, int(out["ctx_lens"][2]))
    assert np.all(new[ctx[2] + 1] == 1.0) and np.all(new[ctx[2] + 2] == 2.0)


def test_validation():
    kc, vc, table, ctx, kt, vt, feat, path, acc = _setup(4)
    bad = path.copy()
    bad[1, 1] = 99
    with pytest.raises(ValueError):
        oracle.tree_commit(kc, vc, table, ctx, kt, vt, bad, acc)
    with pytest.raises(ValueError):
        oracle.tree_commit(kc, vc, table, np.array([5, 16, 95]), kt, vt, path, acc)
