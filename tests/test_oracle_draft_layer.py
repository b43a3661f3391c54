"""Pins of the oracle's drafter decoder layer and its parts (RMSNorm,
rotate-half RoPE, SiLU).  Each pin checks a property the definitions fix
rather than retyping them: scale invariance, rotation identities, a library
sigmoid, shift invariance of attention under a common position offset, the
closed form when a node sees only itself, GQA = MHA with replicated kv heads,
permutation invariance over the new nodes, and zero-weight residual paths."""
import math

import numpy as np
import pytest
import scipy.special

import oracle


def _rng(seed):
    return np.random.default_rng(seed)


def test_rms_norm_unit_rms_scale_invariance_constant_row():
    x = _rng(1).normal(size=(4, 16))
    y = oracle.rms_norm(x, np.ones(16), 0.0)
    assert np.allclose(np.mean(y * y, axis=1), 1.0, atol=1e-12)
    assert np.allclose(oracle.rms_norm(3.7 * x, np.ones(16), 0.0), y, atol=1e-12)
    w = _rng(2).normal(size=16)
    c = np.full((1, 16), -2.5)
    assert np.allclose(oracle.rms_norm(c, w, 0.25), -2.5 / math.sqrt(6.25 + 0.25) * w, atol=1e-12)


def test_rope_identity_at_zero_and_norm_preserved():
    x = _rng(3).normal(size=(5, 3, 8))
    assert np.allclose(oracle.rope(x, np.zeros((5, 1)), 10000.0), x, atol=0)
    y = oracle.rope(x, np.arange(5)[:, None] * 37, 10000.0)
    pair = lambda a: a[..., :4] ** 2 + a[..., 4:] ** 2
    assert np.allclose(pair(y), pair(x), atol=1e-12)


def test_rope_two_dims_is_complex_rotation():
    # D = 2: one pair with frequency theta^0 = 1, i.e. multiplication by e^{i pos}
    x = np.array([[0.3, -1.2]])
    for pos in (0, 1, 5, 1000):
        z = complex(0.3, -1.2) * complex(math.cos(pos), math.sin(pos))
        assert np.allclose(oracle.rope(x, np.array([pos]), 123.0)[0], [z.real, z.imag], atol=1e-12)


def test_rope_scores_depend_on_relative_position_only():
    r = _rng(4)
    q, k = r.normal(size=64), r.normal(size=64)
    for m, n in ((10, 3), (1000, 993), (7, 7), (50000, 0)):
        lhs = oracle.rope(q, np.array(m), 500000.0) @ oracle.rope(k, np.array(n), 500000.0)
        rhs = oracle.rope(q, np.array(m - n), 500000.0) @ k
        assert abs(lhs - rhs) < 1e-9 * (1 + abs(rhs))


def test_silu_matches_library_sigmoid():
    x = np.linspace(-30, 30, 121)
    assert np.allclose(oracle.silu(x), x * scipy.special.expit(x), rtol=1e-13, atol=1e-300)
    assert oracle.silu(np.array([0.0]))[0] == 0.0


def _layer_case(seed, B=1, W=3, d=16, Hq=4, Hkv=2, D=8, I=24, ctx=5, Rmax=6, r0=1):
    r = _rng(seed)
    wts = dict(norm1=1 + 0.1 * r.normal(size=d), qkv=0.3 * r.normal(size=((Hq + 2 * Hkv) * D, d)),
               o=0.3 * r.normal(size=(d, Hq * D)), norm2=1 + 0.1 * r.normal(size=d),
               gu=0.3 * r.normal(size=(2 * I, d)), down=0.3 * r.normal(size=(d, I)))
    x = r.normal(size=(B * W, d))
    P = B * 2
    kc, vc = r.normal(size=(P, 16, Hkv, D)), r.normal(size=(P, 16, Hkv, D))
    table = np.arange(P).reshape(B, 2)
    ctx_lens = np.full(B, ctx)
    kt, vt = r.normal(size=(B, Rmax, Hkv, D)), r.normal(size=(B, Rmax, Hkv, D))
    return wts, x, kc, vc, table, ctx_lens, kt, vt


def test_layer_single_visible_key_closed_form():
    # ctx 0 and a mask holding only the row itself: the softmax has one key, so
    # the attention output is that row's own v and q / k / RoPE drop out
    d, Hq, Hkv, D, I, W = 16, 4, 2, 8, 24, 3
    wts, x, kc, vc, table, _, kt, vt = _layer_case(5)
    mask = np.array([[1 << i for i in range(6)]], dtype=np.uint64)
    pos = np.array([[4, 9, 2]])
    out, _, vnew = oracle.draft_layer(x, wts, pos, kc, vc, table, np.zeros(1, int), kt, vt, mask, 1, Hq, Hkv)
    h = x / np.sqrt(np.mean(x * x, axis=1, keepdims=True) + 1e-5) * wts["norm1"]
    v = (h @ wts["qkv"][(Hq + Hkv) * D:].T).reshape(W, Hkv, D)
    a = np.repeat(v, Hq // Hkv, axis=1).reshape(W, Hq * D)  # query head h reads kv head h // G
    x1 = x + a @ wts["o"].T
    h2 = x1 / np.sqrt(np.mean(x1 * x1, axis=1, keepdims=True) + 1e-5) * wts["norm2"]
    g, u = h2 @ wts["gu"][:I].T, h2 @ wts["gu"][I:].T
    expect = x1 + (g * scipy.special.expit(g) * u) @ wts["down"].T
    assert np.abs(out - expect).max() < 1e-10
    assert np.allclose(vnew[0], v, atol=1e-12)


def test_layer_shift_invariance_of_positions():
    # all keys come from the layer itself (ctx 0, chain over the new rows):
    # moving every position by the same offset changes no score
    Hq, Hkv = 4, 2
    wts, x, kc, vc, table, _, kt, vt = _layer_case(6)
    # rows 1..3 are the new nodes; row 0 (an earlier node) is hidden from them
    mask = np.array([[1, 0b10, 0b110, 0b1110, 1 << 4, 1 << 5]], dtype=np.uint64)
    base = np.array([[3, 4, 5]])
    o1, _, _ = oracle.draft_layer(x, wts, base, kc, vc, table, np.zeros(1, int), kt, vt, mask, 1, Hq, Hkv)
    o2, k2, _ = oracle.draft_layer(x, wts, base + 777, kc, vc, table, np.zeros(1, int), kt, vt, mask, 1, Hq, Hkv)
    assert np.abs(o1 - o2).max() < 1e-9
    o3, k3, _ = oracle.draft_layer(x, wts, base + 777, kc, vc, table, np.zeros(1, int), kt, vt, mask, 1, Hq, Hkv,
                                   theta=10000.0)
    assert np.abs(k3 - k2).max() > 1e-3  # the keys themselves do move with theta / position


def test_layer_gqa_equals_replicated_mha():
    d, Hq, Hkv, D, I = 16, 4, 2, 8, 24
    wts, x, kc, vc, table, ctx, kt, vt = _layer_case(7)
    mask = np.array([[1, 0b11, 0b101, 0b1001, 1 << 4, 1 << 5]], dtype=np.uint64)
    pos = np.array([[5, 6, 6]])
    out, _, _ = oracle.draft_layer(x, wts, pos, kc, vc, table, ctx, kt, vt, mask, 1, Hq, Hkv)
    # MHA: kv head of query head h is h // 2, so duplicate each kv head's rows
    qw, kw, vw = wts["qkv"][:Hq * D], wts["qkv"][Hq * D:(Hq + Hkv) * D], wts["qkv"][(Hq + Hkv) * D:]
    dup = lambda w: np.repeat(w.reshape(Hkv, D, d), 2, axis=0).reshape(Hq * D, d)
    w2 = dict(wts, qkv=np.vstack([qw, dup(kw), dup(vw)]))
    dupc = lambda c: np.repeat(c, 2, axis=-2)
    out2, _, _ = oracle.draft_layer(x, w2, pos, dupc(kc), dupc(vc), table, ctx, dupc(kt), dupc(vt), mask, 1,
                                    Hq, Hq)
    assert np.abs(out - out2).max() < 1e-10


def test_layer_permutation_of_new_nodes():
    Hq, Hkv = 4, 2
    wts, x, kc, vc, table, ctx, kt, vt = _layer_case(8)
    # new rows 1..3 each see row 0 and themselves
    mask = np.array([[1, 0b11, 0b101, 0b1001, 1 << 4, 1 << 5]], dtype=np.uint64)
    pos = np.array([[6, 7, 8]])
    out, knew, _ = oracle.draft_layer(x, wts, pos, kc, vc, table, ctx, kt, vt, mask, 1, Hq, Hkv)
    perm = [2, 0, 1]
    outp, knewp, _ = oracle.draft_layer(x[perm], wts, pos[:, perm], kc, vc, table, ctx, kt, vt, mask, 1, Hq, Hkv)
    assert np.abs(outp - out[perm]).max() < 1e-12
    assert np.abs(knewp[0] - knew[0][perm]).max() < 1e-12


def test_layer_zero_weight_residual_paths():
    Hq, Hkv, I = 4, 2, 24
    wts, x, kc, vc, table, ctx, kt, vt = _layer_case(9)
    mask = np.array([[1, 0b11, 0b101, 0b1001, 1 << 4, 1 << 5]], dtype=np.uint64)
    pos = np.array([[6, 7, 8]])
    z = dict(wts, o=np.zeros_like(wts["o"]), down=np.zeros_like(wts["down"]))
    out, _, _ = oracle.draft_layer(x, z, pos, kc, vc, table, ctx, kt, vt, mask, 1, Hq, Hkv)
    assert np.array_equal(out, x)
    z2 = dict(wts, o=np.zeros_like(wts["o"]))
    out2, _, _ = oracle.draft_layer(x, z2, pos, kc, vc, table, ctx, kt, vt, mask, 1, Hq, Hkv)
    h2 = oracle.rms_norm(x, wts["norm2"], 1e-5)
    gu = h2 @ wts["gu"].T
    assert np.abs(out2 - (x + (oracle.silu(gu[:, :I]) * gu[:, I:]) @ wts["down"].T)).max() < 1e-12
    with pytest.raises(ValueError):
        oracle.draft_layer(x, wts, pos, kc, vc, table, ctx, kt, vt, mask, 4, Hq, Hkv)


def test_linear_bruteforce_bias_residual():
    r = _rng(10)
    x, w, b, res = r.normal(size=(3, 5)), r.normal(size=(4, 5)), r.normal(size=4), r.normal(size=(3, 4))
    y = oracle.linear(x, w, b, res)
    for i in range(3):
        for o in range(4):
            acc = b[o] + res[i, o]
            for c in range(5):
                acc += w[o, c] * x[i, c]
            assert abs(y[i, o] - acc) < 1e-12
