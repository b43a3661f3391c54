"""Pins of the oracle's tree attention."""
import math

import numpy as np
import pytest
import torch
from scipy.special import softmax

import oracle
from eagle_speculative_decoding_gb300 import synth


def causal_attention(q, k, v, scale):
    """Independent dense causal attention: q,k,v [S, H, D] (k,v may have
    fewer heads; head h uses kv head h // G).  Returns [S, H, D]."""
    S, H, D = q.shape
    G = H // k.shape[1]
    out = np.zeros_like(q)
    mask = np.triu(np.full((S, S), -np.inf), 1)
    for h in range(H):
        s = scale * np.einsum("id,jd->ij", q[:, h], k[:, h // G]) + mask
        out[:, h] = softmax(s, axis=1) @ v[:, h // G]
    return out


def _case(seed, R, ctx, Hq=4, Hkv=2, D=16, page=4, parent=None):
    gen = synth.generator(seed)
    B = 1
    q = synth.normal((B, R, Hq, D), 1.0, torch.float32, gen).double().numpy()
    kt = synth.normal((B, R, Hkv, D), 1.0, torch.float32, gen).double().numpy()
    vt = synth.normal((B, R, Hkv, D), 1.0, torch.float32, gen).double().numpy()
    kc, vc, table = synth.paged_kv([ctx], Hkv, D, page, torch.float32, gen)
    if parent is None:
        parent, _ = synth.random_tree(R, 4, gen)
    mask = oracle.ancestor_mask(np.asarray(parent))[None]
    return q, kt, vt, kc.double().numpy(), vc.double().numpy(), table.numpy(), np.array([ctx]), mask, np.asarray(parent)


def _prefix(kc, table, ctx, page):
    npg = (ctx + page - 1) // page
    return kc[table[0, :npg]].reshape(npg * page, *kc.shape[2:])[:ctx]


def test_chain_tree_equals_causal_attention():
    R, ctx, page = 7, 21, 4
    q, kt, vt, kc, vc, table, cl, mask, parent = _case(0, R, ctx, page=page, parent=synth.chain_tree(R).numpy())
    out, lse = oracle.tree_attn(q, kt, vt, kc, vc, table, cl, mask, page_size=page)
    D = q.shape[3]
    kp, vp = _prefix(kc, table, ctx, page), _prefix(vc, table, ctx, page)
    # sequence = prefix then chain; queries for the prefix positions are unused
    Hq = q.shape[2]
    qs = np.concatenate([np.zeros((ctx, Hq, D)), q[0]], axis=0)
    ks = np.concatenate([kp, kt[0]], axis=0)
    vs = np.concatenate([vp, vt[0]], axis=0)
    ref = causal_attention(qs, ks, vs, 1 / math.sqrt(D))[ctx:]
    assert np.abs(out[0] - ref).max() < 1e-12


@pytest.mark.parametrize("seed", range(4))
def test_any_tree_row_equals_causal_attention_over_its_path(seed):
    R, ctx, page = 12, 9, 4
    q, kt, vt, kc, vc, table, cl, mask, parent = _case(seed, R, ctx, page=page)
    out, _ = oracle.tree_attn(q, kt, vt, kc, vc, table, cl, mask, page_size=page)
    D = q.shape[3]
    kp, vp = _prefix(kc, table, ctx, page), _prefix(vc, table, ctx, page)
    for r in range(R):
        path = [r]
        while path[-1] != 0:
            path.append(int(parent[path[-1]]))
        path = path[::-1]
        ks = np.concatenate([kp, kt[0, path]], axis=0)
        vs = np.concatenate([vp, vt[0, path]], axis=0)
        qs = np.concatenate([np.zeros((len(ks) - 1, q.shape[2], D)), q[0, [r]]], axis=0)
        ref = causal_attention(qs, ks, vs, 1 / math.sqrt(D))[-1]
        assert np.abs(out[0, r] - ref).max() < 1e-12


def test_single_row_is_decode_attention_and_lse():
    q, kt, vt, kc, vc, table, cl, mask, parent = _case(5, 1, 13, page=4, parent=np.array([-1]))
    out, lse = oracle.tree_attn(q, kt, vt, kc, vc, table, cl, mask, page_size=4)
    kp, vp = _prefix(kc, table, 13, 4), _prefix(vc, table, 13, 4)
    ks = np.concatenate([kp, kt[0]], 0)
    vs = np.concatenate([vp, vt[0]], 0)
    D = q.shape[3]
    for h in range(q.shape[2]):
        s = (ks[:, h // 2] @ q[0, 0, h]) / math.sqrt(D)
        w = np.exp(s - s.max())
        assert np.abs(out[0, 0, h] - (w / w.sum()) @ vs[:, h // 2]).max() < 1e-12
        assert abs(lse[0, 0, h] - math.log(np.exp(s).sum())) < 1e-12


def test_unrelated_branch_permutation_invariance():
    # root with two branches: rows 1,2 (chain) and row 3; swapping the order of
    # the branches in the flattening permutes outputs and nothing else
    R = 4
    q, kt, vt, kc, vc, table, cl, mask, _ = _case(6, R, 10, page=4, parent=np.array([-1, 0, 1, 0]))
    out, _ = oracle.tree_attn(q, kt, vt, kc, vc, table, cl, mask, page_size=4)
    perm = [0, 3, 1, 2]  # new row i holds old row perm[i]
    parent2 = np.array([-1, 0, 0, 2])
    mask2 = oracle.ancestor_mask(parent2)[None]
    out2, _ = oracle.tree_attn(q[:, perm], kt[:, perm], vt[:, perm], kc, vc, table, cl, mask2, page_size=4)
    assert np.abs(out2[0] - out[0, perm]).max() < 1e-12


def test_gqa_maps_head_to_kv_head_h_div_G():
    # replicating kv heads to MHA must give the same outputs (pins h // G)
    q, kt, vt, kc, vc, table, cl, mask, _ = _case(7, 5, 11, Hq=6, Hkv=2, page=4)
    out, _ = oracle.tree_attn(q, kt, vt, kc, vc, table, cl, mask, page_size=4)
    rep = lambda a: np.repeat(a, 3, axis=2)
    out2, _ = oracle.tree_attn(q, rep(kt), rep(vt), rep(kc), rep(vc), table, cl, mask, page_size=4)
    assert np.abs(out - out2).max() < 1e-12


def test_page_table_layout_invariance_and_sampling():
    q, kt, vt, kc, vc, table, cl, mask, _ = _case(8, 6, 18, page=4)
    out, lse = oracle.tree_attn(q, kt, vt, kc, vc, table, cl, mask, page_size=4)
    # contiguous re-layout of the same prefix
    kp, vp = _prefix(kc, table, 18, 4), _prefix(vc, table, 18, 4)
    pad = lambda a: np.concatenate([a, np.zeros((2,) + a.shape[1:])], 0).reshape(5, 4, *a.shape[1:])
    out2, lse2 = oracle.tree_attn(q, kt, vt, pad(kp), pad(vp), np.arange(5)[None], cl, mask, page_size=4)
    assert np.abs(out - out2).max() < 1e-12
    smp = oracle.tree_attn(q, kt, vt, kc, vc, table, cl, mask, page_size=4, sample=[(0, 3, 1), (0, 5, 2)])
    assert np.abs(smp[(0, 3, 1)][0] - out[0, 3, 1]).max() == 0
    assert smp[(0, 5, 2)][1] == lse[0, 5, 2]


def test_empty_prefix_sees_only_tree():
    q, kt, vt, kc, vc, table, cl, mask, parent = _case(9, 3, 0, page=4, parent=np.array([-1, 0, 0]))
    out, _ = oracle.tree_attn(q, kt, vt, kc, vc, np.zeros((1, 1), np.int64), np.array([0]), mask, page_size=4)
    # root row sees only itself: output is its own value row
    assert np.abs(out[0, 0, 0] - vt[0, 0, 0]).max() < 1e-12
