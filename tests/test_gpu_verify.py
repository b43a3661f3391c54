"""GPU parity of eagle_tree_verify against the oracle (through the C-ABI)."""
import numpy as np
import pytest
import torch
from scipy import stats

import oracle
from eagle_speculative_decoding_gb300 import synth
from gpu_helpers import need_gpu

pytestmark = pytest.mark.gpu
MARGIN = 1e-5  # decisions closer than this to their threshold are not asserted


def _run(b, parent, tok, T, max_depth, logits=None, argmax=None, n_rows=None, seed=0, offset=0,
         override=None):
    dev = "cuda"
    B, R = parent.shape
    acc = torch.empty(B, dtype=torch.int32, device=dev)
    path = torch.empty((B, max_depth + 1), dtype=torch.int32, device=dev)
    out = torch.empty((B, max_depth + 1), dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    V = logits.shape[2] if logits is not None else 1 << 20
    b.eagle_tree_verify(
        parent.to(dev), tok.to(dev), T, max_depth, acc, path, out,
        n_rows=None if n_rows is None else n_rows.to(dev),
        target_logits=None if logits is None else logits.to(dev),
        target_argmax=None if argmax is None else argmax.to(dev),
        seed=seed, offset=offset, V=V,
        uniforms_override=None if override is None else override.to(dev), status=st)
    torch.cuda.synchronize()
    return acc.cpu().numpy(), path.cpu().numpy(), out.cpu().numpy(), int(st.item())


def _trees(B, R, max_depth, V, gen):
    parents, toks = [], []
    for _ in range(B):
        p, _ = synth.random_tree(R, max_depth, gen)
        parents.append(p)
        toks.append(synth.distinct_sibling_tokens(p, V, gen))
    return torch.stack(parents), torch.stack(toks)


@pytest.mark.parametrize("B,R,V,depth", [(1, 17, 1024, 4), (3, 61, 5000, 6), (16, 9, 128256, 4),
                                         (1, 61, 128256, 6), (4, 64, 128256, 8)])
@pytest.mark.parametrize("use_argmax", [False, True])
def test_greedy_bit_exact(B, R, V, depth, use_argmax):
    b = need_gpu()
    gen = synth.generator(B * 1000 + R)
    parent, tok = _trees(B, R, depth, V, gen)
    z = synth.target_logits((B, R, V), gen, min_top2_gap=1e-2)
    # steer argmaxes onto children so that paths are long
    rng = np.random.default_rng(R)
    zn = z.numpy()
    for bb in range(B):
        for r in range(R):
            ch = [c for c in range(1, R) if parent[bb, c] == r]
            if ch and rng.random() < 0.7:
                zn[bb, r, int(tok[bb, rng.choice(ch)])] = zn[bb, r].max() + 1.0
    am = torch.from_numpy(zn.argmax(axis=2).astype(np.int32))
    ref = oracle.tree_verify(parent.numpy(), tok.numpy(), 0.0, depth, target_logits=zn)
    acc, path, out, st = _run(b, parent, tok, 0.0, depth, logits=None if use_argmax else z,
                              argmax=am if use_argmax else None)
    assert st == 0
    assert np.array_equal(acc, ref["accept_len"])
    assert np.array_equal(path, ref["path_rows"])
    assert np.array_equal(out, ref["out_tokens"])


def _stochastic_case(B, R, V, depth, T, seed):
    gen = synth.generator(seed)
    parent, tok = _trees(B, R, depth, V, gen)
    z = synth.target_logits((B, R, V), gen, std=1.0 if V < 100 else synth.LOGIT_STD)
    # lift each drafted token near the top of its parent's target row so that
    # acceptances happen at every depth
    zn = z.numpy()
    rng = np.random.default_rng(seed)
    top = zn.max(axis=2)
    for bb in range(B):
        for c in range(1, R):
            r = int(parent[bb, c])
            zn[bb, r, int(tok[bb, c])] = top[bb, r] + rng.uniform(-1.0, 2.0) * T
    return parent, tok, torch.from_numpy(zn)


@pytest.mark.parametrize("B,R,V,depth,T", [(8, 17, 1024, 4, 1.0), (64, 9, 128256, 4, 1.0),
                                           (4, 61, 128256, 8, 0.6), (2, 61, 128256, 6, 1.0)])
def test_stochastic_matches_oracle_on_shared_philox(B, R, V, depth, T):
    b = need_gpu()
    T = float(np.float32(T))
    parent, tok, z = _stochastic_case(B, R, V, depth, T, seed=R + B)
    seed, offset = 1234567 + B, 99
    ref = oracle.tree_verify(parent.numpy(), tok.numpy(), T, depth, target_logits=z.numpy(),
                             seed=seed, offset=offset)
    acc, path, out, st = _run(b, parent, tok, T, depth, logits=z, seed=seed, offset=offset)
    assert st == 0
    close = {bb for kind, bb, m in ref["margins"] if m < MARGIN}
    checked = 0
    for bb in range(B):
        if bb in close:
            continue
        checked += 1
        assert acc[bb] == ref["accept_len"][bb], bb
        assert np.array_equal(path[bb], ref["path_rows"][bb]), bb
        assert np.array_equal(out[bb], ref["out_tokens"][bb]), bb
    print(f"B={B} R={R} V={V}: {B - checked} of {B} requests within {MARGIN} of a threshold")
    assert checked == B  # these seeds put no decision within MARGIN of its threshold
    assert ref["accept_len"].max() >= 1  # the case exercises accepted paths


def test_override_uniforms_and_n_rows():
    b = need_gpu()
    parent = torch.tensor([[-1, 0, 0, 1, 3, 0]], dtype=torch.int32)
    tok = torch.tensor([[0, 1, 2, 3, 4, 7]], dtype=torch.int32)
    z = torch.zeros((1, 6, 8))
    n_rows = torch.tensor([5], dtype=torch.int32)
    acc, path, out, st = _run(b, parent, tok, 1.0, 4, logits=z, n_rows=n_rows,
                              override=torch.zeros((1, 6)))
    assert st == 0 and path[0, :4].tolist() == [0, 1, 3, 4]
    ref = oracle.tree_verify(parent.numpy(), tok.numpy(), 1.0, 4, n_rows=[5], target_logits=z.numpy(),
                             accept_u=np.full((1, 6), 1 - 2 ** -24))
    acc, path, out, st = _run(b, parent, tok, 1.0, 4, logits=z, n_rows=n_rows,
                              override=torch.full((1, 6), 1 - 2 ** -24))
    assert acc[0] == 0 and out[0, 0] == ref["out_tokens"][0, 0]


def test_device_detects_bad_tree():
    b = need_gpu()
    parent = torch.tensor([[-1, 0, 2]], dtype=torch.int32)  # row 2 is its own parent
    tok = torch.tensor([[0, 1, 2]], dtype=torch.int32)
    acc, path, out, st = _run(b, parent, tok, 0.0, 2, argmax=torch.zeros((1, 3), dtype=torch.int32))
    assert st == 5 and acc[0] == 0 and out[0].tolist() == [-1, -1, -1]
    # path deeper than max_depth
    parent = torch.tensor([[-1, 0, 1]], dtype=torch.int32)
    tok = torch.tensor([[0, 0, 0]], dtype=torch.int32)
    acc, path, out, st = _run(b, parent, tok, 0.0, 1, argmax=torch.zeros((1, 3), dtype=torch.int32))
    assert st == 5


def test_host_rejects_invalid_arguments():
    b = need_gpu()
    d = "cuda"
    parent = torch.zeros((1, 4), dtype=torch.int32, device=d)
    acc = torch.empty(1, dtype=torch.int32, device=d)
    path = torch.empty((1, 3), dtype=torch.int32, device=d)
    with pytest.raises(b.EagleError) as e:
        b.eagle_tree_verify(parent, parent, 1.0, 2, acc, path, path, V=8)  # T>0 without logits
    assert e.value.code == 1
    with pytest.raises(b.EagleError) as e:  # sampled proposals need the draft logits
        b.eagle_tree_verify(parent, parent, 1.0, 2, acc, path, path,
                            target_logits=torch.zeros((1, 4, 8), device=d), proposal_mode=1)
    assert e.value.code == 1


def test_chi_square_one_million_gpu_draws():
    """The GPU verifier's first two emitted tokens follow the target
    distribution (vocab-8 toy tree, 2^20 seeded requests)."""
    b = need_gpu()
    rng = np.random.default_rng(5)
    parent = np.array([-1, 0, 0, 0, 1, 1, 2, 2, 3, 3])
    R, V, T = len(parent), 8, 1.0
    z = rng.normal(0, 1.5, (R, V)).astype(np.float32)
    zd = (z + rng.normal(0, 0.5, (R, V))).astype(np.float32)
    tok = np.zeros(R, np.int32)
    for r in range(R):
        ch = [c for c in range(1, R) if parent[c] == r]
        order = np.argsort(-zd[r], kind="stable")
        for i, c in enumerate(ch):
            tok[c] = order[i]
    N = 1 << 20
    P = torch.from_numpy(np.ascontiguousarray(np.broadcast_to(parent.astype(np.int32), (N, R))))
    Tk = torch.from_numpy(np.ascontiguousarray(np.broadcast_to(tok, (N, R))))
    Z = torch.from_numpy(np.ascontiguousarray(np.broadcast_to(z, (N, R, V))))
    acc, path, out, st = _run(b, P, Tk, T, 2, logits=Z, seed=2024, offset=7)
    assert st == 0

    def sm(x):
        w = np.exp(x - x.max())
        return w / w.sum()
    p0 = sm(z[0].astype(np.float64))
    child_of = {int(tok[c]): c for c in (1, 2, 3)}
    probs = {}
    for y in range(V):
        if y in child_of:
            pc = sm(z[child_of[y]].astype(np.float64))
            for y2 in range(V):
                probs[(y, y2)] = p0[y] * pc[y2]
        else:
            probs[(y,)] = p0[y]
    keys = sorted(probs)
    idx = {k: i for i, k in enumerate(keys)}
    first, second = out[:, 0], out[:, 1]
    counts = np.zeros(len(keys))
    is_child = np.isin(first, list(child_of))
    for y in range(V):
        if y in child_of:
            sel = second[first == y]
            counts[[idx[(y, y2)] for y2 in range(V)]] += np.bincount(sel, minlength=V)
        else:
            counts[idx[(y,)]] = np.sum(first == y)
    assert counts.sum() == N
    f_exp = np.array([probs[k] for k in keys]) * N
    assert stats.chisquare(counts, f_exp).pvalue > 1e-3
    assert is_child.mean() > 0.3


def _sampled_case(B, R, V, depth, T, seed):
    """Trees whose siblings are i.i.d. draws from q = softmax(draft / T) of
    their parent row (repeats allowed), draft logits near the target's."""
    gen = synth.generator(seed)
    rng = np.random.default_rng(seed)
    z = synth.target_logits((B, R, V), gen, std=1.5).numpy()
    zd = (z + rng.normal(0, 0.5, z.shape)).astype(np.float32)
    parent = np.zeros((B, R), np.int32)
    tok = np.zeros((B, R), np.int32)
    for b in range(B):
        parent[b] = synth.random_tree(R, depth, gen)[0].numpy()
        for c in range(1, R):
            r = parent[b, c]
            q = np.exp((zd[b, r] - zd[b, r].max()) / T)
            tok[b, c] = rng.choice(V, p=q / q.sum())
    return torch.from_numpy(parent), torch.from_numpy(tok), torch.from_numpy(z), torch.from_numpy(zd)


# The kernel runs a cluster of 1, 2, 4 or 8 CTAs per request (fewer when B is
# large or V small): (16, 64) and (8, 500) take one CTA, (64, 4096) two,
# (20, 8192) four, and (4, 32000), (3, 20001) (V not a multiple of 4) and the
# 8B-shaped (1, 128256) eight, on a 152-SM GPU.
@pytest.mark.parametrize("B,R,V,depth,T", [(16, 13, 64, 4, 1.0), (8, 21, 500, 5, 0.7),
                                           (4, 9, 32000, 3, 1.0), (64, 9, 4096, 4, 1.0),
                                           (20, 13, 8192, 4, 0.8), (3, 9, 20001, 3, 1.0),
                                           (1, 61, 128256, 6, 1.0)])
def test_sampled_proposals_match_oracle(B, R, V, depth, T):
    b = need_gpu()
    T = float(np.float32(T))
    parent, tok, z, zd = _sampled_case(B, R, V, depth, T, seed=B + V)
    seed, offset = 99 + R, 5
    ref = oracle.tree_verify(parent.numpy(), tok.numpy(), T, depth, target_logits=z.numpy(),
                             draft_logits=zd.numpy(), mode="sampled", seed=seed, offset=offset)
    dev = "cuda"
    acc = torch.empty(B, dtype=torch.int32, device=dev)
    path = torch.empty((B, depth + 1), dtype=torch.int32, device=dev)
    out = torch.empty((B, depth + 1), dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    b.eagle_tree_verify(parent.to(dev), tok.to(dev), T, depth, acc, path, out,
                        target_logits=z.to(dev), draft_logits=zd.to(dev), proposal_mode=1,
                        seed=seed, offset=offset, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    close = {bb for kind, bb, m in ref["margins"] if m < 1e-4}
    checked = 0
    for bb in range(B):
        if bb in close:
            continue
        checked += 1
        assert acc[bb].item() == ref["accept_len"][bb], bb
        assert path[bb].tolist() == ref["path_rows"][bb].tolist(), bb
        assert out[bb].tolist() == ref["out_tokens"][bb].tolist(), bb
    print(f"sampled B={B} R={R} V={V}: {B - checked} of {B} requests within 1e-4 of a threshold")
    assert checked == B  # these seeds put no decision within 1e-4 of its threshold


def test_sampled_proposals_chi_square():
    """Algorithm 1 is lossless: with three siblings drawn i.i.d. from q for
    every request, the first emitted token follows p (2^16 requests)."""
    b = need_gpu()
    rng = np.random.default_rng(11)
    V, N, T = 8, 1 << 16, 1.0
    z = rng.normal(0, 1.5, V).astype(np.float32)
    zd = (z + rng.normal(0, 1.0, V)).astype(np.float32)
    q = np.exp(zd - zd.max())
    q /= q.sum()
    parent = np.tile(np.array([-1, 0, 0, 0], np.int32), (N, 1))
    tok = np.zeros((N, 4), np.int32)
    tok[:, 1:] = rng.choice(V, size=(N, 3), p=q)
    Z = np.broadcast_to(z, (N, 4, V)).copy()
    ZD = np.broadcast_to(zd, (N, 4, V)).copy()
    dev = "cuda"
    acc = torch.empty(N, dtype=torch.int32, device=dev)
    path = torch.empty((N, 2), dtype=torch.int32, device=dev)
    out = torch.empty((N, 2), dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    b.eagle_tree_verify(torch.from_numpy(parent).to(dev), torch.from_numpy(tok).to(dev), T, 1, acc,
                        path, out, target_logits=torch.from_numpy(Z).to(dev),
                        draft_logits=torch.from_numpy(ZD).to(dev), proposal_mode=1, seed=2025,
                        status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    first = out[:, 0].cpu().numpy()
    p = np.exp(z.astype(np.float64) - z.max())
    p /= p.sum()
    counts = np.bincount(first, minlength=V)
    assert counts.sum() == N
    assert stats.chisquare(counts, p * N).pvalue > 1e-3
    assert (acc.cpu().numpy() >= 1).mean() > 0.3  # acceptances carry much of the mass
