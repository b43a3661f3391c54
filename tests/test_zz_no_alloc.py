"""eagle_tree_verify_noalloc: verification for callers that cannot allocate.

Some callers hold no device allocator of their own (a plugin whose host
framework owns all device memory and passes only its tensors; a loop that may
not call cudaMalloc because it can synchronise the device).  This entry point
keeps its row statistics in a fixed buffer inside the library.  Its outputs
must equal those of eagle_tree_verify (integer outputs: bit-exact) on two
calls in a row, the second on different inputs, so stale buffer contents
from the first call would show; each call is also checked against the CPU
oracle on every request whose decisions are not within rounding of a
threshold.  Both proposal modes go through the fixed buffer, and calls beyond
its capacity are refused before anything launches.  This file runs last in
the suite.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from eagle_speculative_decoding_gb300 import synth
from gpu_helpers import need_gpu

pytestmark = pytest.mark.gpu


def _case(seed, B, R, V, depth, T):
    gen = synth.generator(seed)
    parents, toks = [], []
    for _ in range(B):
        p, _ = synth.random_tree(R, depth, gen)
        parents.append(p)
        toks.append(synth.distinct_sibling_tokens(p, V, gen))
    parent, tok = torch.stack(parents), torch.stack(toks)
    z = synth.target_logits((B, R, V), gen)
    zn = z.numpy()
    top = zn.max(axis=2)
    rng = np.random.default_rng(seed)
    for b in range(B):
        for c in range(1, R):
            r = int(parent[b, c])
            zn[b, r, int(tok[b, c])] = top[b, r] + rng.uniform(-1.0, 2.0) * max(T, 0.5)
    return parent, tok, torch.from_numpy(zn)


def _sampled_case(seed, B, R, V, depth, T):
    """Siblings drawn i.i.d. from q = softmax(draft / T) of their parent row
    (repeats allowed), draft logits near the target's."""
    gen = synth.generator(seed)
    rng = np.random.default_rng(seed)
    z = synth.target_logits((B, R, V), gen, std=1.5).numpy()
    zd = (z + rng.normal(0, 0.5, z.shape)).astype(np.float32)
    parent = np.zeros((B, R), np.int32)
    tok = np.zeros((B, R), np.int32)
    for b in range(B):
        parent[b] = synth.random_tree(R, depth, gen)[0].numpy()
        for c in range(1, R):
            q = np.exp((zd[b, parent[b, c]] - zd[b, parent[b, c]].max()) / T)
            tok[b, c] = rng.choice(V, p=q / q.sum())
    return (torch.from_numpy(parent), torch.from_numpy(tok), torch.from_numpy(z),
            torch.from_numpy(zd))


def _outputs(B, depth):
    z = lambda *s: torch.full(s, -7, dtype=torch.int32, device="cuda")
    return z(B), z(B, depth + 1), z(B, depth + 1), torch.zeros(1, dtype=torch.int32, device="cuda")


def _call_noalloc(L, parent, tok, z, T, depth, outs, seed, zd=None, mode=0):
    B, R = parent.shape
    acc, path, out, st = outs
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    return L.eagle_tree_verify_noalloc(
        B, R, z.shape[2], p(parent), p(tok), None, p(z), None, None if zd is None else p(zd),
        float(T), mode, seed, 3, None, depth, p(acc), p(path), p(out), p(st),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _check_oracle(ref, got, B):
    """Integer outputs equal the oracle's on every request whose decisions
    all clear their thresholds by more than float rounding; returns how many
    requests were exempt."""
    close = {bb for _, bb, m in ref["margins"] if m < 1e-4}
    acc, path, out = (t.cpu() for t in got[:3])
    for bb in range(B):
        if bb in close:
            continue
        assert int(acc[bb]) == ref["accept_len"][bb], bb
        assert path[bb].tolist() == ref["path_rows"][bb].tolist(), bb
        assert out[bb].tolist() == ref["out_tokens"][bb].tolist(), bb
    return len(close)


@pytest.mark.parametrize("T", [1.0, 0.0])
def test_noalloc_matches_workspace_entry_point_twice(T):
    b = need_gpu()
    L = b.lib()
    cases = [(_case(11, 8, 61, 128256, 6, T), 6, 101), (_case(12, 64, 9, 32000, 4, T), 4, 202)]
    for (parent_h, tok_h, z_h), depth, seed in cases:  # two calls in a row, different inputs
        parent, tok, z = parent_h.cuda(), tok_h.cuda(), z_h.cuda()
        B = parent.shape[0]
        ref = _outputs(B, depth)
        b.eagle_tree_verify(parent, tok, T, depth, ref[0], ref[1], ref[2], target_logits=z,
                            seed=seed, offset=3, status=ref[3])
        got = _outputs(B, depth)
        assert _call_noalloc(L, parent, tok, z, T, depth, got, seed) == 0
        torch.cuda.synchronize()
        assert int(ref[3].item()) == 0 and int(got[3].item()) == 0
        for r, g in zip(ref[:3], got[:3]):
            assert torch.equal(r, g)
        assert int(ref[0].max()) >= 1  # the case accepts drafted nodes
        want = oracle.tree_verify(parent_h.numpy(), tok_h.numpy(), T, depth,
                                  target_logits=z_h.numpy(), seed=seed, offset=3)
        exempt = _check_oracle(want, got, B)
        print(f"T={T} B={B}: {exempt} of {B} requests within 1e-4 of a threshold")
        assert exempt <= max(1, B // 8)


def test_noalloc_sampled_proposals_twice():
    """Sampled proposals (Algorithm 1 with the draft distribution) through
    the fixed buffer: equal to eagle_tree_verify and to the oracle."""
    b = need_gpu()
    for (B, R, V, depth, T, seed) in [(16, 13, 500, 4, 1.0, 31), (4, 9, 32000, 3, 0.7, 32)]:
        T = float(np.float32(T))
        parent_h, tok_h, z_h, zd_h = _sampled_case(seed, B, R, V, depth, T)
        parent, tok, z, zd = parent_h.cuda(), tok_h.cuda(), z_h.cuda(), zd_h.cuda()
        ref = _outputs(B, depth)
        b.eagle_tree_verify(parent, tok, T, depth, ref[0], ref[1], ref[2], target_logits=z,
                            draft_logits=zd, proposal_mode=b.EAGLE_PROPOSAL_SAMPLED, seed=seed,
                            offset=3, status=ref[3])
        got = _outputs(B, depth)
        b.eagle_tree_verify_noalloc(parent, tok, T, depth, got[0], got[1], got[2], target_logits=z,
                                    draft_logits=zd, proposal_mode=b.EAGLE_PROPOSAL_SAMPLED,
                                    seed=seed, offset=3, status=got[3])
        torch.cuda.synchronize()
        assert int(ref[3].item()) == 0 and int(got[3].item()) == 0
        for r, g in zip(ref[:3], got[:3]):
            assert torch.equal(r, g)
        want = oracle.tree_verify(parent_h.numpy(), tok_h.numpy(), T, depth,
                                  target_logits=z_h.numpy(), draft_logits=zd_h.numpy(),
                                  mode="sampled", seed=seed, offset=3)
        exempt = _check_oracle(want, got, B)
        print(f"sampled B={B} V={V}: {exempt} of {B} requests within 1e-4 of a threshold")
        assert exempt <= max(1, B // 4)


def test_noalloc_rejects_rows_beyond_capacity():
    b = need_gpu()
    L = b.lib()
    B, R = 2048, 33  # 67584 rows > 65536
    parent = torch.zeros((B, R), dtype=torch.int32, device="cuda")
    z = torch.zeros((B, R, 8), device="cuda")
    outs = _outputs(B, 2)
    assert _call_noalloc(L, parent, parent, z, 1.0, 2, outs, 0) == 3  # EAGLE_ERR_WORKSPACE


def test_noalloc_rejects_race_chunks_beyond_capacity():
    """At T > 0 the bonus-token race keeps one partial per 4096 vocabulary
    ids per request: 2000 requests x 33 chunks = 66000 > 65536."""
    b = need_gpu()
    L = b.lib()
    B, R, V = 2000, 1, 33 * 4096
    parent = torch.full((B, R), -1, dtype=torch.int32, device="cuda")
    tok = torch.zeros((B, R), dtype=torch.int32, device="cuda")
    z = torch.zeros((B, R, V), device="cuda")
    outs = _outputs(B, 1)
    assert _call_noalloc(L, parent, tok, z, 1.0, 1, outs, 0) == 3  # EAGLE_ERR_WORKSPACE
    assert _call_noalloc(L, parent, tok, z, 0.0, 1, outs, 0) == 0  # greedy: no race partials
    torch.cuda.synchronize()
    assert int(outs[3].item()) == 0
    del z
