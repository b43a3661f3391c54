"""Seeded synthetic inputs shaped like the EAGLE pages' workloads.

This module only draws random numbers and lays them out; it contains none of
the method's arithmetic (no attention, no softmax, no tree ranking), so both
the CUDA path and the CPU oracle can consume its outputs.  Everything is
generated on the CPU with a seeded ``torch.Generator`` unless a ``device`` is
given (the benchmark draws its large weights on the device for speed; parity
tests always draw on the CPU).

Workloads (the pages' target models are LLaMA-3.1-8B / LLaMA-3.3-70B shaped;
their datasets and trained weights are not used, only the shapes):
  toy      batch 1, d 256, 4/2 heads x 64, V 1024, ctx 128, 16-node trees
           (depth 4, top-k 4), fp32
  llama8b  batch 1, d 4096, 32/8 heads x 128, V 128256, ctx 2048, EAGLE-2
           tree depth 6, top-k 10, expansion width 10, budget 60, bf16
  llama70b batch 1, d 8192, 64/8 heads x 128, V 128256, ctx 4096, budget 60,
           depth 6, top-k 10, width 10, bf16
  serve64  batch 64, 8B shape, per-request ctx uniform in [1024, 4096],
           8-node trees depth 4 top-k 2 width 2, T = 1.0, bf16
  long4    batch 4, 8B shape, ctx 32768, 60-node trees depth 8 top-k 8
           width 8, T = 0.6, bf16
"""

import math

import torch

CONFIGS = {
    "toy": dict(B=1, d=256, Hq=4, Hkv=2, D=64, V=1024, ctx=(128, 128), page=16,
                N=16, depth=4, topk=4, width=4, temps=(0.0, 1.0), dtype="fp32"),
    "llama8b": dict(B=1, d=4096, Hq=32, Hkv=8, D=128, V=128256, ctx=(2048, 2048), page=16,
                    N=60, depth=6, topk=10, width=10, temps=(0.0, 1.0), dtype="bf16"),
    "llama70b": dict(B=1, d=8192, Hq=64, Hkv=8, D=128, V=128256, ctx=(4096, 4096), page=16,
                     N=60, depth=6, topk=10, width=10, temps=(0.0, 1.0), dtype="bf16"),
    "serve64": dict(B=64, d=4096, Hq=32, Hkv=8, D=128, V=128256, ctx=(1024, 4096), page=16,
                    N=8, depth=4, topk=2, width=2, temps=(1.0,), dtype="bf16"),
    "long4": dict(B=4, d=4096, Hq=32, Hkv=8, D=128, V=128256, ctx=(32768, 32768), page=16,
                  N=60, depth=8, topk=8, width=8, temps=(0.6,), dtype="bf16"),
    # chain drafts of length 3 (top-1 at each depth: a degenerate tree), as in
    # the serving-engine comparisons, at batch 64
    "chain3": dict(B=64, d=4096, Hq=32, Hkv=8, D=128, V=128256, ctx=(1024, 4096), page=16,
                   N=3, depth=3, topk=1, width=1, temps=(0.0,), dtype="bf16"),
}

# feed-forward width of the drafter's decoder layer: the LLaMA-3 8B / 70B
# intermediate sizes at d 4096 / 8192 (a toy value below)
FFN_WIDTH = {256: 512, 4096: 14336, 8192: 28672}

WEIGHT_STD = 0.02      # W_proj, W_U ~ N(0, 0.02^2)
LOGIT_STD = 3.0        # target logits ~ N(0, 3^2) per row
DRAFT_NOISE_STD = 0.5  # draft logits = target + N(0, 0.5^2)


def torch_dtype(name):
    return {"fp32": torch.float32, "bf16": torch.bfloat16}[name]


def generator(seed, device="cpu"):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def normal(shape, std, dtype, gen, device="cpu"):
    """N(0, std^2) samples rounded to ``dtype`` (the values both sides see)."""
    x = torch.randn(tuple(shape), generator=gen, dtype=torch.float32, device=device)
    if std != 1.0:
        x.mul_(std)
    return x.to(dtype)


def ctx_lengths(cfg, gen):
    """Per-request committed-prefix lengths: fixed, or uniform in [lo, hi]."""
    lo, hi = cfg["ctx"]
    if lo == hi:
        return torch.full((cfg["B"],), lo, dtype=torch.int32)
    return torch.randint(lo, hi + 1, (cfg["B"],), generator=gen, dtype=torch.int32)


def paged_kv(ctx_lens, Hkv, D, page, dtype, gen, extra_pages=3, device="cpu"):
    """Paged KV cache [P, page, Hkv, D] x2 and a block table [B, max_pages].

    Page ids are a seeded random permutation of the pool so that consecutive
    logical pages are scattered; a few unused pages are added to the pool.
    """
    ctx_lens = [int(c) for c in ctx_lens]
    B = len(ctx_lens)
    npages = [(c + page - 1) // page for c in ctx_lens]
    max_pages = max(1, max(npages))
    P = sum(npages) + extra_pages
    perm = torch.randperm(P, generator=gen)
    table = torch.full((B, max_pages), -1, dtype=torch.int32)
    pos = 0
    for b, n in enumerate(npages):
        table[b, :n] = perm[pos:pos + n].to(torch.int32)
        pos += n
    k_cache = normal((P, page, Hkv, D), 1.0, dtype, gen, device)
    v_cache = normal((P, page, Hkv, D), 1.0, dtype, gen, device)
    return k_cache, v_cache, table


def random_tree(R, max_depth, gen):
    """Random topology: parent of node i uniform among earlier nodes whose
    depth is below ``max_depth``.  Returns (parent_row [R] int32, depth list)."""
    parent = [-1]
    depth = [0]
    for i in range(1, R):
        cands = [j for j in range(i) if depth[j] < max_depth]
        j = cands[int(torch.randint(len(cands), (1,), generator=gen))]
        parent.append(j)
        depth.append(depth[j] + 1)
    return torch.tensor(parent, dtype=torch.int32), depth


def chain_tree(R):
    """A chain: row i's parent is row i-1."""
    return torch.arange(-1, R - 1, dtype=torch.int32)


def random_tokens(shape, V, gen):
    return torch.randint(0, V, tuple(shape), generator=gen, dtype=torch.int32)


def distinct_sibling_tokens(parent_row, V, gen):
    """Tokens for a tree such that siblings carry distinct ids."""
    R = parent_row.shape[0]
    counts = torch.bincount(parent_row[1:].long() + 1) if R > 1 else torch.zeros(1)
    if R > 1 and int(counts.max()) > V:
        raise ValueError("more siblings than vocabulary ids")
    tok = torch.empty(R, dtype=torch.int32)
    used = {}
    for i in range(R):
        p = int(parent_row[i])
        s = used.setdefault(p, set())
        while True:
            t = int(torch.randint(V, (1,), generator=gen))
            if t not in s:
                break
        s.add(t)
        tok[i] = t
    return tok


def target_logits(shape, gen, std=LOGIT_STD, min_top2_gap=None, device="cpu"):
    """fp32 logits ~ N(0, std^2).  With ``min_top2_gap``, rows whose two
    largest entries are closer than the gap are re-drawn (greedy cases)."""
    z = normal(shape, std, torch.float32, gen, device)
    if min_top2_gap is not None:
        flat = z.reshape(-1, shape[-1])
        while True:
            top2 = flat.topk(2, dim=1).values
            bad = (top2[:, 0] - top2[:, 1]) <= min_top2_gap
            if not bool(bad.any()):
                break
            idx = bad.nonzero().flatten()
            flat[idx] = normal((idx.numel(), shape[-1]), std, torch.float32, gen, device)
    return z


def draft_candidates(n_par, k, V, gen, alpha=0.3):
    """Synthetic drafter output for tree-expansion tests: for each parent, k
    distinct ids with log-probabilities of a random distribution over
    ``V`` ids (Dirichlet(alpha) via normalised Gamma draws), sorted
    descending.  Values are fp32."""
    ids = torch.empty((n_par, k), dtype=torch.int32)
    lps = torch.empty((n_par, k), dtype=torch.float32)
    conc = torch.full((V,), float(alpha), dtype=torch.float64)
    for j in range(n_par):
        gam = torch._standard_gamma(conc, generator=gen)
        p = gam / gam.sum()
        top = torch.topk(p, k)
        ids[j] = top.indices.to(torch.int32)
        lps[j] = torch.log(top.values).to(torch.float32)
    return ids, lps


def scaled(cfg_name, **overrides):
    """A copy of a workload's shape dict with fields overridden (small cases)."""
    cfg = dict(CONFIGS[cfg_name])
    cfg.update(overrides)
    return cfg


def n_candidates(cfg):
    """Stored nodes after ``depth`` steps (seed excluded)."""
    k, w = cfg["topk"], cfg["width"]
    n, par = 0, 1
    for _ in range(cfg["depth"]):
        n += par * k
        par = min(w, par * k)
    return n


assert n_candidates(CONFIGS["llama8b"]) == 510
assert n_candidates(CONFIGS["serve64"]) == 14
assert n_candidates(CONFIGS["long4"]) == 456
assert math.isclose(WEIGHT_STD, 0.02)
