"""Plain CPU oracle of the EAGLE hot path.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py`` for who may import it
and for the source keys [E3], [E1], [M7.5], [E3-blog], [Philox]).

Every floating-point result is computed in fp64 from the exact values the GPU
sees (bf16/fp32 inputs widen exactly).  The one exception is the EAGLE-2 path
value used to rank tree candidates: that ranking decides integers (which node
is expanded / kept), the pages fix no precision for it, and so both the oracle
and the kernel take it in fp32 -- one correctly rounded fp32 addition per tree
level, which has a single possible result.
"""

import math

import numpy as np

from .philox import accept_uniforms, race_uniforms, race_uniforms_batch

# ---------------------------------------------------------------------------
# a1: EAGLE-3 multi-layer feature fusion
# ---------------------------------------------------------------------------


def fuse_proj(h_low, h_mid, h_high, w_proj, bias=None):
    """Fused feature g = W_proj [h_low; h_mid; h_high] (+ bias), fp64.

    [E3] section 3.4, "Change 2: The fusion FC layer": the three k-dimensional
    features l, m, h are concatenated into a 3k vector and a fully connected
    layer maps it back to k dimensions; the bias is optional.  [M7.5] 0x08B
    writes the same map as r_t = W_R [f_low; f_mid; f_high], W_R in R^{d x 3d};
    [E3-blog] "What EAGLE-3 changes" as g_t = W_proj @ concat(h_low, h_mid, h_high).

    Shapes: h_* [M, d]; w_proj [d, 3d] (out x in, row-major); bias [d] or None.
    """
    x = np.concatenate([np.asarray(h_low, np.float64), np.asarray(h_mid, np.float64),
                        np.asarray(h_high, np.float64)], axis=1)
    w = np.asarray(w_proj, np.float64)
    if x.shape[1] != w.shape[1]:
        raise ValueError("w_proj must be [d, 3d] with d the width of each feature")
    g = x @ w.T
    if bias is not None:
        g = g + np.asarray(bias, np.float64)[None, :]
    return g


def fuse_proj_accepted(h_low, h_mid, h_high, w_proj, path_rows, accept_len, bias=None):
    """Fused feature of the accepted rows only, fp64.

    [M7.5] 0x05D "Feature And KV Commit": after verification only the
    accepted path is published -- its target features are gathered for the
    next draft round and every other tree row is discarded; [E3] "Stage 2:
    Verification" and section 3.4 "Change 2: The fusion FC layer": the
    drafter's next input is the fusion g = W_proj [l; m; h] of those target
    features.  So the fusion is needed on the accepted rows only.

    Reading (as for the commit): the accepted rows of request b are
    path_rows[b, 0 .. accept_len[b]] in path order; the feature rows of
    request b are rows b*R + row of h_* [B*R, d].  Output [B, Dmax+1, d]:
    slot j <= accept_len[b] holds the fusion of row path_rows[b, j]; the
    other slots are zero (the commit's layout of gathered features).
    """
    path = np.asarray(path_rows)
    acc = np.asarray(accept_len)
    B, slots = path.shape
    hs = [np.asarray(h, np.float64) for h in (h_low, h_mid, h_high)]
    if hs[0].shape[0] % B:
        raise ValueError("h_* must hold B*R rows")
    R = hs[0].shape[0] // B
    d = np.asarray(w_proj).shape[0]
    out = np.zeros((B, slots, d))
    for b in range(B):
        n = int(acc[b]) + 1
        if not 1 <= n <= slots:
            raise ValueError("accept_len out of range")
        rows = [int(path[b, j]) for j in range(n)]
        if any(not 0 <= r < R for r in rows):
            raise ValueError("path row out of range")
        idx = [b * R + r for r in rows]
        out[b, :n] = fuse_proj(hs[0][idx], hs[1][idx], hs[2][idx], w_proj, bias)
    return out


def draft_input(r, token_ids, embed, w_in, bias=None):
    """Drafter input u = W_I [r; e(x)] (+ bias), fp64.

    [M7.5] section 0x08B: after the feature fusion, the fused state r_t is
    joined with the embedding of the sampled token and a second FC,
    u_t = W_I [r_t; e(x_{t+1})] with W_I in R^{d x 2d}, feeds the draft
    decoder.  [E3] section 3.4 ("Input representation", "Input projection FC
    layer"): the k-wide feature and the k-wide token embedding from the target
    model's own table are concatenated to 2k and projected back to k.  [E1]
    "Draft Model Architecture" (FC layer): the same map with a bias,
    h = FC([f; e]); [M7.5] section 0x03 "EAGLE-1 Tensor Path" writes it
    u_t = W_F c_t + b_F.  The embedding is a plain row lookup in the frozen
    table ([E1] "Draft Model Architecture", Embedding Layer).

    Shapes: r [M, d]; token_ids [M] ints in [0, vocab); embed [vocab, d];
    w_in [d, 2d] (out x in); bias [d] or None.  Returns [M, d] fp64.
    """
    r = np.asarray(r, np.float64)
    ids = np.asarray(token_ids).astype(np.int64).reshape(-1)
    table = np.asarray(embed, np.float64)
    if r.ndim != 2 or ids.shape[0] != r.shape[0]:
        raise ValueError("r must be [M, d] and token_ids [M]")
    if ids.size and (ids.min() < 0 or ids.max() >= table.shape[0]):
        raise ValueError("token id outside the embedding table")
    e = table[ids]
    x = np.concatenate([r, e], axis=1)
    w = np.asarray(w_in, np.float64)
    if w.shape != (r.shape[1], 2 * r.shape[1]) or table.shape[1] != r.shape[1]:
        raise ValueError("w_in must be [d, 2d] and embed [vocab, d]")
    u = x @ w.T
    if bias is not None:
        u = u + np.asarray(bias, np.float64)[None, :]
    return u


# ---------------------------------------------------------------------------
# a5 helper: tree ancestry mask (flatten step)
# ---------------------------------------------------------------------------


def ancestor_mask(parent_row, n_rows=None):
    """Visibility bitmask of each flattened tree row.

    Bit j of mask[r] is set iff row j is row r itself or one of its ancestors
    (the root, row 0, is an ancestor of every row).  This is the draft part of
    the visibility rule A(u, v) = 1 iff v in TargetPrefix(u) u DraftAncestors(u)
    u {u} of [M7.5] 0x08C; [E3] "The Attention Mechanism Modifications" states
    the same: a drafted token sees its ancestors but NOT tokens in other
    branches.  Rows at or beyond ``n_rows`` see only themselves.

    parent_row: int array [R] (row 0 = -1, parent_row[i] < i).  Returns uint64 [R].
    """
    parent_row = np.asarray(parent_row)
    R = parent_row.shape[0]
    if R > 64:
        raise ValueError("at most 64 tree rows fit a 64-bit mask")
    n = R if n_rows is None else int(n_rows)
    mask = np.zeros(R, dtype=np.uint64)
    for r in range(R):
        bits = 1 << r
        if r < n:
            j = r
            while True:
                pj = int(parent_row[j])
                if j == 0:
                    break
                if not 0 <= pj < j:
                    raise ValueError("parent_row must be topological: 0 <= parent_row[i] < i")
                bits |= 1 << pj
                j = pj
        mask[r] = np.uint64(bits)
    return mask


# ---------------------------------------------------------------------------
# a2: tree-masked attention against a paged KV cache plus the tree's own rows
# ---------------------------------------------------------------------------


def tree_attn(q, k_tree, v_tree, k_cache, v_cache, block_table, ctx_lens, tree_mask,
              page_size=16, scale=None, sample=None):
    """Tree attention, fp64, max-subtracted softmax.

    For tree row r of request b and query head h (kv head h // G, G = Hq/Hkv):
        keys = the ctx_lens[b] committed prefix tokens (read through the page
               table) followed by the tree rows j with bit j of tree_mask[b, r];
        o    = sum_j softmax_j(scale * q . k_j) v_j,  lse = log sum_j exp(scale q.k_j).
    [M7.5] 0x08C visibility rule (TargetPrefix u DraftAncestors u self);
    [E1] "Tree-Structured Draft Generation": each node attends only to its
    ancestors; [M7.5] 0x05D: tree K/V are temporary branch rows, separate from
    the committed cache.  Readings: scale = 1/sqrt(D); kv head = h // G; Q and
    K arrive with positions already applied.

    Shapes: q [B,R,Hq,D]; k_tree, v_tree [B,R,Hkv,D]; k_cache, v_cache
    [P, page_size, Hkv, D]; block_table [B, max_pages]; ctx_lens [B];
    tree_mask uint64 [B,R].  ``sample``: optional list of (b, r, h) to compute
    only those outputs (returns dict keyed by the tuple).
    Returns (out [B,R,Hq,D], lse [B,R,Hq]) in fp64, or the sampled dict.
    """
    q = np.asarray(q, np.float64)
    B, R, Hq, D = q.shape
    Hkv = k_tree.shape[2]
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    G = Hq // Hkv
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    k_tree = np.asarray(k_tree, np.float64)
    v_tree = np.asarray(v_tree, np.float64)
    block_table = np.asarray(block_table)
    ctx_lens = np.asarray(ctx_lens)
    tree_mask = np.asarray(tree_mask, dtype=np.uint64)

    def prefix(b):
        n = int(ctx_lens[b])
        npg = (n + page_size - 1) // page_size
        pages = block_table[b, :npg].astype(np.int64)
        kc = np.asarray(k_cache[pages], np.float64).reshape(npg * page_size, Hkv, D)[:n]
        vc = np.asarray(v_cache[pages], np.float64).reshape(npg * page_size, Hkv, D)[:n]
        return kc, vc

    def one_row(b, r, kc, vc, heads):
        m = int(tree_mask[b, r])
        vis = [j for j in range(R) if (m >> j) & 1]
        keys = np.concatenate([kc, k_tree[b, vis]], axis=0)  # [n+t, Hkv, D]
        vals = np.concatenate([vc, v_tree[b, vis]], axis=0)
        res = {}
        for h in heads:
            kv = h // G
            s = scale * (keys[:, kv, :] @ q[b, r, h])
            mx = s.max()
            w = np.exp(s - mx)
            z = w.sum()
            res[h] = ((w @ vals[:, kv, :]) / z, mx + math.log(z))
        return res

    if sample is not None:
        out = {}
        by_b = {}
        for (b, r, h) in sample:
            by_b.setdefault(b, []).append((r, h))
        for b, items in by_b.items():
            kc, vc = prefix(b)
            for r in sorted({r for r, _ in items}):
                heads = [h for rr, h in items if rr == r]
                for h, val in one_row(b, r, kc, vc, heads).items():
                    out[(b, r, h)] = val
        return out

    out = np.zeros((B, R, Hq, D))
    lse = np.zeros((B, R, Hq))
    for b in range(B):
        kc, vc = prefix(b)
        for r in range(R):
            for h, (o, l) in one_row(b, r, kc, vc, range(Hq)).items():
                out[b, r, h] = o
                lse[b, r, h] = l
    return out, lse


# ---------------------------------------------------------------------------
# a3: LM head with per-row top-k and log-softmax
# ---------------------------------------------------------------------------


def lmhead_topk(x, w_lm, k, temperature=1.0, bias=None, rows=None):
    """Vocabulary logits z = W_U a (+ b), per-row top-k ids and log-probs.

    [E3] "Output path to LM head": logits_i = W_LM a_i + b_LM (bias if
    present), tokens drawn from softmax(logits / T).  [E1] "Tree-Structured
    Draft Generation": in greedy mode the top-k tokens become child nodes.
    [M7.5] 0x06B: a child's confidence is its conditional probability under
    the parent's prefix, normalised over the whole vocabulary ("omitted
    vocabulary mass is allowed").  Readings: top-k order is z descending with
    ties to the lower id; log-prob = z/T - logsumexp(z/T) over all V.

    x [M, d]; w_lm [V, d]; bias [V] or None; rows: optional row subset.
    Returns dict(ids [M,k] int64, logprobs [M,k], row_max [M] = max z/T,
    row_sumexp [M] = sum exp(z/T - row_max), z [M, V] fp64).
    """
    if not (1 <= k):
        raise ValueError("k must be >= 1")
    if not temperature > 0:
        raise ValueError("temperature must be > 0")
    x = np.asarray(x, np.float64)
    if rows is not None:
        x = x[np.asarray(rows)]
    w = np.asarray(w_lm, np.float64)
    V = w.shape[0]
    if k > V:
        raise ValueError("k must not exceed V")
    z = x @ w.T
    if bias is not None:
        z = z + np.asarray(bias, np.float64)[None, :]
    y = z / temperature
    m = y.max(axis=1)
    s = np.exp(y - m[:, None]).sum(axis=1)
    lse = m + np.log(s)
    vid = np.arange(V)
    ids = np.empty((z.shape[0], k), dtype=np.int64)
    for i in range(z.shape[0]):
        ids[i] = np.lexsort((vid, -z[i]))[:k]
    logprobs = np.take_along_axis(y, ids, axis=1) - lse[:, None]
    return dict(ids=ids, logprobs=logprobs, row_max=m, row_sumexp=s, z=z)


# ---------------------------------------------------------------------------
# a4/a5: EAGLE-2 dynamic tree expansion, rerank and flatten
# ---------------------------------------------------------------------------

EPSILON = 1e-12
LOG_EPS32 = np.float32(math.log(EPSILON))  # ranking floor log(1e-12) in fp32
MASS_TOL = 1e-4  # sibling-mass slack for fp32 log-probabilities (reading)


def _key(st, n):
    """Ranking key (-log V, depth, node_id) of [M7.5] 0x06B (fp32 log V)."""
    return (-float(st["logv"][n]), st["depth"][n], n)


def tree_expand_init(root_token):
    """Tree store holding only the seed: depth 0, log path value 0, node_id 0.

    [M7.5] 0x06B: the seed is the context anchor at depth zero with log path
    value zero and is not counted in the verification budget.
    """
    return dict(parent=[-1], token=[int(root_token)], logv=[np.float32(0.0)],
                depth=[0], frontier=[0])


def tree_expand_step(st, cand_ids, cand_logprobs, width):
    """One expansion step of EAGLE-2 ([M7.5] 0x06A, 0x06B).

    ``st["frontier"]`` is the list of expandable parents (node ids, in key
    order) that the drafter was run on; row j of ``cand_ids`` /
    ``cand_logprobs`` [n_par, k] holds the top-k children of frontier[j] with
    their log conditional probabilities.  Every child becomes a stored node:
        log V(child) = log V(parent) + log max(c, 1e-12)      (fp32)
    with log c clamped to <= 0, depth = parent depth + 1 and node ids in
    creation order (parent slot, then child rank); an id < 0 marks a missing
    alternative and creates no node.  The next expandable set is
    the top-``width`` of the new nodes by (-log V, depth, node_id).

    Validation follows the pages' eagle2_tree checks: finite probabilities
    (log-prob NaN or +inf rejected), no duplicate token under one parent,
    sibling mass <= 1 (with MASS_TOL slack for fp32 inputs).
    Returns the new expandable list (also stored in st["frontier"]).
    """
    if type(width) is not int or width < 1:
        raise ValueError("expansion width must be a positive integer")
    cand_ids = np.asarray(cand_ids)
    cand_lp = np.asarray(cand_logprobs, dtype=np.float32)
    parents = list(st["frontier"])
    if cand_ids.shape[0] < len(parents) or cand_lp.shape != cand_ids.shape:
        raise ValueError("need one candidate row per expandable parent")
    new = _add_children(st, parents, cand_ids, cand_lp, [cand_ids.shape[1]] * len(parents))
    st["frontier"] = sorted(new, key=lambda n: _key(st, n))[:width]
    return list(st["frontier"])


def _add_children(st, parents, cand_ids, cand_lp, limits):
    """Store the children of each parent (ranks below its limit) with the
    values and validation of ``tree_expand_step``; returns their node ids."""
    new = []
    for j, p in enumerate(parents):
        seen = set()
        mass = 0.0
        for i in range(min(int(limits[j]), cand_ids.shape[1])):
            tok = int(cand_ids[j, i])
            if tok < 0:  # fewer than k alternatives for this parent
                continue
            lp = cand_lp[j, i]
            if np.isnan(lp) or lp == np.inf:
                raise ValueError("confidence must be a finite probability")
            if tok in seen:
                raise ValueError("duplicate token alternative under one parent")
            seen.add(tok)
            lp = min(lp, np.float32(0.0))
            mass += math.exp(float(lp))
            if mass > 1.0 + MASS_TOL:
                raise ValueError("sibling probability mass exceeds one")
            term = max(lp, LOG_EPS32)
            logv = np.float32(st["logv"][p] + term)  # one fp32 addition
            n = len(st["parent"])
            st["parent"].append(p)
            st["token"].append(tok)
            st["logv"].append(logv)
            st["depth"].append(st["depth"][p] + 1)
            new.append(n)
    return new


def static_tree_step(st, cand_ids, cand_logprobs, fanout):
    """One depth of a static draft tree (EAGLE-1, [E1] "Tree-Structured Draft
    Generation": a fixed tree, the root branching into its top-4 tokens and
    deeper nodes into fewer).  The tree is given depth by depth as the number
    of children of each node of the current depth, in creation order:
    frontier[j] takes the tokens of its top-``fanout[j]`` candidates (ranks
    0 .. fanout[j]-1).  Values, depths, node ids and validation are those of
    ``tree_expand_step``; the next frontier is every new node, in creation
    order (no reranking: the shape is fixed)."""
    cand_ids = np.asarray(cand_ids)
    cand_lp = np.asarray(cand_logprobs, dtype=np.float32)
    parents = list(st["frontier"])
    fanout = [int(f) for f in fanout]
    if len(fanout) < len(parents) or cand_ids.shape[0] < len(parents) or cand_lp.shape != cand_ids.shape:
        raise ValueError("need one fan-out and one candidate row per node of the depth")
    if any(f < 0 or f > cand_ids.shape[1] for f in fanout[:len(parents)]):
        raise ValueError("a fan-out must lie in [0, k]")
    st["frontier"] = _add_children(st, parents, cand_ids, cand_lp, fanout)
    return list(st["frontier"])


def tree_expand_finalize(st, budget, ctx_len=0, R_out=None):
    """Global rerank + flatten ([M7.5] 0x06A, 0x06B, 0x05C).

    selected = the first ``budget`` non-root nodes in (-log V, depth, node_id)
    order; because a child's value never exceeds its parent's and ties go to
    the shallower node, every prefix of that order is ancestor-closed, so no
    ancestors are added afterwards.  Flattened rows: row 0 = seed, row i =
    selected[i-1]; parent_row = row of the parent (seed -> 0); depth; position
    = ctx_len + depth ([M7.5] 0x05C ancestry-aware positions); mask = ancestry
    bits (see ``ancestor_mask``); node_id = retrieve map from row to node.
    Rows past n_rows (when R_out is larger) are padding: token -1,
    parent_row -1, depth 0, position ctx_len, node_id -1, mask = own bit.
    """
    for value in (budget,):
        if type(value) is not int or value < 0:
            raise ValueError("verification budget must be a nonnegative integer")
    nodes = list(range(1, len(st["parent"])))
    selected = sorted(nodes, key=lambda n: _key(st, n))[:budget]
    n_rows = 1 + len(selected)
    R = n_rows if R_out is None else int(R_out)
    if R < n_rows:
        raise ValueError("R_out smaller than 1 + budget")
    row_of = {0: 0}
    for i, n in enumerate(selected):
        row_of[n] = i + 1
    token = np.full(R, -1, np.int64)
    parent_row = np.full(R, -1, np.int64)
    depth = np.zeros(R, np.int64)
    node_id = np.full(R, -1, np.int64)
    token[0] = st["token"][0]
    node_id[0] = 0
    for i, n in enumerate(selected):
        p = st["parent"][n]
        if p not in row_of or row_of[p] >= i + 1:
            raise AssertionError("selection is not ancestor-closed")
        token[i + 1] = st["token"][n]
        parent_row[i + 1] = row_of[p]
        depth[i + 1] = st["depth"][n]
        node_id[i + 1] = n
    mask = ancestor_mask(parent_row, n_rows) if R <= 64 else None
    position = ctx_len + depth
    return dict(token=token, parent_row=parent_row, depth=depth, mask=mask,
                node_id=node_id, position=position, n_rows=n_rows)


def eagle2_tree(draft, root_token, expand_width, verify_budget, max_depth, ctx_len=0):
    """The pages' eagle2_tree composition ([M7.5] 0x06B) over a ``draft``
    callback: draft(step, parents) -> (cand_ids [len(parents), k],
    cand_logprobs [len(parents), k]).  Returns (flat tree dict, tree store)."""
    if type(expand_width) is not int or expand_width < 1:
        raise ValueError("expansion width must be a positive integer")
    for value in (verify_budget, max_depth):
        if type(value) is not int or value < 0:
            raise ValueError("verification budget and depth must be nonnegative integers")
    st = tree_expand_init(root_token)
    if verify_budget == 0:
        return tree_expand_finalize(st, 0, ctx_len), st
    for step in range(max_depth):
        if not st["frontier"]:
            break
        ids, lps = draft(step, list(st["frontier"]))
        tree_expand_step(st, ids, lps, expand_width)
    return tree_expand_finalize(st, verify_budget, ctx_len), st


# ---------------------------------------------------------------------------
# a6/a7: lossless tree verification
# ---------------------------------------------------------------------------


def _softmax64(row, temperature):
    y = np.asarray(row, np.float64) / temperature
    y = y - y.max()
    w = np.exp(y)
    return w / w.sum()


def _argmax_low(row):
    row = np.asarray(row)
    return int(np.flatnonzero(row == row.max())[0])


def tree_verify(parent_row, token, temperature, max_depth, n_rows=None,
                target_logits=None, target_argmax=None, draft_logits=None,
                mode="deterministic", seed=0, offset=0, accept_u=None, race_u=None):
    """Tree verification: greedy longest accepted path, or multi-round
    speculative sampling with residual correction.

    [E1] "Verification Phase: Multi-Round Speculative Sampling on Trees"
    (the paper's Algorithm 1): the candidates under one node are tried in
    order; candidate t_i is accepted when r < p(t_i) / p_hat_i(t_i) with
    r ~ U(0,1); after a rejection p <- norm(max(0, p - p_hat_i)) (read as the
    vector update: the page prints it garbled as a scalar); if every candidate
    is rejected a token is drawn from the final p.  [E3] "Stage 2:
    Verification" gives the same min(1, p/p_hat) rule.  At T = 0 p is the
    one-hot argmax of the target logits (lowest id on ties), which reduces the
    walk to "accept the child whose token is the parent row's argmax".

    Target logits row r give the distribution of the children of row r.
    ``mode``:
      * "deterministic" (default; EAGLE-2 trees are deterministic top-k, not
        draws): proposal of each candidate is the point mass on its token, so
        accept iff u < p(t) and on rejection p loses t and is renormalised;
      * "sampled": the siblings were i.i.d. draws from q = softmax(draft
        logits of the parent row / T): Algorithm 1 verbatim with p_hat = q.
    Readings: the children of a row are tried in row order; a residual whose
    mass is zero leaves p unchanged; the final draw is an exponential race
    argmax_y (log w_y - log(-log u_y)) over allowed ids (ties to lower id).

    Uniforms come from ``oracle.philox`` (accept test per row, race per id) or
    from ``accept_u`` [B,R] / ``race_u`` callable(b) -> [V] overrides.
    Returns dict(accept_len [B], path_rows [B, max_depth+1] (row 0 first,
    -1 padded), out_tokens [B, max_depth+1] (accepted tokens then the bonus
    token, -1 padded), margins: list of (kind, b, |decision margin|)).
    """
    parent_row = np.asarray(parent_row)
    token = np.asarray(token)
    B, R = parent_row.shape
    greedy = temperature == 0
    if temperature < 0 or not math.isfinite(temperature):
        raise ValueError("temperature must be finite and >= 0")
    if mode not in ("deterministic", "sampled"):
        raise ValueError("unknown proposal mode")
    if mode == "sampled" and (greedy or draft_logits is None):
        raise ValueError("sampled proposals need T > 0 and draft logits")
    if greedy and target_logits is None and target_argmax is None:
        raise ValueError("greedy verification needs target logits or argmax")
    if not greedy and target_logits is None:
        raise ValueError("stochastic verification needs target logits")
    if accept_u is None and not greedy:
        accept_u = accept_uniforms(seed, offset, B, R)
    V = None if target_logits is None else np.asarray(target_logits).shape[2]

    accept_len = np.zeros(B, np.int64)
    path_rows = np.full((B, max_depth + 1), -1, np.int64)
    out_tokens = np.full((B, max_depth + 1), -1, np.int64)
    margins = []
    for b in range(B):
        n = R if n_rows is None else int(n_rows[b])
        if not 1 <= n <= R or parent_row[b, 0] != -1:
            raise ValueError("row 0 must be the root and 1 <= n_rows <= R")
        for i in range(1, n):
            if not 0 <= parent_row[b, i] < i:
                raise ValueError("parent_row must be topological")
        cur = 0
        path = [0]
        toks = []
        while True:
            children = [c for c in range(cur + 1, n) if parent_row[b, c] == cur]
            accepted = None
            if greedy:
                a = (int(target_argmax[b, cur]) if target_argmax is not None
                     else _argmax_low(target_logits[b, cur]))
                for c in children:
                    if int(token[b, c]) == a:
                        accepted = c
                        break
                bonus_dist = None
            else:
                p = _softmax64(target_logits[b, cur], temperature)
                q = (_softmax64(draft_logits[b, cur], temperature)
                     if mode == "sampled" else None)
                for c in children:
                    t = int(token[b, c])
                    u = float(accept_u[b, c])
                    if mode == "deterministic":
                        ratio = p[t]
                    else:
                        ratio = p[t] / q[t] if q[t] > 0 else (math.inf if p[t] > 0 else 0.0)
                    margins.append(("accept", b, abs(u - ratio) if math.isfinite(ratio) else math.inf))
                    if u < ratio:
                        accepted = c
                        break
                    if mode == "deterministic":
                        res = p.copy()
                        res[t] = 0.0
                    else:
                        res = np.maximum(0.0, p - q)
                    mass = res.sum()
                    if mass > 0:
                        p = res / mass
                bonus_dist = p
            if accepted is None:
                if greedy:
                    bonus = a
                else:
                    ur = race_u(b) if race_u is not None else race_uniforms(seed, offset, b, V)
                    with np.errstate(divide="ignore"):
                        keyv = np.where(bonus_dist > 0,
                                        np.log(bonus_dist) - np.log(-np.log(ur)), -np.inf)
                    bonus = _argmax_low(keyv)
                    top2 = np.sort(keyv)[-2:]
                    margins.append(("race", b, float(top2[1] - top2[0])))
                toks.append(bonus)
                break
            if len(path) > max_depth:
                raise ValueError("tree deeper than max_depth")
            path.append(accepted)
            toks.append(int(token[b, accepted]))
            cur = accepted
        accept_len[b] = len(path) - 1
        path_rows[b, :len(path)] = path
        out_tokens[b, :len(toks)] = toks
    return dict(accept_len=accept_len, path_rows=path_rows, out_tokens=out_tokens,
                margins=margins)


# ---------------------------------------------------------------------------
# K8 (follow-on): stochastic-verification statistics from the verification
# LM head, so that verification never needs the [B, R, V] target logits
# ---------------------------------------------------------------------------


def verify_stats(x, w_lm, parent_row, token, temperature, race_k, seed=0, offset=0, bias=None,
                 n_rows=None, race_u=None, rows=None):
    """Everything deterministic-proposal stochastic verification reads from
    the target logits z = W_U a (+ b) of the verify rows, computed from the
    verification LM head's inputs instead of from stored logits.

    Rows are [B * R] (request-major).  The walk of [E1] "Verification Phase:
    Multi-Round Speculative Sampling on Trees" (deterministic point-mass
    proposals) reads, for the current row r: p(t) = exp(z_r[t]/T) / sum_v
    exp(z_r[v]/T) for each child token t, and at the stop row the
    exponential race over the ids not rejected there.  So it needs
      row_max[r] = max_v z_r/T, row_sumexp[r] = sum_v exp(z_r/T - row_max[r]);
      child_logit[c] = z[parent(c)][token(c)] for each row c >= 1 (0 for the
        root and for rows past n_rows);
      the race candidates of every row: the race_k ids of largest key
        z_r[y]/T - log(-log u_{b,y}) (ties to the lower id), sorted, with their
        keys.  The race's renormalisation constant is common to all allowed
        ids, so the stop-row winner is the first candidate not rejected there;
        race_k must exceed the number of children of any row.
    Uniforms: oracle.philox race uniforms per (request, id), or race_u [B, V].
    rows: optional subset of row indices to compute (the others are NaN / -1).
    Returns dict(row_max [B*R], row_sumexp [B*R], child_logit [B*R],
    race_ids [B*R, race_k] int64, race_keys [B*R, race_k]).
    """
    parent_row = np.asarray(parent_row)
    token = np.asarray(token)
    B, R = parent_row.shape
    if not temperature > 0:
        raise ValueError("temperature must be > 0")
    x = np.asarray(x, np.float64)
    w = np.asarray(w_lm, np.float64)
    if x.shape[0] != B * R:
        raise ValueError("x must hold B * R rows")
    V = w.shape[0]
    if not 1 <= race_k <= V:
        raise ValueError("race_k must be in 1..V")
    bvec = None if bias is None else np.asarray(bias, np.float64)
    todo = range(B * R) if rows is None else sorted(set(int(r) for r in rows))
    need_b = sorted(set(r // R for r in todo))
    if race_u is not None:
        ur = {b: np.asarray(race_u, np.float64)[b] for b in need_b}
    else:
        ur = {b: race_uniforms(seed, offset, b, V) for b in need_b}
    row_max = np.full(B * R, np.nan)
    row_sumexp = np.full(B * R, np.nan)
    child_logit = np.full(B * R, np.nan)
    race_ids = np.full((B * R, race_k), -1, np.int64)
    race_keys = np.full((B * R, race_k), np.nan)
    vid = np.arange(V)
    for row in todo:
        b, c = divmod(row, R)
        z = w @ x[row]
        if bvec is not None:
            z = z + bvec
        y = z / temperature
        row_max[row] = y.max()
        row_sumexp[row] = np.exp(y - row_max[row]).sum()
        key = y - np.log(-np.log(ur[b]))
        order = np.lexsort((vid, -key))[:race_k]
        race_ids[row] = order
        race_keys[row] = key[order]
        n = R if n_rows is None else int(n_rows[b])
        if 1 <= c < n:
            p, t = int(parent_row[b, c]), int(token[b, c])
            child_logit[row] = float(np.dot(x[b * R + p], w[t])) + (0.0 if bvec is None else bvec[t])
        else:
            child_logit[row] = 0.0
    return dict(row_max=row_max, row_sumexp=row_sumexp, child_logit=child_logit,
                race_ids=race_ids, race_keys=race_keys)


def tree_verify_stats(parent_row, token, temperature, max_depth, row_max, row_sumexp,
                      child_logit, race_ids, n_rows=None, seed=0, offset=0, accept_u=None):
    """Deterministic-proposal stochastic verification from verify_stats
    outputs ([E1] "Verification Phase", the deterministic reading of
    tree_verify): children of the current row are tried in row order; child c
    with token t is accepted when u_c < p(t) / (1 - sum of p over the
    distinct tokens already rejected at this row), p(t) = exp(child_logit[c]/T
    - row_max) / row_sumexp; a repeated token has p = 0.  At the stop row the
    bonus token is the first race candidate not rejected there.
    Same outputs as tree_verify (accept_len, path_rows, out_tokens, margins).
    """
    parent_row = np.asarray(parent_row)
    token = np.asarray(token)
    B, R = parent_row.shape
    if not temperature > 0:
        raise ValueError("temperature must be > 0")
    if accept_u is None:
        accept_u = accept_uniforms(seed, offset, B, R)
    accept_len = np.zeros(B, np.int64)
    path_rows = np.full((B, max_depth + 1), -1, np.int64)
    out_tokens = np.full((B, max_depth + 1), -1, np.int64)
    margins = []
    for b in range(B):
        n = R if n_rows is None else int(n_rows[b])
        if not 1 <= n <= R or parent_row[b, 0] != -1:
            raise ValueError("row 0 must be the root and 1 <= n_rows <= R")
        for i in range(1, n):
            if not 0 <= parent_row[b, i] < i:
                raise ValueError("parent_row must be topological")
        cur, path, toks = 0, [0], []
        while True:
            children = [c for c in range(cur + 1, n) if parent_row[b, c] == cur]
            rm, rs = float(row_max[b * R + cur]), float(row_sumexp[b * R + cur])
            rejected, rem, accepted = [], 1.0, None
            for c in children:
                t = int(token[b, c])
                pt = 0.0 if t in rejected else math.exp(child_logit[b * R + c] / temperature - rm) / rs
                ratio = pt / rem
                u = float(accept_u[b, c])
                margins.append(("accept", b, abs(u - ratio)))
                if u < ratio:
                    accepted = c
                    break
                if t not in rejected and rem - pt > 0:
                    rem -= pt
                    rejected.append(t)
            if accepted is None:
                cands = [int(v) for v in race_ids[b * R + cur] if int(v) not in rejected]
                if not cands:
                    raise ValueError("race_k too small: every candidate was rejected")
                toks.append(cands[0])
                break
            if len(path) > max_depth:
                raise ValueError("tree deeper than max_depth")
            path.append(accepted)
            toks.append(int(token[b, accepted]))
            cur = accepted
        accept_len[b] = len(path) - 1
        path_rows[b, :len(path)] = path
        out_tokens[b, :len(toks)] = toks
    return dict(accept_len=accept_len, path_rows=path_rows, out_tokens=out_tokens,
                margins=margins)


# ---------------------------------------------------------------------------
# K9 (follow-on): publish the verified path
# ---------------------------------------------------------------------------


def tree_commit(k_cache, v_cache, block_table, ctx_lens, k_tree, v_tree, path_rows, accept_len,
                features=None):
    """Publish the verified path of each request ([M7.5] 0x05D "Feature And
    KV Commit", the publish_verified_path transaction): the target K/V of the
    accepted rows are appended to the committed prefix and their target
    features are gathered for the next draft round; every other tree row is
    discarded.  Rows are taken by their flat row index (the path from
    verification), never by token id.

    Reading: the accepted rows are path_rows[b, 0 .. accept_len[b]] -- row 0
    (the root: the previous round's frontier token, whose K/V this verify
    forward computed) and the accepted drafted rows, in path order.  They
    land at positions ctx .. ctx + accept_len of the paged cache (page =
    block_table[b, pos // 16], slot = pos % 16) and ctx grows by
    accept_len + 1.  The new frontier (bonus) token is not one of the verified
    rows: its K/V and feature need a later target append, so nothing is
    written for it.

    k_cache, v_cache [P, 16, Hkv, D]; block_table [B, max_pages];
    ctx_lens [B]; k_tree, v_tree [B, R, Hkv, D]; path_rows [B, max_depth+1];
    accept_len [B]; features [B*R, F] or None.
    Returns dict(k_cache, v_cache (copies), ctx_lens [B],
    features [B, max_depth+1, F] (zeros past accept_len) or None).
    """
    kc = np.array(k_cache, copy=True)
    vc = np.array(v_cache, copy=True)
    table = np.asarray(block_table)
    ctx = np.array(ctx_lens, dtype=np.int64, copy=True)
    path = np.asarray(path_rows)
    acc = np.asarray(accept_len)
    B, R = np.asarray(k_tree).shape[:2]
    P = kc.shape[0]
    out_f = None
    if features is not None:
        f = np.asarray(features)
        out_f = np.zeros((B, path.shape[1], f.shape[1]), dtype=f.dtype)
    for b in range(B):
        n = int(acc[b]) + 1
        if not 1 <= n <= path.shape[1]:
            raise ValueError("accept_len out of range")
        for i in range(n):
            row = int(path[b, i])
            if not 0 <= row < R:
                raise ValueError("path row out of range")
            pos = int(ctx[b]) + i
            if pos // 16 >= table.shape[1]:
                raise ValueError("no page for the committed position")
            page = int(table[b, pos // 16])
            if not 0 <= page < P:
                raise ValueError("page id out of range")
            kc[page, pos % 16] = k_tree[b, row]
            vc[page, pos % 16] = v_tree[b, row]
            if out_f is not None:
                out_f[b, i] = f[b * R + row]
        ctx[b] += n
    return dict(k_cache=kc, v_cache=vc, ctx_lens=ctx, features=out_f)


# ---------------------------------------------------------------------------
# drafter decoder layer (the step after the input FC)
# ---------------------------------------------------------------------------
# [E3] section 3.4 "The transformer decoder layer": one standard decoder layer
# -- self-attention and a position-wise feed-forward sublayer, each with a
# residual connection and normalisation.  The pages fix no further detail;
# the reading taken is the form of the LLaMA-family targets the pages
# evaluate ([E3] section 6, Limitation 6: pre-normalisation, SwiGLU, rotary
# position embeddings, grouped-query attention): RMSNorm before each
# sublayer, rotate-half RoPE on q and k, GQA attention, SwiGLU feed-forward,
# no biases.  The attention is tree attention over the drafter's own KV
# ([M7.5] 0x03C "The Drafter Has Its Own KV State"; 0x05B: the nodes of one
# depth are expanded in one pass with tree attention, each node holding its
# position and its draft-KV row).


def linear(x, w, bias=None, residual=None):
    """y = x w^T (+ bias) (+ residual), fp64: the projections of the decoder
    layer ([E3] section 3.4 "The transformer decoder layer")."""
    y = np.asarray(x, np.float64) @ np.asarray(w, np.float64).T
    if bias is not None:
        y = y + np.asarray(bias, np.float64)[None, :]
    if residual is not None:
        y = y + np.asarray(residual, np.float64)
    return y


def rms_norm(x, w, eps):
    """y = x / sqrt(mean(x^2) + eps) * w over the last axis, fp64."""
    x = np.asarray(x, np.float64)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps) * np.asarray(w, np.float64)


def rope(x, positions, theta):
    """Rotate-half rotary embedding of x [..., D] at integer positions
    (broadcast over x.shape[:-1]): element pair (i, i + D/2) is rotated by
    the angle position * theta^(-2i/D)."""
    x = np.asarray(x, np.float64)
    D = x.shape[-1]
    half = D // 2
    inv = np.power(float(theta), -2.0 * np.arange(half) / D)
    ang = np.asarray(positions, np.float64)[..., None] * inv
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def silu(x):
    x = np.asarray(x, np.float64)
    return x / (1.0 + np.exp(-x))


def draft_layer(x, weights, positions, k_cache, v_cache, block_table, ctx_lens, k_tree, v_tree,
                tree_mask, r0, Hq, Hkv, eps=1e-5, theta=500000.0, page_size=16, store=None):
    """One drafter decoder layer over the B x W new tree nodes of one depth.

    x [B*W, d] rows of the input (request-major).  weights: dict with
    norm1 [d], qkv [(Hq + 2 Hkv) D, d] (q heads, then k heads, then v heads),
    o [d, Hq D], norm2 [d], gu [2 I, d] (gate rows, then up rows), down [d, I].
    positions [B, W].  The drafter's prefix K/V come from the paged cache;
    k_tree / v_tree [B, Rmax, Hkv, D] hold the earlier nodes' rows, and the new
    node j of request b takes row r0 + j; tree_mask [B, Rmax] (bit i of row r:
    row i is visible).  ``store``: optional rounding applied wherever the
    layer stores an intermediate tensor (identity by default).

    Returns (out [B*W, d], k_new [B, W, Hkv, D], v_new [B, W, Hkv, D]).
    """
    st = store if store is not None else (lambda a: a)
    x = np.asarray(x, np.float64)
    positions = np.asarray(positions)
    B, W = positions.shape
    M, d = x.shape
    D = np.asarray(weights["qkv"]).shape[0] // (Hq + 2 * Hkv)
    Rmax = k_tree.shape[1]
    if M != B * W or r0 < 0 or r0 + W > Rmax:
        raise ValueError("x must be [B*W, d] and the new rows must fit the tree arrays")
    h = st(rms_norm(x, weights["norm1"], eps))
    qkv = st(h @ np.asarray(weights["qkv"], np.float64).T)
    q = qkv[:, :Hq * D].reshape(M, Hq, D)
    k = qkv[:, Hq * D:(Hq + Hkv) * D].reshape(M, Hkv, D)
    v = qkv[:, (Hq + Hkv) * D:].reshape(M, Hkv, D)
    pos = positions.reshape(M)[:, None]
    q, k = st(rope(q, pos, theta)), st(rope(k, pos, theta))
    kt = np.array(k_tree, np.float64)
    vt = np.array(v_tree, np.float64)
    qt = np.zeros((B, Rmax, Hq, D))
    for b in range(B):
        for j in range(W):
            kt[b, r0 + j] = k[b * W + j]
            vt[b, r0 + j] = v[b * W + j]
            qt[b, r0 + j] = q[b * W + j]
    want = [(b, r0 + j, hh) for b in range(B) for j in range(W) for hh in range(Hq)]
    att = tree_attn(qt, kt, vt, k_cache, v_cache, block_table, ctx_lens, tree_mask,
                    page_size=page_size, sample=want)
    a = np.zeros((M, Hq, D))
    for b in range(B):
        for j in range(W):
            for hh in range(Hq):
                a[b * W + j, hh] = att[(b, r0 + j, hh)][0]
    a = st(a.reshape(M, Hq * D))
    x1 = st(x + a @ np.asarray(weights["o"], np.float64).T)
    h2 = st(rms_norm(x1, weights["norm2"], eps))
    I = np.asarray(weights["down"]).shape[1]
    gu = st(h2 @ np.asarray(weights["gu"], np.float64).T)
    act = st(silu(gu[:, :I]) * gu[:, I:])
    out = st(x1 + act @ np.asarray(weights["down"], np.float64).T)
    return out, k.reshape(B, W, Hkv, D), v.reshape(B, W, Hkv, D)


def draft_rows(step, width, st, node_row, row_mask, ctx_len, prev, root_token=None):
    """Bookkeeping of one drafter pass over the nodes of one depth ([M7.5]
    0x05B: the nodes of a depth are expanded in one pass, each holding its
    token, parent index, position and draft-KV row; [E3] "Input
    representation": a drafted node's feature input is the drafter's own
    output at its parent, the target's fused feature only at the root).

    Reading: the root is processed first (step 0, row 0, feature input = the
    target feature g, its token the seed token); at step s >= 1 slot j of the
    frontier (the nodes the expansion step s - 1 chose) takes row
    1 + (s - 1) * width + j, sees its parent's row and the rows that row sees,
    sits at position ctx + depth, and its feature input is the drafter output
    of its parent's slot at step s - 1 (``prev`` rows, slot order).

    st: the expansion store (parent / token / depth / frontier), or None at
    step 0.  node_row: dict node -> row (updated); row_mask: dict row -> bits
    (updated).  Returns (rows, tokens, positions, feature inputs [n, d])."""
    prev = np.asarray(prev, np.float64)
    if step == 0:
        node_row[0] = 0
        row_mask[0] = 1
        return [0], [int(root_token)], [int(ctx_len)], prev[:1].copy()
    rows, toks, pos, feats = [], [], [], []
    r0_prev = 0 if step == 1 else 1 + (step - 2) * width
    for j, n in enumerate(st["frontier"]):
        p = st["parent"][n]
        if p not in node_row:
            raise ValueError("a frontier node whose parent the drafter has not processed")
        prow = node_row[p]
        row = 1 + (step - 1) * width + j
        node_row[n] = row
        row_mask[row] = row_mask[prow] | (1 << row)
        rows.append(row)
        toks.append(int(st["token"][n]))
        pos.append(int(ctx_len) + int(st["depth"][n]))
        feats.append(prev[prow - r0_prev])
    return rows, toks, pos, np.asarray(feats).reshape(len(rows), prev.shape[1])
