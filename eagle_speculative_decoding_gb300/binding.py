"""Thin ctypes binding of libeagle_gb300.so (include/eagle.h).

Argument marshalling only: every function takes torch tensors that already
live on the current CUDA device, passes their data pointers, shapes and the
current stream to the C entry point of the same name, and raises if the call
returns an error.  No computation happens here and there is no fallback: if
the library is missing, the first call raises.
"""
import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libeagle_gb300.so")

EAGLE_FP32, EAGLE_BF16 = 0, 1
EAGLE_PROPOSAL_DETERMINISTIC, EAGLE_PROPOSAL_SAMPLED = 0, 1
STATUS = {0: "EAGLE_OK", 1: "EAGLE_ERR_INVALID_ARG", 2: "EAGLE_ERR_UNSUPPORTED",
          3: "EAGLE_ERR_WORKSPACE", 4: "EAGLE_ERR_CUDA", 5: "EAGLE_ERR_BAD_TREE",
          6: "EAGLE_ERR_BAD_KV", 7: "EAGLE_ERR_NONFINITE", 8: "EAGLE_ERR_TIMEOUT"}

_P, _I, _F, _Z, _U64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.c_uint64

_SIGS = {
    "eagle_status_string": (ctypes.c_char_p, [_I]),
    "eagle_read_status": (_I, [_P, _P, _P]),
    "eagle_launch_count": (_U64, []),
    "eagle_selftest_wait_timeout": (_I, [ctypes.c_uint, _P, _P]),
    "eagle_fuse_proj_workspace_size": (_Z, [_I, _I, _I]),
    "eagle_fuse_proj": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _P, _Z, _P, _P]),
    "eagle_fuse_proj_accepted_workspace_size": (_Z, [_I, _I, _I, _I]),
    "eagle_fuse_proj_accepted": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _Z, _P, _P]),
    "eagle_draft_input_workspace_size": (_Z, [_I, _I, _I]),
    "eagle_linear_workspace_size": (_Z, [_I, _I, _I, _I]),
    "eagle_linear": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _Z, _P, _P]),
    "eagle_draft_layer_workspace_size": (_Z, [_I, _I, _I, _I, _I, _I, _I, _I, _I, _I]),
    "eagle_draft_rows": (_I, [_I, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                              _P, _P]),
    "eagle_draft_layer": (_I, [_P, _P, _P, _P, _P, _P, _P, _F, _F, _P, _P, _P, _I, _P, _I, _P, _P, _P, _P,
                               _P, _I, _I, _P, _I, _I, _I, _I, _I, _I, _I, _I, _P, _Z, _P, _P]),
    "eagle_draft_input": (_I, [_P, _P, _P, _I, _P, _P, _P, _I, _I, _I, _P, _Z, _P, _P]),
    "eagle_tree_attn_workspace_size": (_Z, [_I, _I, _I, _I, _I, _I, _I, _I, _I]),
    "eagle_tree_attn": (_I, [_P, _P, _P, _P, _P, _I, _P, _I, _P, _P, _P, _P, _I, _I, _I, _I, _I,
                             _I, _F, _I, _I, _P, _Z, _P, _P]),
    "eagle_lmhead_topk_workspace_size": (_Z, [_I, _I, _I, _I, _I]),
    "eagle_lmhead_topk": (_I, [_P, _P, _P, _I, _I, _I, _I, _F, _P, _P, _P, _P, _I, _P, _Z, _P, _P]),
    "eagle_lmhead_topk_partial": (_I, [_P, _P, _P, _I, _I, _I, _I, _F, _I, _P, _Z, _P, _P]),
    "eagle_lmhead_topk_merge": (_I, [_I, _I, _I, _I, _F, _P, _P, _P, _P, _I, _P, _Z, _P, _P]),
    "eagle_tree_expand": (_I, [_I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "eagle_tree_expand_lmhead": (_I, [_I, _I, _I, _I, _I, _P, _Z, _I, _I, _F, _I, _P, _P, _P, _P, _P, _P, _P,
                                      _P, _P, _P]),
    "eagle_tree_expand_static": (_I, [_I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                      _P]),
    "eagle_tree_expand_finalize": (_I, [_I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                        _P, _P, _P, _P, _P]),
    "eagle_tree_verify_workspace_size": (_Z, [_I, _I, _I]),
    "eagle_tree_verify": (_I, [_I, _I, _I, _P, _P, _P, _P, _P, _P, _F, _I, _U64, _U64, _P, _I, _P,
                               _P, _P, _P, _Z, _P, _P]),
    "eagle_tree_verify_noalloc": (_I, [_I, _I, _I, _P, _P, _P, _P, _P, _P, _F, _I, _U64, _U64, _P,
                                       _I, _P, _P, _P, _P, _P]),
    "eagle_lmhead_verify_stats": (_I, [_P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _F, _U64, _U64, _I,
                                       _P, _P, _P, _P, _P, _I, _P, _Z, _P, _P]),
    "eagle_tree_commit": (_I, [_I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _I, _P, _I, _P, _P,
                               _I, _P, _P, _P]),
    "eagle_tree_verify_stats": (_I, [_I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _I, _F, _U64, _U64,
                                     _P, _I, _P, _P, _P, _P, _P]),
}

_lib = None


class EagleError(RuntimeError):
    def __init__(self, fn, code):
        super().__init__(f"{fn} returned {STATUS.get(code, code)}")
        self.code = code


def lib():
    """Load the library (once).  Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"CUDA library not built: {LIB_PATH} is missing "
                               "(run python -c 'import __graft_entry__ as g; g.build()')")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _dtype(t):
    if t.dtype == torch.bfloat16:
        return EAGLE_BF16
    if t.dtype == torch.float32:
        return EAGLE_FP32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _check(fn, code):
    if code != 0:
        raise EagleError(fn, code)


def workspace(nbytes, device=None):
    """A caller-owned device buffer of at least ``nbytes`` (torch allocation)."""
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8,
                       device=device if device is not None else "cuda")


def launch_count():
    return int(lib().eagle_launch_count())


def eagle_selftest_wait_timeout(limit_us, status, stream=None):
    """Bounded-wait self-test: expects status[0] = EAGLE_ERR_TIMEOUT and
    status[1] = 1 once the stream has run it."""
    _check("eagle_selftest_wait_timeout",
           lib().eagle_selftest_wait_timeout(int(limit_us), _ptr(status), _stream(stream)))


def read_status(status, stream=None):
    host = ctypes.c_int32(0)
    lib().eagle_read_status(_ptr(status), _stream(stream), ctypes.byref(host))
    return int(host.value)


# ------------------------------------------------------------------ a1
def eagle_fuse_proj_workspace_size(M, d, dtype):
    return int(lib().eagle_fuse_proj_workspace_size(M, d, dtype))


def eagle_fuse_proj(h_low, h_mid, h_high, w_proj, g, bias=None, ws=None, status=None, stream=None):
    M, d = h_low.shape
    dt = _dtype(h_low)
    if ws is None:
        ws = workspace(eagle_fuse_proj_workspace_size(M, d, dt), h_low.device)
    _check("eagle_fuse_proj", lib().eagle_fuse_proj(
        _ptr(h_low), _ptr(h_mid), _ptr(h_high), _ptr(w_proj), _ptr(bias), _ptr(g), M, d, dt,
        _ptr(ws), ws.numel(), _ptr(status), _stream(stream)))
    return g


def eagle_fuse_proj_accepted_workspace_size(B, max_depth, d, dtype):
    return int(lib().eagle_fuse_proj_accepted_workspace_size(B, max_depth, d, dtype))


def eagle_fuse_proj_accepted(h_low, h_mid, h_high, w_proj, path_rows, accept_len, g, bias=None, ws=None,
                             status=None, stream=None):
    """g[b, j] = W_proj [h_low; h_mid; h_high] of row path_rows[b, j] (rows
    b*R + row of the [B*R, d] features) for j <= accept_len[b], zero past it;
    g is [B, max_depth+1, d]."""
    B, slots = path_rows.shape
    d = h_low.shape[1]
    R = h_low.shape[0] // B
    dt = _dtype(h_low)
    if ws is None:
        ws = workspace(eagle_fuse_proj_accepted_workspace_size(B, slots - 1, d, dt), h_low.device)
    _check("eagle_fuse_proj_accepted", lib().eagle_fuse_proj_accepted(
        _ptr(h_low), _ptr(h_mid), _ptr(h_high), _ptr(w_proj), _ptr(bias), _ptr(path_rows), _ptr(accept_len),
        B, R, slots - 1, d, dt, _ptr(g), _ptr(ws), ws.numel(), _ptr(status), _stream(stream)))
    return g


def eagle_draft_input_workspace_size(M, d, dtype):
    return int(lib().eagle_draft_input_workspace_size(M, d, dtype))


def eagle_draft_input(r, token_ids, embed, w_in, u, bias=None, ws=None, status=None, stream=None):
    """u = W_I [r; embed[token_ids]] (+ bias); token_ids int32 [M] on the device."""
    M, d = r.shape
    dt = _dtype(r)
    if ws is None:
        ws = workspace(eagle_draft_input_workspace_size(M, d, dt), r.device)
    _check("eagle_draft_input", lib().eagle_draft_input(
        _ptr(r), _ptr(token_ids), _ptr(embed), embed.shape[0], _ptr(w_in), _ptr(bias), _ptr(u), M, d,
        dt, _ptr(ws), ws.numel(), _ptr(status), _stream(stream)))
    return u


def eagle_linear_workspace_size(M, n_out, k_in, dtype):
    return int(lib().eagle_linear_workspace_size(M, n_out, k_in, dtype))


def eagle_linear(x, w, y, bias=None, residual=None, ws=None, status=None, stream=None):
    """y = x w^T (+ bias) (+ residual)."""
    M, k_in = x.shape
    n_out = w.shape[0]
    dt = _dtype(x)
    if ws is None:
        ws = workspace(eagle_linear_workspace_size(M, n_out, k_in, dt), x.device)
    _check("eagle_linear", lib().eagle_linear(
        _ptr(x), _ptr(w), _ptr(bias), _ptr(residual), _ptr(y), M, n_out, k_in, dt, _ptr(ws), ws.numel(),
        _ptr(status), _stream(stream)))
    return y


def eagle_draft_layer_workspace_size(B, W, d, Hq, Hkv, D, I, Rmax, max_pages, dtype):
    return int(lib().eagle_draft_layer_workspace_size(B, W, d, Hq, Hkv, D, I, Rmax, max_pages, dtype))


def eagle_draft_layer(x, weights, positions, k_cache, v_cache, block_table, ctx_lens, q_tree, k_tree,
                      v_tree, tree_mask, r0, out, eps=1e-5, theta=500000.0, ws=None, status=None,
                      stream=None):
    """The drafter's decoder layer over the B x W new nodes of one depth.
    weights: dict norm1, qkv, o, norm2, gu, down (see include/eagle.h)."""
    B, W = positions.shape
    d = x.shape[1]
    Rmax, Hq, D = q_tree.shape[1], q_tree.shape[2], q_tree.shape[3]
    Hkv = k_tree.shape[2]
    I = weights["down"].shape[1]
    dt = _dtype(x)
    if ws is None:
        ws = workspace(eagle_draft_layer_workspace_size(B, W, d, Hq, Hkv, D, I, Rmax, block_table.shape[1], dt),
                       x.device)
    _check("eagle_draft_layer", lib().eagle_draft_layer(
        _ptr(x), _ptr(weights["norm1"]), _ptr(weights["qkv"]), _ptr(weights["o"]), _ptr(weights["norm2"]),
        _ptr(weights["gu"]), _ptr(weights["down"]), eps, theta, _ptr(positions), _ptr(k_cache),
        _ptr(v_cache), k_cache.shape[0], _ptr(block_table), block_table.shape[1], _ptr(ctx_lens),
        _ptr(q_tree), _ptr(k_tree), _ptr(v_tree), _ptr(tree_mask), r0, Rmax, _ptr(out), B, W, d, Hq, Hkv, D,
        I, dt, _ptr(ws), ws.numel(), _ptr(status), _stream(stream)))
    return out


def eagle_draft_rows(step, width, ctx_lens, node_row, row_mask, prev, r_in, tokens, positions, root_token=None,
                     frontier=None, n_frontier=None, node_parent=None, node_token=None, node_depth=None,
                     status=None, stream=None):
    """Bookkeeping of one drafter pass (see include/eagle.h)."""
    B, max_nodes = node_row.shape
    Rmax = row_mask.shape[1]
    d = prev.shape[-1]
    _check("eagle_draft_rows", lib().eagle_draft_rows(
        B, step, width, Rmax, max_nodes, d, _dtype(prev), _ptr(root_token), _ptr(frontier), _ptr(n_frontier),
        _ptr(node_parent), _ptr(node_token), _ptr(node_depth), _ptr(ctx_lens), _ptr(node_row), _ptr(row_mask),
        _ptr(prev), _ptr(r_in), _ptr(tokens), _ptr(positions), _ptr(status), _stream(stream)))


# ------------------------------------------------------------------ a2
def eagle_tree_attn_workspace_size(B, R, Hq, Hkv, D, max_pages, page_size=16, num_splits=0,
                                   dtype=EAGLE_BF16):
    return int(lib().eagle_tree_attn_workspace_size(B, R, Hq, Hkv, D, max_pages, page_size,
                                                    num_splits, dtype))


def eagle_tree_attn(q, k_tree, v_tree, k_cache, v_cache, block_table, ctx_lens, tree_mask, out,
                    lse=None, scale=None, num_splits=0, ws=None, status=None, stream=None):
    B, R, Hq, D = q.shape
    Hkv = k_tree.shape[2]
    P, page = k_cache.shape[0], k_cache.shape[1]
    max_pages = block_table.shape[1]
    dt = _dtype(q)
    if scale is None:
        scale = D ** -0.5
    if ws is None:
        ws = workspace(eagle_tree_attn_workspace_size(B, R, Hq, Hkv, D, max_pages, page, num_splits,
                                                      dt), q.device)
    _check("eagle_tree_attn", lib().eagle_tree_attn(
        _ptr(q), _ptr(k_tree), _ptr(v_tree), _ptr(k_cache), _ptr(v_cache), P, _ptr(block_table),
        max_pages, _ptr(ctx_lens), _ptr(tree_mask), _ptr(out), _ptr(lse), B, R, Hq, Hkv, D, page,
        float(scale), num_splits, dt, _ptr(ws), ws.numel(), _ptr(status), _stream(stream)))
    return out


# ------------------------------------------------------------------ a3
def eagle_lmhead_topk_workspace_size(M, d, V, k, dtype):
    return int(lib().eagle_lmhead_topk_workspace_size(M, d, V, k, dtype))


def eagle_lmhead_topk(x, w_lm, k, topk_ids, topk_logprobs, temperature=1.0, bias=None,
                      row_max=None, row_sumexp=None, ws=None, status=None, stream=None):
    M, d = x.shape
    V = w_lm.shape[0]
    dt = _dtype(x)
    if ws is None:
        ws = workspace(eagle_lmhead_topk_workspace_size(M, d, V, k, dt), x.device)
    _check("eagle_lmhead_topk", lib().eagle_lmhead_topk(
        _ptr(x), _ptr(w_lm), _ptr(bias), M, d, V, k, float(temperature), _ptr(topk_ids),
        _ptr(topk_logprobs), _ptr(row_max), _ptr(row_sumexp), dt, _ptr(ws), ws.numel(),
        _ptr(status), _stream(stream)))
    return topk_ids, topk_logprobs


def eagle_lmhead_topk_partial(x, w_lm, k, ws, temperature=1.0, bias=None, status=None, stream=None):
    """First half of eagle_lmhead_topk: the GEMM, partials left in ws."""
    M, d = x.shape
    V = w_lm.shape[0]
    _check("eagle_lmhead_topk_partial", lib().eagle_lmhead_topk_partial(
        _ptr(x), _ptr(w_lm), _ptr(bias), M, d, V, k, float(temperature), _dtype(x), _ptr(ws), ws.numel(),
        _ptr(status), _stream(stream)))


def eagle_lmhead_topk_merge(M, d, V, topk_ids, topk_logprobs, ws, dtype=EAGLE_BF16, temperature=1.0,
                            row_max=None, row_sumexp=None, status=None, stream=None):
    """Second half of eagle_lmhead_topk: merge the partials a partial call left in ws."""
    k = topk_ids.shape[-1]
    _check("eagle_lmhead_topk_merge", lib().eagle_lmhead_topk_merge(
        M, d, V, k, float(temperature), _ptr(topk_ids), _ptr(topk_logprobs), _ptr(row_max), _ptr(row_sumexp),
        dtype, _ptr(ws), ws.numel(), _ptr(status), _stream(stream)))


# ------------------------------------------------------------------ a4 / a5
def eagle_tree_expand(step, width, cand_ids, cand_logprobs, root_token, node_parent, node_token,
                      node_logv, node_depth, node_count, frontier, n_frontier, status=None,
                      stream=None):
    B, max_nodes = node_parent.shape
    k = cand_ids.shape[-1]
    _check("eagle_tree_expand", lib().eagle_tree_expand(
        B, step, width, k, max_nodes, _ptr(cand_ids), _ptr(cand_logprobs), _ptr(root_token),
        _ptr(node_parent), _ptr(node_token), _ptr(node_logv), _ptr(node_depth), _ptr(node_count),
        _ptr(frontier), _ptr(n_frontier), _ptr(status), _stream(stream)))


def eagle_tree_expand_lmhead(step, width, k, lm_ws, d, V, root_token, node_parent, node_token, node_logv,
                             node_depth, node_count, frontier, n_frontier, temperature=1.0, dtype=None,
                             status=None, stream=None):
    """One expansion step whose candidate lists are merged from the partials
    that eagle_lmhead_topk_partial left in lm_ws (B * P rows, P = 1 at step 0,
    else width)."""
    B, max_nodes = node_parent.shape
    if dtype is None:
        dtype = EAGLE_BF16
    _check("eagle_tree_expand_lmhead", lib().eagle_tree_expand_lmhead(
        B, step, width, k, max_nodes, _ptr(lm_ws), lm_ws.numel(), d, V, float(temperature), dtype,
        _ptr(root_token), _ptr(node_parent), _ptr(node_token), _ptr(node_logv), _ptr(node_depth),
        _ptr(node_count), _ptr(frontier), _ptr(n_frontier), _ptr(status), _stream(stream)))


def eagle_tree_expand_static(step, width, fanout, cand_ids, cand_logprobs, root_token, node_parent, node_token,
                             node_logv, node_depth, node_count, frontier, n_frontier, status=None, stream=None):
    """One depth of a static tree: frontier node j keeps its top-fanout[j] candidates."""
    B, max_nodes = node_parent.shape
    k = cand_ids.shape[-1]
    _check("eagle_tree_expand_static", lib().eagle_tree_expand_static(
        B, step, width, k, max_nodes, _ptr(fanout), _ptr(cand_ids), _ptr(cand_logprobs), _ptr(root_token),
        _ptr(node_parent), _ptr(node_token), _ptr(node_logv), _ptr(node_depth), _ptr(node_count),
        _ptr(frontier), _ptr(n_frontier), _ptr(status), _stream(stream)))


def eagle_tree_expand_finalize(budget, node_parent, node_token, node_logv, node_depth, node_count,
                               ctx_lens, token, parent_row, depth, mask, node_id, position, n_rows,
                               status=None, stream=None):
    B, max_nodes = node_parent.shape
    R = token.shape[1]
    _check("eagle_tree_expand_finalize", lib().eagle_tree_expand_finalize(
        B, max_nodes, budget, R, _ptr(node_parent), _ptr(node_token), _ptr(node_logv),
        _ptr(node_depth), _ptr(node_count), _ptr(ctx_lens), _ptr(token), _ptr(parent_row),
        _ptr(depth), _ptr(mask), _ptr(node_id), _ptr(position), _ptr(n_rows), _ptr(status),
        _stream(stream)))


# ------------------------------------------------------------------ a6 / a7
def eagle_tree_verify_workspace_size(B, R, V):
    return int(lib().eagle_tree_verify_workspace_size(B, R, V))


def eagle_tree_verify(parent_row, token, temperature, max_depth, accept_len, path_rows, out_tokens,
                      n_rows=None, target_logits=None, target_argmax=None, draft_logits=None,
                      proposal_mode=EAGLE_PROPOSAL_DETERMINISTIC, seed=0, offset=0,
                      uniforms_override=None, V=None, ws=None, status=None, stream=None):
    B, R = parent_row.shape
    if V is None:
        V = target_logits.shape[2]
    if ws is None:
        ws = workspace(eagle_tree_verify_workspace_size(B, R, V), parent_row.device)
    _check("eagle_tree_verify", lib().eagle_tree_verify(
        B, R, V, _ptr(parent_row), _ptr(token), _ptr(n_rows), _ptr(target_logits),
        _ptr(target_argmax), _ptr(draft_logits), float(temperature), proposal_mode, int(seed),
        int(offset), _ptr(uniforms_override), max_depth, _ptr(accept_len), _ptr(path_rows),
        _ptr(out_tokens), _ptr(ws), ws.numel(), _ptr(status), _stream(stream)))


def eagle_tree_verify_noalloc(parent_row, token, temperature, max_depth, accept_len, path_rows,
                              out_tokens, n_rows=None, target_logits=None, target_argmax=None,
                              draft_logits=None, proposal_mode=EAGLE_PROPOSAL_DETERMINISTIC, seed=0,
                              offset=0, uniforms_override=None, V=None, status=None, stream=None):
    """eagle_tree_verify for callers that cannot allocate: no workspace
    argument, statistics kept in the library's fixed device buffer
    (B * R <= 65536; at T > 0 also B * ceil(V / 4096) <= 65536)."""
    B, R = parent_row.shape
    if V is None:
        V = target_logits.shape[2]
    _check("eagle_tree_verify_noalloc", lib().eagle_tree_verify_noalloc(
        B, R, V, _ptr(parent_row), _ptr(token), _ptr(n_rows), _ptr(target_logits),
        _ptr(target_argmax), _ptr(draft_logits), float(temperature), proposal_mode, int(seed), int(offset),
        _ptr(uniforms_override), max_depth, _ptr(accept_len), _ptr(path_rows), _ptr(out_tokens),
        _ptr(status), _stream(stream)))


# ------------------------------------------------------------------ K8
def eagle_lmhead_verify_stats(x, w_lm, parent_row, token, temperature, race_k, race_ids,
                              race_keys, row_max, row_sumexp, child_logit, n_rows=None, bias=None,
                              seed=0, offset=0, ws=None, status=None, stream=None):
    """Verification statistics from the LM head (rows of x: request-major
    B*R); see include/eagle.h."""
    B, R = parent_row.shape
    M, d = x.shape
    V = w_lm.shape[0]
    dt = _dtype(x)
    if ws is None:
        ws = workspace(eagle_lmhead_topk_workspace_size(M, d, V, race_k, dt), x.device)
    _check("eagle_lmhead_verify_stats", lib().eagle_lmhead_verify_stats(
        _ptr(x), _ptr(w_lm), _ptr(bias), B, R, d, V, _ptr(parent_row), _ptr(token), _ptr(n_rows),
        float(temperature), int(seed), int(offset), race_k, _ptr(race_ids), _ptr(race_keys),
        _ptr(row_max), _ptr(row_sumexp), _ptr(child_logit), dt, _ptr(ws), ws.numel(),
        _ptr(status), _stream(stream)))


def eagle_tree_verify_stats(parent_row, token, temperature, max_depth, row_max, row_sumexp,
                            child_logit, race_ids, accept_len, path_rows, out_tokens, V,
                            n_rows=None, seed=0, offset=0, uniforms_override=None, status=None,
                            stream=None):
    B, R = parent_row.shape
    race_k = race_ids.shape[-1]
    _check("eagle_tree_verify_stats", lib().eagle_tree_verify_stats(
        B, R, V, _ptr(parent_row), _ptr(token), _ptr(n_rows), _ptr(row_max), _ptr(row_sumexp),
        _ptr(child_logit), _ptr(race_ids), race_k, float(temperature), int(seed), int(offset),
        _ptr(uniforms_override), max_depth, _ptr(accept_len), _ptr(path_rows), _ptr(out_tokens),
        _ptr(status), _stream(stream)))


# ------------------------------------------------------------------ K9
def eagle_tree_commit(k_tree, v_tree, path_rows, accept_len, k_cache, v_cache, block_table,
                      ctx_lens, features=None, features_out=None, status=None, stream=None):
    """Publish the verified path into the paged cache (see include/eagle.h)."""
    B, R, Hkv, D = k_tree.shape
    max_depth = path_rows.shape[1] - 1
    F = 0 if features is None else features.shape[1]
    _check("eagle_tree_commit", lib().eagle_tree_commit(
        B, R, Hkv, D, max_depth, _dtype(k_tree), _ptr(k_tree), _ptr(v_tree), _ptr(path_rows),
        _ptr(accept_len), _ptr(k_cache), _ptr(v_cache), k_cache.shape[0], _ptr(block_table),
        block_table.shape[1], _ptr(ctx_lens), _ptr(features), F, _ptr(features_out),
        _ptr(status), _stream(stream)))
