"""The C-ABI library builds, loads without a GPU, exports every call that
include/eagle.h declares, and validates arguments on the host (no GPU needed:
every case below returns before any CUDA call)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "eagle.h")


@pytest.fixture(scope="module")
def L():
    from eagle_speculative_decoding_gb300 import binding, build
    if not os.path.exists(binding.LIB_PATH):
        build.build()
    return binding.lib()


def declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(eagle_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_hot_path_calls():
    names = declared()
    for n in ("eagle_fuse_proj", "eagle_tree_attn", "eagle_lmhead_topk", "eagle_tree_expand",
              "eagle_tree_expand_finalize", "eagle_tree_verify", "eagle_draft_input"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    for n in declared():
        assert hasattr(L, n), n


def test_status_strings(L):
    assert L.eagle_status_string(0) == b"EAGLE_OK"
    assert L.eagle_status_string(8) == b"EAGLE_ERR_TIMEOUT"
    assert L.eagle_status_string(99) == b"EAGLE_ERR_UNKNOWN"


def test_host_validation_without_gpu(L):
    N = None
    # verify: null pointers, sampled proposals at T = 0 or without draft logits, deep trees, no ws
    assert L.eagle_tree_verify(1, 4, 8, N, N, N, N, N, N, 1.0, 0, 0, 0, N, 2, N, N, N, N, 0, N, N) == 1
    p = ctypes.c_void_p(16)
    assert L.eagle_tree_verify(1, 4, 8, p, p, N, p, N, p, 0.0, 1, 0, 0, N, 2, p, p, p, N, 0, N, N) == 1
    assert L.eagle_tree_verify(1, 4, 8, p, p, N, p, N, N, 1.0, 1, 0, 0, N, 2, p, p, p, N, 0, N, N) == 1
    assert L.eagle_tree_verify(1, 4, 8, p, p, N, p, N, p, 1.0, 1, 0, 0, N, 2, p, p, p, N, 0, N, N) == 3
    assert L.eagle_tree_verify(1, 4, 8, p, p, N, p, N, N, 1.0, 0, 0, 0, N, 65, p, p, p, N, 0, N, N) == 2
    assert L.eagle_tree_verify(1, 4, 8, p, p, N, p, N, N, 1.0, 0, 0, 0, N, 2, p, p, p, N, 0, N, N) == 3
    # lm head: k > 32 unsupported, k > V invalid, V not a multiple of 16
    assert L.eagle_lmhead_topk(p, p, N, 4, 64, 256, 33, 1.0, p, p, N, N, 1, N, 0, N, N) == 2
    assert L.eagle_lmhead_topk(p, p, N, 4, 64, 128, 200, 1.0, p, p, N, N, 1, N, 0, N, N) == 1
    assert L.eagle_lmhead_topk(p, p, N, 4, 64, 100, 1, 1.0, p, p, N, N, 1, N, 0, N, N) == 2
    assert L.eagle_lmhead_topk(p, p, N, 4, 64, 256, 1, 0.0, p, p, N, N, 1, N, 0, N, N) == 1
    assert L.eagle_lmhead_topk(p, p, N, 4, 64, 256, 1, 1.0, p, p, N, N, 1, N, 0, N, N) == 3
    # split LM head: partial without x, merge without outputs, merge without ws
    assert L.eagle_lmhead_topk_partial(N, p, N, 4, 64, 256, 1, ctypes.c_float(1.0), 1, p, 1 << 30, N, N) == 1
    assert L.eagle_lmhead_topk_merge(4, 64, 256, 1, ctypes.c_float(1.0), N, p, N, N, 1, p, 1 << 30, N, N) == 1
    assert L.eagle_lmhead_topk_merge(4, 64, 256, 1, ctypes.c_float(1.0), p, p, N, N, 1, N, 0, N, N) == 3
    # bounded-wait self-test: the limit must be 1 .. 10^6 microseconds
    assert L.eagle_selftest_wait_timeout(0, p, N) == 1
    assert L.eagle_selftest_wait_timeout(1000001, p, N) == 1
    assert L.eagle_selftest_wait_timeout(10, N, N) == 1
    # fuse_proj: d not a multiple of 128
    assert L.eagle_fuse_proj(p, p, p, p, N, p, 4, 100, 1, N, 0, N, N) == 2
    assert L.eagle_fuse_proj(p, p, p, p, N, p, 4, 128, 1, N, 0, N, N) == 3
    # draft_input: null token ids, vocab 0, d not a multiple of 128, M too large, no ws
    assert L.eagle_draft_input(p, N, p, 10, p, N, p, 4, 128, 1, N, 0, N, N) == 1
    assert L.eagle_draft_input(p, p, p, 0, p, N, p, 4, 128, 1, N, 0, N, N) == 1
    assert L.eagle_draft_input(p, p, p, 10, p, N, p, 4, 100, 1, N, 0, N, N) == 2
    assert L.eagle_draft_input(p, p, p, 10, p, N, p, 4097, 128, 1, N, 0, N, N) == 2
    assert L.eagle_draft_input(p, p, p, 10, p, N, p, 4, 128, 1, N, 0, N, N) == 3
    assert L.eagle_draft_input_workspace_size(4, 128, 1) > 0
    # linear: x aliasing y, n_out not a multiple of 128, k_in not a multiple of 64, no ws
    assert L.eagle_linear(p, p, N, N, p, 4, 128, 64, 1, N, 0, N, N) == 1
    q = ctypes.c_void_p(32)
    assert L.eagle_linear(p, p, N, N, q, 4, 100, 64, 1, N, 0, N, N) == 2
    assert L.eagle_linear(p, p, N, N, q, 4, 128, 48, 1, N, 0, N, N) == 2
    assert L.eagle_linear(p, p, N, N, q, 4, 128, 64, 1, N, 0, N, N) == 3
    # draft layer: null pointer, rows past Rmax, D = 96, no ws
    lay = lambda r0, Rmax, D, ws_b: L.eagle_draft_layer(
        p, p, p, p, p, p, p, ctypes.c_float(1e-5), ctypes.c_float(5e5), p, p, p, 4, p, 2, p, p, p, p, p,
        r0, Rmax, q, 1, 4, 256, 4, 2, D, 256, 1, N, ws_b, N, N)
    assert lay(6, 8, 64, 0) == 2
    assert lay(0, 8, 96, 0) == 2
    assert lay(0, 8, 64, 0) == 3
    assert L.eagle_draft_layer(N, p, p, p, p, p, p, ctypes.c_float(1e-5), ctypes.c_float(5e5), p, p, p, 4, p, 2,
                               p, p, p, p, p, 0, 8, q, 1, 4, 256, 4, 2, 64, 256, 1, N, 0, N, N) == 1
    assert L.eagle_draft_layer_workspace_size(1, 4, 256, 4, 2, 64, 256, 8, 2, 1) > 0
    # draft rows: step 0 without root tokens, width over 64, rows past Rmax
    rows = lambda step, width, Rmax, root: L.eagle_draft_rows(1, step, width, Rmax, 64, 256, 1, root, p, p, p, p,
                                                              p, p, p, p, p, q, p, p, N, N)
    assert rows(0, 4, 8, N) == 1
    assert rows(1, 65, 64, p) == 2
    assert rows(2, 4, 8, p) == 1
    # attention: R > 64, D not in {64, 128}, page size != 16, Hq % Hkv
    base = [p, p, p, p, p, 4, p, 2, p, p, p, N]
    assert L.eagle_tree_attn(*base, 1, 65, 4, 2, 128, 16, ctypes.c_float(0.1), 0, 1, N, 0, N, N) == 2
    assert L.eagle_tree_attn(*base, 1, 8, 4, 2, 96, 16, ctypes.c_float(0.1), 0, 1, N, 0, N, N) == 2
    assert L.eagle_tree_attn(*base, 1, 8, 4, 2, 128, 32, ctypes.c_float(0.1), 0, 1, N, 0, N, N) == 2
    assert L.eagle_tree_attn(*base, 1, 8, 5, 2, 128, 16, ctypes.c_float(0.1), 0, 1, N, 0, N, N) == 1
    # expand: width 0, k > 32, max_nodes too small for the step
    assert L.eagle_tree_expand(1, 0, 0, 2, 16, p, p, p, p, p, p, p, p, p, p, N, N) == 1
    # static expansion: no fan-out array, width over 64
    assert L.eagle_tree_expand_static(1, 0, 4, 2, 64, N, p, p, p, p, p, p, p, p, p, p, N, N) == 1
    assert L.eagle_tree_expand_static(1, 0, 65, 2, 512, p, p, p, p, p, p, p, p, p, p, p, N, N) == 2
    assert L.eagle_tree_expand(1, 0, 2, 33, 64, p, p, p, p, p, p, p, p, p, p, N, N) == 2
    assert L.eagle_tree_expand(1, 3, 2, 2, 12, p, p, p, p, p, p, p, p, p, p, N, N) == 1
    assert L.eagle_tree_expand_finalize(1, 16, 8, 4, p, p, p, p, p, N, p, p, p, p, p, p, p, N, N) == 1
    assert L.eagle_tree_expand_finalize(1, 16, 8, 65, p, p, p, p, p, N, p, p, p, p, p, p, p, N, N) == 2


def test_workspace_queries(L):
    assert L.eagle_lmhead_topk_workspace_size(61, 4096, 128256, 1, 1) > 0
    assert L.eagle_fuse_proj_workspace_size(61, 4096, 1) > 0
    assert L.eagle_tree_verify_workspace_size(4, 61, 128256) >= 4 * 61 * 12


def _declared_arity():
    """Parameter count of every call the header declares."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    out = {}
    for m in re.finditer(r"\b(eagle_[a-z0-9_]+)\s*\(([^;{]*?)\)\s*;", text, flags=re.S):
        args = m.group(2).strip()
        out[m.group(1)] = 0 if args in ("", "void") else args.count(",") + 1
    return out


def test_binding_signatures_match_the_header():
    """Every call the Python binding marshals passes exactly as many
    arguments as the header's prototype declares."""
    from eagle_speculative_decoding_gb300 import binding
    arity = _declared_arity()
    for name, (_, args) in binding._SIGS.items():
        assert name in arity, name
        assert len(args) == arity[name], (name, len(args), arity[name])
