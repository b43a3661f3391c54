"""Pins of the oracle's drafter-row bookkeeping over an EAGLE-2 round: the
row masks equal the ancestry masks of the processed rows (an independent
function), positions are prefix length + depth, tokens come from the store,
and each row's feature input is its parent's output of the previous pass."""
import numpy as np
import pytest
import torch

import oracle
from eagle_speculative_decoding_gb300 import synth


def _round(depth, k, width, seed, ctx=37, d=3):
    gen = synth.generator(seed)
    st = oracle.tree_expand_init(11)
    node_row, row_mask = {}, {}
    rows_all, parent_of_row, feats_all = [], {}, {}
    prev = np.array([[1000.0] * d])  # the target feature of the root
    for s in range(depth):
        rows, toks, pos, feats = oracle.draft_rows(s, width, st if s else None, node_row, row_mask, ctx, prev,
                                                   root_token=11)
        for r, f in zip(rows, feats):
            feats_all[r] = f
        rows_all.append(rows)
        # the drafter's outputs of this pass: identify each row by its number
        prev = np.array([[float(r)] * d for r in rows])
        ids, lps = synth.draft_candidates(len(st["frontier"]), k, 500, gen)
        oracle.tree_expand_step(st, ids.numpy(), lps.numpy(), width)
        for r in rows:
            n = [m for m, rr in node_row.items() if rr == r][0]
            parent_of_row[r] = -1 if n == 0 else node_row[st["parent"][n]]
    return st, node_row, row_mask, rows_all, parent_of_row, feats_all


def test_row_masks_are_ancestry_of_processed_rows():
    st, node_row, row_mask, rows_all, parent_of_row, _ = _round(4, 3, 3, 1)
    R = 1 + max(r for rows in rows_all for r in rows)
    par = np.array([parent_of_row[r] for r in range(R)])
    ref = oracle.ancestor_mask(par)
    assert [int(row_mask[r]) for r in range(R)] == [int(x) for x in ref]


def test_rows_positions_tokens_and_contiguous_numbering():
    width, ctx = 3, 37
    st, node_row, _, rows_all, _, _ = _round(4, 3, width, 2, ctx=ctx)
    assert rows_all[0] == [0]
    for s, rows in enumerate(rows_all[1:], start=1):
        assert rows == list(range(1 + (s - 1) * width, 1 + (s - 1) * width + len(rows)))
    for n, r in node_row.items():
        assert st["depth"][n] == (0 if r == 0 else 1 + (r - 1) // width)


def test_feature_input_is_the_parents_output():
    st, node_row, _, rows_all, parent_of_row, feats = _round(4, 3, 3, 3)
    assert np.all(feats[0] == 1000.0)  # the root takes the target feature
    for r, f in feats.items():
        if r:
            assert np.all(f == float(parent_of_row[r]))


def test_unprocessed_parent_is_an_error():
    st = oracle.tree_expand_init(4)
    ids, lps = synth.draft_candidates(1, 2, 50, synth.generator(0))
    oracle.tree_expand_step(st, ids.numpy(), lps.numpy(), 2)
    with pytest.raises(ValueError):
        oracle.draft_rows(1, 2, st, {}, {}, 10, np.zeros((1, 2)))
