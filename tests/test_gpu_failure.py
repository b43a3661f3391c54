"""Failure detection on the GPU without a fault: a bounded wait on an
mbarrier that nothing completes gives up with EAGLE_ERR_TIMEOUT, the other
waiter of the CTA leaves through the abort flag, and the context stays
usable for ordinary calls afterwards."""
import time

import numpy as np
import pytest
import torch

import oracle
from eagle_speculative_decoding_gb300 import synth
from gpu_helpers import need_gpu

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_survives():
    b = need_gpu()
    st = torch.zeros(2, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    b.eagle_selftest_wait_timeout(2000, st)  # 2 ms limit
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert st.tolist() == [8, 1]  # EAGLE_ERR_TIMEOUT; second waiter left via the abort flag
    assert elapsed < 1.0          # neither wait ran to the 2 s default
    # the device still runs ordinary work: a greedy verify matches the oracle
    gen = synth.generator(3)
    parent, _ = synth.random_tree(17, 4, gen)
    tok = synth.distinct_sibling_tokens(parent, 50, gen)
    am = torch.randint(0, 50, (1, 17), generator=gen, dtype=torch.int32)
    acc = torch.zeros(1, dtype=torch.int32, device="cuda")
    path = torch.zeros((1, 5), dtype=torch.int32, device="cuda")
    out = torch.zeros((1, 5), dtype=torch.int32, device="cuda")
    b.eagle_tree_verify(parent[None].cuda(), tok[None].cuda(), 0.0, 4, acc, path, out,
                        target_argmax=am.cuda(), V=50)
    ref = oracle.tree_verify(parent[None].numpy(), tok[None].numpy(), 0.0, 4,
                             target_argmax=am.numpy())
    assert np.array_equal(out.cpu().numpy(), ref["out_tokens"])


def test_selftest_host_validation():
    b = need_gpu()
    st = torch.zeros(2, dtype=torch.int32, device="cuda")
    for bad in (0, 1000001):
        with pytest.raises(b.EagleError):
            b.eagle_selftest_wait_timeout(bad, st)
