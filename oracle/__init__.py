"""CPU oracle for the EAGLE-family speculative-decoding hot path.

TEST INFRASTRUCTURE ONLY.  This package is a plain, slow, obviously-correct
restatement of what the hot path computes, written in fp64 numpy (fp32 only
where a decision must be taken in the kernel's precision, as stated per
function).  It shares no code with the CUDA library in
``eagle_speculative_decoding_gb300/csrc``; neither side imports the other.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import it.  The product path
never routes through it.

Sources (web pages, cited by title and section):
  * "EAGLE-3: Scaling up Inference Acceleration of Large Language Models via
    Training-Time Test" (paper summary page)                      -> [E3]
  * "EAGLE: Speculative Sampling Requires Rethinking Feature Uncertainty"
    (paper summary page)                                          -> [E1]
  * "M7.5 - EAGLE Feature Drafting: Uncertainty, Dynamic Trees, HASS, and
    EAGLE-3" (transformer-system article)                         -> [M7.5]
  * "EAGLE-3: Why the Best Draft Models Stopped Predicting Features" (blog)
                                                                  -> [E3-blog]
  * Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3"
    (SC'11) for Philox4x32-10                                     -> [Philox]

Pins: every function here is checked by ``tests/test_oracle_*.py`` against
values the pages print, closed forms, invariants, or brute force.  Functions
with no such pin say "parity unpinned" in their docstring (none at present).
"""

from .eagle_oracle import (  # noqa: F401
    LOG_EPS32,
    ancestor_mask,
    draft_input,
    draft_layer,
    draft_rows,
    eagle2_tree,
    fuse_proj,
    fuse_proj_accepted,
    linear,
    lmhead_topk,
    rms_norm,
    rope,
    silu,
    static_tree_step,
    tree_attn,
    tree_expand_finalize,
    tree_expand_init,
    tree_expand_step,
    tree_verify,
    tree_commit,
    tree_verify_stats,
    verify_stats,
)
from .philox import (  # noqa: F401
    accept_uniforms, bits_to_uniform, philox4x32_10, race_uniforms, race_uniforms_batch)
