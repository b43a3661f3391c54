"""EAGLE speculative-decoding hot path for GB300 (sm_103a).

The compute lives in the CUDA library built from ``csrc/`` (C-ABI declared in
``include/eagle.h``); ``binding`` marshals torch tensors into it and
``synth`` draws seeded synthetic inputs.  Importing the package does not load
the library; the first binding call does, and raises if it is missing.
"""
__all__ = ["binding", "synth", "build"]
