"""Plain float64 CPU oracle for exact attention. TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package. The CUDA library never calls it, and the two share
no code. Every function is pinned by the CPU tests (closed forms, invariants,
finite differences, an independent library routine); none is "parity
unpinned".
"""
from .attention import (  # noqa: F401
    backward,
    forward,
    gqa_backward,
    gqa_forward,
    merge,
    partial_forward,
    softmax_weights,
    split_forward,
    varlen_backward,
    varlen_forward,
)
