"""The CPU oracle against facts fixed outside itself (no GPU needed)."""
import types

import pytest

import oracle
import oracle_pins as pins

IMPL = types.SimpleNamespace(
    forward=oracle.forward,
    backward=oracle.backward,
    partial_forward=oracle.partial_forward,
    merge=oracle.merge,
    softmax_weights=oracle.softmax_weights,
    varlen_forward=oracle.varlen_forward,
    varlen_backward=oracle.varlen_backward,
    gqa_forward=oracle.gqa_forward,
    gqa_backward=oracle.gqa_backward,
)


@pytest.mark.parametrize("check", pins.ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(check):
    if check is pins.check_mpmath_bruteforce:
        pytest.importorskip("mpmath")
    check(IMPL)


def test_split_forward_matches_forward():
    import numpy as np

    r = np.random.default_rng(0)
    q, k, v = (r.normal(size=(1, 2, L, 4)) for L in (3, 10, 10))
    o1, l1 = oracle.split_forward(q, k, v, 0.5, [(0, 4), (4, 4), (4, 10)])
    o2, l2 = oracle.forward(q, k, v, 0.5)
    assert abs(o1 - o2).max() < 1e-12 and abs(l1 - l2).max() < 1e-12
