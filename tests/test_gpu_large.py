"""Tensors of more than 2^31 elements: every offset past that point must be 64-bit.

Three problems whose inputs hold just over 2^31 elements each (4.3 GB of
bf16 per tensor): short sequences on the packed-tile path, 256-token heads on
the dense path (forward and backward), and a split-KV merge of two fp32
partials. Outputs are checked for finiteness everywhere and against the
oracle on heads (rows) before, around and past element 2^31. Peak device
memory is about 50 GB.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as W

pytestmark = pytest.mark.gpu

TOL = 2e-2
TOL_LSE = 1e-3
E31 = 2 ** 31


@pytest.fixture(scope="module")
def eba():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from exact_blockwise_attention_gb300 import _build

    _build.build()
    import exact_blockwise_attention_gb300 as m

    return m


@pytest.fixture(autouse=True)
def no_bounded_wait_gave_up(eba):
    eba.poll_device_status()
    yield
    assert eba.poll_device_status() == 0, "a bounded in-kernel wait gave up"
    torch.cuda.empty_cache()


def _np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def _check_heads(q, k, v, do, o, lse, dq, dk, dv, scale, heads):
    for b, h in heads:
        sl = (slice(b, b + 1), slice(h, h + 1))
        hq, hk, hv, hdo = (x[sl].cpu() for x in (q, k, v, do))
        ro, rl = oracle.forward(hq, hk, hv, scale)
        rdq, rdk, rdv = oracle.backward(hq, hk, hv, hdo, scale)
        assert np.abs(_np(o[sl]) - ro).max() <= TOL, (b, h)
        assert np.abs(_np(lse[sl]) - rl).max() <= TOL_LSE, (b, h)
        for g, r in ((dq, rdq), (dk, rdk), (dv, rdv)):
            assert np.abs(_np(g[sl]) - r).max() <= TOL, (b, h)


@pytest.mark.parametrize("B,H,L", [
    (1025, 1024, 32),   # packed tiles: 4 sequences of 32 tokens per tile
    (2049, 64, 256),    # dense: two query tiles per head
])
def test_past_2_31_elements(eba, B, H, L):
    d = 64
    w = W.Workload("large", B=B, H=H, Lq=L, Lk=L, d=d, seed=31)
    assert B * H * L * d > E31
    q, k, v, do = W.make_inputs_device(w, torch.device("cuda"))
    o, lse = eba.fwd(q, k, v, w.scale)
    dq, dk, dv = eba.bwd(q, k, v, o, do, lse, w.scale)
    torch.cuda.synchronize()
    for t in (o, lse, dq, dk, dv):
        assert torch.isfinite(t).all()
    # the head holding element 2^31, its neighbours, the first and the last
    h31 = E31 // (L * d)
    heads = [(0, 0), ((h31 - 1) // H, (h31 - 1) % H), (h31 // H, h31 % H), (B - 1, H - 1)]
    _check_heads(q, k, v, do, o, lse, dq, dk, dv, w.scale, heads)


def test_merge_past_2_31_elements(eba):
    C, rows, d = 2, E31 // 64 + 384, 64
    g = torch.Generator(device="cuda").manual_seed(31)
    o_parts = torch.randn((C, 1, 1, rows, d), generator=g, device="cuda")
    lse_parts = torch.randn((C, 1, 1, rows), generator=g, device="cuda") * 3
    o, lse = eba.merge(o_parts, lse_parts)
    torch.cuda.synchronize()
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
    for r0 in (0, E31 // 64 - 100, rows - 200):
        sl = (slice(None), slice(None), slice(None), slice(r0, r0 + 200))
        ro, rl = oracle.merge(_np(o_parts[sl]), _np(lse_parts[sl]))
        assert np.abs(_np(o[sl[1:]]) - ro).max() <= TOL
        assert np.abs(_np(lse[sl[1:]]) - rl).max() <= TOL_LSE
