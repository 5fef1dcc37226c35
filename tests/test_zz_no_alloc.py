"""attn_bwd_noalloc: the backward for callers that cannot allocate device memory.

Some callers may not call cudaMalloc (a plugin inside a host application that
owns all GPU memory, a serving loop whose memory is fixed at start-up), so
they cannot pass attn_bwd a workspace. attn_bwd_noalloc takes its scratch from
a buffer built into the library instead. This file checks, through the C ABI,
that two calls in a row give the same gradients as attn_bwd (within the
parity tolerance; dQ is accumulated with atomics, so its low bits may differ)
and match the float64 oracle, that a B = 0 call only sets the buffer up, and
that a problem too large for the built-in buffer is refused. It is named to
run last, and passes both alone and after the other tests.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as W

pytestmark = pytest.mark.gpu

TOL = 2e-2


@pytest.fixture(scope="module")
def eba():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from exact_blockwise_attention_gb300 import _build

    _build.build()
    import exact_blockwise_attention_gb300 as m

    return m


def _call_noalloc(eba, q, k, v, o, do, lse, scale):
    B, H, Lq, d = q.shape
    Lk = k.shape[2]
    outs = [torch.full(t.shape, float("nan"), device="cuda", dtype=torch.bfloat16) for t in (q, k, v)]
    st = eba.lib().attn_bwd_noalloc(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(), lse.data_ptr(),
        outs[0].data_ptr(), outs[1].data_ptr(), outs[2].data_ptr(), B, H, Lq, Lk, d, scale,
        torch.cuda.current_stream().cuda_stream)
    assert st == 0, eba.status_string(st)
    return outs


def test_setup_call_reserves_the_buffer(eba):
    # B = 0: only loads the buffer onto this device and looks up its address
    # (what start-up code calls before memory runs short or a stream capture).
    assert eba.lib().attn_bwd_noalloc(None, None, None, None, None, None, None, None, None, 0,
                                      0, 0, 0, 0, 0.0, None) == 0


@pytest.mark.parametrize("shape,heads", [
    ((2, 8, 1568, 1568, 64), [(0, 0), (1, 7)]),
    ((1, 3, 300, 513, 128), [(0, 0), (0, 1), (0, 2)]),
], ids=["vit_heads", "ragged_d128"])
def test_two_calls_in_a_row_match_attn_bwd_and_the_oracle(eba, shape, heads):
    B, H, Lq, Lk, d = shape
    scale = 1.0 / math.sqrt(d)
    # Two different problems back to back: the second call must not see the
    # first call's leftovers in the shared buffer.
    for seed in (31, 32):
        qc, kc, vc, doc = W.make_inputs(W.VIT_L, seed=seed, B=B, H=H, Lq=Lq, Lk=Lk, d=d)
        q, k, v, do = (x.cuda() for x in (qc, kc, vc, doc))
        o, lse = eba.fwd(q, k, v, scale)
        ref = eba.bwd(q, k, v, o, do, lse, scale)
        got = _call_noalloc(eba, q, k, v, o, do, lse, scale)
        torch.cuda.synchronize()
        for name, g, r in zip(("dq", "dk", "dv"), got, ref):
            assert torch.isfinite(g.float()).all(), name
            err = (g.float() - r.float()).abs().max().item()
            assert err <= TOL, (name, seed, err)
        # and against the definition itself, on sampled heads
        for b, h in heads:
            sl = (slice(b, b + 1), slice(h, h + 1))
            rg = oracle.backward(qc[sl], kc[sl], vc[sl], doc[sl], scale)
            for name, g, r in zip(("dq", "dk", "dv"), got, rg):
                err = float(np.abs(g[sl].float().cpu().numpy() - r).max())
                assert err <= TOL, (name, seed, (b, h), err)
        assert eba.poll_device_status() == 0


def test_too_large_problem_is_refused(eba):
    x = torch.zeros(64, device="cuda", dtype=torch.bfloat16)
    p = x.data_ptr()
    # 16 x 16 heads at N = 1568, d = 64 need ~106 MB of scratch: above 64 MiB.
    st = eba.lib().attn_bwd_noalloc(p, p, p, p, p, p, p, p, p, 16, 16, 1568, 1568, 64, 0.125,
                                    None)
    assert st == 6
    assert eba.lib().attn_bwd_workspace_size(16, 16, 1568, 1568, 64) > 64 << 20
