"""FP8 (e4m3) forward on the GPU against the float64 oracle.

The oracle runs on the dequantised inputs (stored e4m3 value x per-tensor
scale, exact in float64), so the scores are the same numbers on both sides;
what remains is the one rounding this path adds: the softmax weights are
rounded to e4m3 before the P V product. For each output element the test
checks the first-order bound of that rounding, derived from the e4m3 format
(3 mantissa bits: relative error <= 2^-4 for normal numbers; absolute error
<= 2^-10 below 2^-6) and the weights' reference maximum (the kernel's weights
are exp(S - max) * c with 1 <= c <= 2^8, so their sum is >= l = sum exp(S - max)):

  |O_gpu - O| <= 2^-4 * sum_j P_j (|v_j - O| + |O|)
               + 2^-10 * sum_j (|v_j - O| + |O|) / l + 2^-8 |O| + 1e-3

(the 2^-8 |O| is the bf16 rounding of the output, the 1e-3 the fp32
accumulation), and lse within 1e-3 as in the bf16 parity tests (lse uses
the fp32 weights).
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as W

pytestmark = pytest.mark.gpu

TOL_LSE = 1e-3
E4M3_MAX = 448.0


@pytest.fixture(scope="module")
def eba():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("this torch has no float8_e4m3fn")
    from exact_blockwise_attention_gb300 import _build

    _build.build()
    import exact_blockwise_attention_gb300 as m

    return m


@pytest.fixture(autouse=True)
def no_bounded_wait_gave_up(eba):
    eba.poll_device_status()
    yield
    assert eba.poll_device_status() == 0, "a bounded in-kernel wait gave up"


def quantize(x):
    """Per-tensor e4m3: (stored tensor, dequantisation scale)."""
    amax = float(x.float().abs().max())
    s = amax / E4M3_MAX if amax > 0 else 1.0
    return (x.float() / s).to(torch.float8_e4m3fn), s


def dequant(x8, s):
    return x8.to(torch.float64) * s


def check_rows(o_gpu, lse_gpu, q, k, v, scale):
    """q [Lq, d], k, v [Lk, d] float64 (dequantised); o_gpu, lse_gpu of the same rows."""
    S = scale * (q @ k.T)
    mx = S.max(axis=1, keepdims=True)
    E = np.exp(S - mx)
    l = E.sum(axis=1, keepdims=True)
    P = E / l
    O = P @ v
    lse = (mx + np.log(l))[:, 0]
    g = o_gpu.astype(np.float64)
    dev = np.abs(v[None, :, :] - O[:, None, :]) + np.abs(O)[:, None, :]  # [Lq, Lk, d]
    bound = (2.0 ** -4) * np.einsum("ij,ijc->ic", P, dev) + (2.0 ** -10) * dev.sum(axis=1) / l \
        + (2.0 ** -8) * np.abs(O) + 1e-3
    err = np.abs(g - O)
    assert np.isfinite(g).all()
    assert (err <= bound).all(), f"max err {err.max():.4g}, worst err / bound {(err / bound).max():.3f}"
    assert np.abs(lse_gpu.astype(np.float64) - lse).max() <= TOL_LSE
    return float(err.max()), float((err / bound).max())


def _case(eba, B, H, Lq, Lk, seed, heads=None):
    d = 128
    q, k, v, _ = W.make_inputs(W.TINY, seed=seed, B=B, H=H, Lq=Lq, Lk=Lk, d=d)
    q8, sq = quantize(q)
    k8, sk = quantize(k)
    v8, sv = quantize(v)
    vt8 = v8.transpose(-1, -2).contiguous()
    scale = 1.0 / math.sqrt(d)
    o, lse = eba.fwd_fp8(q8.cuda(), k8.cuda(), vt8.cuda(), sq, sk, sv, scale)
    torch.cuda.synchronize()
    og = o.float().cpu().numpy()
    lg = lse.cpu().numpy()
    qd, kd, vd = dequant(q8, sq).numpy(), dequant(k8, sk).numpy(), dequant(v8, sv).numpy()
    worst = 0.0
    for b, h in heads or [(b, h) for b in range(B) for h in range(H)]:
        _, r = check_rows(og[b, h], lg[b, h], qd[b, h], kd[b, h], vd[b, h], scale)
        worst = max(worst, r)
    return worst


FP8_CASES = [
    # B, H, Lq, Lk
    (1, 1, 1, 16),
    (1, 2, 200, 336),     # ragged query and key tiles
    (2, 1, 129, 256),
    (1, 3, 384, 1024),    # odd number of query tiles
]


@pytest.mark.parametrize("B,H,Lq,Lk", FP8_CASES, ids=lambda x: str(x))
def test_fp8_forward_within_the_e4m3_bound(eba, B, H, Lq, Lk):
    _case(eba, B, H, Lq, Lk, seed=9000 + Lq + Lk + H)


def test_fp8_cross_shape_sampled(eba):
    # The long-visual cross-attention shape (512 text queries, 36864 visual keys)
    # in e4m3, sampled heads.
    w = W.CROSS
    _case(eba, w.B, w.H, w.Lq, w.Lk, seed=w.seed + 50, heads=[(0, 0), (1, 31)])


def test_fp8_rejects_other_head_dims_and_ragged_vt(eba):
    x = torch.zeros((1, 1, 16, 64), device="cuda").to(torch.float8_e4m3fn)
    with pytest.raises(eba.AttnError):
        eba.fwd_fp8(x, x, x.transpose(-1, -2).contiguous(), 1.0, 1.0, 1.0)
    q = torch.zeros((1, 1, 16, 128), device="cuda").to(torch.float8_e4m3fn)
    k = torch.zeros((1, 1, 20, 128), device="cuda").to(torch.float8_e4m3fn)
    with pytest.raises(eba.AttnError):
        eba.fwd_fp8(q, k, k.transpose(-1, -2).contiguous(), 1.0, 1.0, 1.0)
