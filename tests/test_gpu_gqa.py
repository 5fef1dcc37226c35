"""Grouped-query attention on the GPU against the float64 oracle.

q, o, dO [B, H, L, d]; k, v [B, H_kv, L, d]; query head h reads K/V head
h // (H // H_kv). Tolerances as in the dense parity tests (2e-2 on O, dQ, dK,
dV; 1e-3 on lse), each element's error divided by max(1, |oracle value|):
dK and dV of a K/V head sum over its group of query heads, so they grow with
the group size. That relative form is used only for problems with more than
4 queries per key; balanced problems with scale 1/sqrt(d) must meet the flat
max-abs 2e-2, and every check prints the flat max-abs error.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W

pytestmark = pytest.mark.gpu

TOL = 2e-2
TOL_LSE = 1e-3


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


def _np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def _rel(g, r):
    g = _np(g) if isinstance(g, torch.Tensor) else g
    assert np.isfinite(g).all(), "GPU output has non-finite (unwritten?) elements"
    return float((np.abs(g - r) / np.maximum(1.0, np.abs(r))).max()) if g.size else 0.0


def _flat(g, r):
    g = _np(g) if isinstance(g, torch.Tensor) else g
    return float(np.abs(g - r).max()) if g.size else 0.0


def _assert_errs(flat, rel, regime, what):
    """Flat bar in the balanced regime (at most 4 queries per key), the
    relative form outside it."""
    print(f"\n{what}: {'balanced' if regime else 'lopsided'}; flat max-abs {flat}")
    for n in flat:
        assert (flat[n] if regime else rel[n]) <= TOL, (what, n, flat, rel)


def _inputs(B, H, Hkv, Lq, Lk, d, seed):
    q, _, _, do = W.make_inputs(W.TINY, seed=seed, B=B, H=H, Lq=Lq, Lk=Lk, d=d)
    _, k, v, _ = W.make_inputs(W.TINY, seed=seed + 1, B=B, H=Hkv, Lq=Lq, Lk=Lk, d=d)
    return q, k, v, do


def _gpu(eba, q, k, v, do, scale):
    qd, kd, vd, dod = (x.cuda() for x in (q, k, v, do))
    o, lse = eba.fwd(qd, kd, vd, scale)
    dq, dk, dv = eba.bwd(qd, kd, vd, o, dod, lse, scale)
    torch.cuda.synchronize()
    return o, lse, dq, dk, dv


GQA_CASES = [
    # B, H, H_kv, Lq, Lk, d
    (1, 4, 1, 200, 300, 64),      # every query head on one K/V head
    (2, 6, 2, 129, 257, 64),
    (1, 8, 4, 384, 100, 64),
    (2, 4, 2, 1, 1, 64),
    (1, 4, 2, 300, 513, 128),
    (2, 2, 1, 100, 129, 128),
]


@pytest.mark.parametrize("B,H,Hkv,Lq,Lk,d", GQA_CASES, ids=lambda x: str(x))
def test_gqa_matches_oracle(eba, B, H, Hkv, Lq, Lk, d):
    q, k, v, do = _inputs(B, H, Hkv, Lq, Lk, d, seed=5000 + H * 10 + Hkv + Lq + d)
    scale = 1.0 / np.sqrt(d)
    o, lse, dq, dk, dv = _gpu(eba, q, k, v, do, scale)
    ro, rl = oracle.gqa_forward(q, k, v, scale)
    rdq, rdk, rdv = oracle.gqa_backward(q, k, v, do, scale)
    assert np.abs(_np(lse) - rl).max() <= TOL_LSE
    errs = {"o": _rel(o, ro), "dq": _rel(dq, rdq), "dk": _rel(dk, rdk), "dv": _rel(dv, rdv)}
    flat = {"o": _flat(o, ro), "dq": _flat(dq, rdq), "dk": _flat(dk, rdk), "dv": _flat(dv, rdv)}
    _assert_errs(flat, errs, Lq <= 4 * Lk, f"gqa B{B} H{H}/{Hkv} Lq{Lq} Lk{Lk} d{d}")


def test_gqa_forward_equals_repeated_heads(eba):
    # The forward of query head h is the multi-head forward with K/V head
    # h // G repeated: bit-identical. dK, dV are the group sums of the
    # multi-head gradients (fp32 accumulation in one place against bf16 sums).
    B, H, Hkv, L, d = 2, 8, 2, 700, 64
    q, k, v, do = _inputs(B, H, Hkv, L, L, d, seed=77)
    G = H // Hkv
    o, lse, dq, dk, dv = _gpu(eba, q, k, v, do, 0.125)
    kr, vr = (x.repeat_interleave(G, dim=1).contiguous() for x in (k, v))
    o2, lse2, dq2, dk2, dv2 = _gpu(eba, q, kr, vr, do, 0.125)
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    assert (dq.float() - dq2.float()).abs().max().item() <= TOL
    for g, g2 in ((dk, dk2), (dv, dv2)):
        summed = g2.float().view(B, Hkv, G, L, d).sum(2)
        assert _rel(g, _np(summed)) <= TOL


def test_gqa_with_one_group_per_head_is_mha(eba):
    B, H, L, d = 1, 4, 500, 64
    q, k, v, do = _inputs(B, H, H, L, L, d, seed=91)
    qd, kd, vd, dod = (x.cuda() for x in (q, k, v, do))
    L_ = eba.lib()
    st = torch.cuda.current_stream().cuda_stream
    o = torch.empty_like(qd)
    lse = torch.empty((B, H, L), device="cuda")
    assert L_.attn_fwd_gqa(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(),
                           lse.data_ptr(), B, H, H, L, L, d, 0.125, st) == 0
    o2, lse2 = eba.fwd(qd, kd, vd, 0.125)
    torch.cuda.synchronize()
    assert torch.equal(o, o2) and torch.equal(lse, lse2)


def test_gqa_full_size_sampled(eba):
    # ViT-L token count and head size with 4 K/V heads for 16 query heads.
    B, H, Hkv, N, d = 8, 16, 4, 1568, 64
    g = torch.Generator(device="cuda").manual_seed(123)
    q = torch.randn((B, H, N, d), generator=g, device="cuda").to(torch.bfloat16)
    k = torch.randn((B, Hkv, N, d), generator=g, device="cuda").to(torch.bfloat16)
    v = torch.randn((B, Hkv, N, d), generator=g, device="cuda").to(torch.bfloat16)
    do = torch.randn((B, H, N, d), generator=g, device="cuda").to(torch.bfloat16)
    o, lse = eba.fwd(q, k, v, 0.125)
    dq, dk, dv = eba.bwd(q, k, v, o, do, lse, 0.125)
    torch.cuda.synchronize()
    G = H // Hkv
    for b, j in ((0, 0), (B - 1, Hkv - 1), (3, 2)):
        hs = slice(j * G, (j + 1) * G)
        sq = (slice(b, b + 1), hs)
        sk = (slice(b, b + 1), slice(j, j + 1))
        args = [x[s].cpu() for x, s in ((q, sq), (k, sk), (v, sk), (do, sq))]
        ro, rl = oracle.gqa_forward(*args[:3], 0.125)
        rdq, rdk, rdv = oracle.gqa_backward(*args, 0.125)
        assert np.abs(_np(lse[sq]) - rl).max() <= TOL_LSE
        flat = {"o": _flat(o[sq], ro), "dq": _flat(dq[sq], rdq), "dk": _flat(dk[sk], rdk),
                "dv": _flat(dv[sk], rdv)}
        _assert_errs(flat, flat, True, f"gqa ViT-L shape b{b} kv-head {j}")


def test_gqa_autograd(eba):
    q, k, v, do = _inputs(1, 4, 2, 150, 260, 64, seed=31)
    qd, kd, vd = (x.cuda().requires_grad_() for x in (q, k, v))
    out = eba.attention(qd, kd, vd)
    out.backward(do.cuda())
    rdq, rdk, rdv = oracle.gqa_backward(q, k, v, do, 0.125)
    assert _rel(qd.grad, rdq) <= TOL and _rel(kd.grad, rdk) <= TOL and _rel(vd.grad, rdv) <= TOL
