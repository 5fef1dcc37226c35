"""Short sequences (at most 64 queries and keys) on the GPU against the oracle.

With max(Lq, Lk) in 5..8, attn_fwd and attn_bwd run on the CUDA cores, one
warp per sequence; otherwise they pack floor(128 / max(Lq, Lk)) consecutive
(batch, head) sequences into one 128-row tile with a block-diagonal mask. This is the temporal attention of
factorised space-time video transformers, (b*h*w, t, d) with t = 8
tubelet-frames. Same tolerances as the dense parity tests (2e-2 on O, dQ, dK,
dV; 1e-3 on lse).
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


def _err(g, r):
    g = _np(g)
    assert np.isfinite(g).all(), "GPU output has non-finite (unwritten?) elements"
    return float(np.abs(g - r).max())


def _nan(shape, dtype):
    return torch.full(shape, float("nan"), device="cuda", dtype=dtype)


def _run(eba, q, k, v, do, scale):
    """attn_fwd + attn_bwd through the C ABI into NaN-prefilled outputs and workspace."""
    B, H, Lq, d = q.shape
    Lk = k.shape[2]
    L = eba.lib()
    st = torch.cuda.current_stream().cuda_stream
    o, lse = _nan(q.shape, torch.bfloat16), _nan((B, H, Lq), torch.float32)
    assert L.attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                      B, H, Lq, Lk, d, scale, st) == 0
    dq, dk, dv = (_nan(x.shape, torch.bfloat16) for x in (q, k, v))
    need = eba.bwd_workspace_size(B, H, Lq, Lk, d)
    ws = torch.full((need // 4,), float("nan"), device="cuda", dtype=torch.float32)
    assert L.attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(),
                      lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, Lq, Lk,
                      d, scale, ws.data_ptr(), need, st) == 0
    torch.cuda.synchronize()
    return o, lse, dq, dk, dv


SHORT = [
    # B, H, Lq, Lk, d         sequences per tile
    (4, 4, 8, 8, 64),         # 16: one full tile
    (3, 5, 7, 7, 64),         # 18: 15 sequences, part of one tile
    (16, 16, 8, 8, 64),       # 16: 16 tiles
    (7, 3, 13, 13, 64),       # 9: ragged packing, last tile partial
    (2, 8, 64, 64, 64),       # 2
    (5, 3, 1, 1, 64),         # 128 single-token sequences
    (4, 4, 8, 50, 64),        # 2: short queries, more keys
    (3, 3, 33, 5, 64),        # 3: more queries than keys
    (4, 4, 8, 8, 128),
    (3, 7, 20, 20, 128),
    (2, 2, 64, 17, 128),
]


@pytest.mark.parametrize("B,H,Lq,Lk,d", SHORT, ids=lambda x: str(x))
def test_short_sequences_match_oracle(eba, B, H, Lq, Lk, d):
    q, k, v, do = W.make_inputs(W.TINY, seed=7000 + B * H + Lq * 3 + Lk + d, B=B, H=H, Lq=Lq,
                                Lk=Lk, d=d)
    scale = 1.0 / math.sqrt(d)
    o, lse, dq, dk, dv = _run(eba, *(x.cuda() for x in (q, k, v, do)), scale)
    ro, rl = oracle.forward(q, k, v, scale)
    rdq, rdk, rdv = oracle.backward(q, k, v, do, scale)
    assert np.abs(_np(lse) - rl).max() <= TOL_LSE
    errs = {"o": _err(o, ro), "dq": _err(dq, rdq), "dk": _err(dk, rdk), "dv": _err(dv, rdv)}
    assert max(errs.values()) <= TOL, errs


# The CUDA-core path (max(Lq, Lk) in 5..8) at row counts in each of its two
# query-row and key-row groups, both head dimensions, and the shapes on either
# side of it (tensor-core packed tiles); sequence counts that are not
# multiples of the warps per block.
SHORT_FWD = [(lq, lk, d) for d in (64, 128)
             for lq, lk in ((1, 1), (1, 8), (8, 1), (2, 3), (4, 4), (3, 7), (5, 5), (7, 2),
                            (6, 8), (8, 8), (9, 6), (8, 9), (16, 16))]


@pytest.mark.parametrize("Lq,Lk,d", SHORT_FWD, ids=lambda x: str(x))
def test_short_sweep_matches_oracle(eba, Lq, Lk, d):
    B, H = 5, 7
    q, k, v, do = W.make_inputs(W.TINY, seed=7400 + 17 * Lq + Lk + d, B=B, H=H, Lq=Lq, Lk=Lk,
                                d=d)
    scale = 1.0 / math.sqrt(d)
    o, lse, dq, dk, dv = _run(eba, *(x.cuda() for x in (q, k, v, do)), scale)
    ro, rl = oracle.forward(q, k, v, scale)
    rdq, rdk, rdv = oracle.backward(q, k, v, do, scale)
    assert np.abs(_np(lse) - rl).max() <= TOL_LSE
    assert _err(o, ro) <= TOL
    if Lq <= 4 * Lk:
        # the flat bar's regime: unit-variance inputs, scale 1/sqrt(d), at most
        # 4 queries per key
        errs = {"dq": _err(dq, rdq), "dk": _err(dk, rdk), "dv": _err(dv, rdv)}
        assert max(errs.values()) <= TOL, errs
        return
    # More queries per key (8 to 1): dV sums up to 8 dO rows, and its own bf16
    # rounding alone exceeds 2e-2 once |dV| >= 8; held to the rounding-model
    # bound of the fuzz tests instead.
    from rounding_model import head_bounds, model_limit

    f64 = [x.double().numpy() for x in (q, k, v, do)]
    for b in range(B):
        for h in range(H):
            _, bq, bk, bv = head_bounds(*(x[b, h] for x in f64), scale)
            for g, ref, R in ((dq, rdq, bq), (dk, rdk, bk), (dv, rdv, bv)):
                err = np.abs(_np(g[b, h]) - ref[b, h])
                assert (err <= model_limit(ref[b, h], R)).all()


def test_short_many_sequences_per_warp(eba):
    # 40 000 sequences of 5 queries and 7 keys: the grid holds fewer warps, so
    # every warp computes several sequences in turn (forward and backward).
    B, H, Lq, Lk, d = 2500, 16, 5, 7, 64
    qc, kc, vc, doc = W.make_inputs(W.TINY, seed=7500, B=B, H=H, Lq=Lq, Lk=Lk, d=d)
    scale = 1.0 / math.sqrt(d)
    o, lse, dq, dk, dv = _run(eba, *(x.cuda() for x in (qc, kc, vc, doc)), scale)
    for b0 in range(0, B, 500):
        sl = slice(b0, b0 + 500)
        ro, rl = oracle.forward(qc[sl], kc[sl], vc[sl], scale)
        rdq, rdk, rdv = oracle.backward(qc[sl], kc[sl], vc[sl], doc[sl], scale)
        assert _err(o[sl], ro) <= TOL
        assert np.abs(_np(lse[sl]) - rl).max() <= TOL_LSE
        assert max(_err(dq[sl], rdq), _err(dk[sl], rdk), _err(dv[sl], rdv)) <= TOL


def test_temporal_attention_forward_every_sequence(eba):
    # The forward of the full temporal workload (16 x 196 positions x 16 heads
    # = 50 176 sequences of 8 frames) against the oracle, every sequence.
    w = W.TEMPORAL
    q, k, v, _ = W.make_inputs_device(w, "cuda")
    L = eba.lib()
    o, lse = _nan(q.shape, torch.bfloat16), _nan(q.shape[:3], torch.float32)
    assert L.attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                      w.B, w.H, w.Lq, w.Lk, w.d, w.scale,
                      torch.cuda.current_stream().cuda_stream) == 0
    torch.cuda.synchronize()
    worst_o = worst_l = 0.0
    for b0 in range(0, w.B, 392):
        sl = slice(b0, b0 + 392)
        ro, rl = oracle.forward(q[sl].cpu(), k[sl].cpu(), v[sl].cpu(), w.scale)
        worst_o = max(worst_o, _err(o[sl], ro))
        worst_l = max(worst_l, float(np.abs(_np(lse[sl]) - rl).max()))
    assert worst_o <= TOL and worst_l <= TOL_LSE, (worst_o, worst_l)


def test_temporal_attention_full_size_sampled(eba):
    # Temporal attention of the ViT-L clip: every one of the 16 x 196 spatial
    # positions attends over its 8 tubelet-frames, H = 16, d = 64.
    w = W.TEMPORAL
    q, k, v, do = W.make_inputs_device(w, "cuda")
    o, lse, dq, dk, dv = _run(eba, q, k, v, do, w.scale)
    g = np.random.default_rng(5)
    for b in sorted(set([0, w.B - 1] + [int(x) for x in g.integers(0, w.B, size=6)])):
        sl = (slice(b, b + 1), slice(None))
        args = [x[sl].cpu() for x in (q, k, v, do)]
        ro, rl = oracle.forward(*args[:3], w.scale)
        rdq, rdk, rdv = oracle.backward(*args, w.scale)
        assert _err(o[sl], ro) <= TOL and np.abs(_np(lse[sl]) - rl).max() <= TOL_LSE
        assert _err(dq[sl], rdq) <= TOL and _err(dk[sl], rdk) <= TOL and _err(dv[sl], rdv) <= TOL


def test_spatial_attention_sampled(eba):
    # Spatial attention of the same clip: each of the 16 x 8 frames attends over
    # its 14 x 14 = 196 patches (two 128-row tiles per head).
    w = W.SPATIAL
    q, k, v, do = W.make_inputs_device(w, "cuda")
    o, lse, dq, dk, dv = _run(eba, q, k, v, do, w.scale)
    for b in (0, 77, w.B - 1):
        sl = (slice(b, b + 1), slice(None))
        args = [x[sl].cpu() for x in (q, k, v, do)]
        ro, rl = oracle.forward(*args[:3], w.scale)
        rdq, rdk, rdv = oracle.backward(*args, w.scale)
        assert _err(o[sl], ro) <= TOL and np.abs(_np(lse[sl]) - rl).max() <= TOL_LSE
        assert _err(dq[sl], rdq) <= TOL and _err(dk[sl], rdk) <= TOL and _err(dv[sl], rdv) <= TOL
