"""Seeded random problems across every entry point, against the oracle.

68 small problems drawn from a fixed seed: dense and grouped-query heads with
lengths on both sides of the packed-tile threshold (64 / 65 tokens) and of
tile boundaries, packed variable-length batches with empty, one-token and
multi-tile sequences, split-KV forwards with random (and empty) chunks and
their merge, and e4m3 forwards; d = 64 and 128, scales up to 0.2. Each is run
through the Python binding and compared with the float64 oracle.

Lopsided shapes (hundreds of queries on a handful of keys) and sharp softmaxes
are outside the unit-variance, balanced regime the fixed 2e-2 bar of the
parity tests is stated for: there the method's own bf16 roundings add up over
many terms and a few elements land just above 2e-2. Such elements are checked
against max(2e-2 relative, 8 R + 1e-3), R being the size those roundings
reach, computed from oracle quantities only (rounding_model.py gives the
model and its calibration). lse is checked within 1e-3.

That bound is used only outside the regime the flat bar is stated for. A case
is in that regime when its inputs are unit-variance bf16, its scale is
1/sqrt(d) and no (sequence of a) problem has more than 4 queries per key
(IN_REGIME_MAX_Q_PER_K); every output of such a case must meet the flat
max-abs 2e-2 (lse 1e-3) with no rounding model. Out-of-regime cases (scale
0.05 or 0.2, or lopsided lengths, where dV is a sum of up to hundreds of dO
rows and its own bf16 rounding exceeds 2e-2) keep the model bound, and every
case prints its flat max-abs error and the number of elements above 2e-2.
"""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

TOL = 2e-2
TOL_LSE = 1e-3
IN_REGIME_MAX_Q_PER_K = 4
LENGTHS = [1, 2, 7, 8, 31, 63, 64, 65, 100, 127, 128, 129, 200, 255, 256, 257, 300]


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


def _bf16(g, shape):
    return torch.randn(shape, generator=g).to(torch.bfloat16)


from rounding_model import head_bounds, model_limit  # noqa: E402


def in_regime(scale, d, pairs):
    """Unit-variance inputs, scale 1/sqrt(d), and at most 4 queries per key in
    every (sequence of the) problem: pairs of (queries, keys), empty ones skipped."""
    if abs(scale - 1.0 / np.sqrt(d)) > 1e-12:
        return False
    return all(lq <= IN_REGIME_MAX_Q_PER_K * lk for lq, lk in pairs if lq and lk)


def check(name, g, ref, R, regime, report):
    """In regime: the flat max-abs bar. Outside: the rounding-model bound.
    Either way the flat error and the count of elements above 2e-2 are recorded."""
    g = _np(g)
    assert np.isfinite(g).all(), f"{name}: non-finite output"
    err = np.abs(g - ref)
    flat = float(err.max()) if err.size else 0.0
    report[name] = (round(flat, 5), int((err > TOL).sum()))
    if regime:
        assert flat <= TOL, (name, flat)
        return
    lim = model_limit(ref, R, TOL)
    bad = err > lim
    assert not bad.any(), (name, float(err[bad].max()), float(lim[bad].min()))


def _print_report(kind, i, regime, report):
    print(f"\nfuzz {kind} {i}: {'in' if regime else 'outside'} regime; flat max-abs and "
          f"elements > 2e-2: {report}")


def _dense_case(i):
    g = torch.Generator().manual_seed(10_000 + i)
    r = np.random.default_rng(10_000 + i)
    d = int(r.choice([64, 128]))
    Hkv = int(r.choice([1, 2, 3]))
    G = int(r.choice([1, 1, 2, 4]))
    B = int(r.integers(1, 3))
    Lq, Lk = (int(r.choice(LENGTHS)) for _ in range(2))
    if r.random() < 0.3:
        Lk = Lq  # self-attention, the packed-tile path when short
    H = Hkv * G
    q = _bf16(g, (B, H, Lq, d))
    k = _bf16(g, (B, Hkv, Lk, d))
    v = _bf16(g, (B, Hkv, Lk, d))
    do = _bf16(g, (B, H, Lq, d))
    scale = float(r.choice([1.0 / np.sqrt(d), 0.05, 0.2]))
    return q, k, v, do, scale


@pytest.mark.parametrize("i", range(32))
def test_fuzz_dense_and_grouped(eba, i):
    q, k, v, do, scale = _dense_case(i)
    o, lse = eba.fwd(*(x.cuda() for x in (q, k, v)), scale)
    dq, dk, dv = eba.bwd(*(x.cuda() for x in (q, k, v)), o, do.cuda(), lse, scale)
    torch.cuda.synchronize()
    ro, rl = oracle.gqa_forward(q, k, v, scale)
    rdq, rdk, rdv = oracle.gqa_backward(q, k, v, do, scale)
    assert np.abs(_np(lse) - rl).max() <= TOL_LSE
    # sizes per query head; a K/V head's dK, dV sizes add in quadrature over its group
    B, H, Lq, d = q.shape
    G = H // k.shape[1]
    qf, kf, vf, dof = (x.double().numpy() for x in (q, k, v, do))
    bo, bq = np.zeros(qf.shape), np.zeros(qf.shape)
    bk, bv = np.zeros(kf.shape), np.zeros(vf.shape)
    for b in range(B):
        for h in range(H):
            eO, q_, k_, v_ = head_bounds(qf[b, h], kf[b, h // G], vf[b, h // G], dof[b, h], scale)
            bo[b, h], bq[b, h] = eO, q_
            bk[b, h // G] = np.hypot(bk[b, h // G], k_)
            bv[b, h // G] = np.hypot(bv[b, h // G], v_)
    regime = in_regime(scale, d, [(Lq, k.shape[2])])
    report = {}
    try:
        check("o", o, ro, bo, regime, report)
        check("dq", dq, rdq, bq, regime, report)
        check("dk", dk, rdk, bk, regime, report)
        check("dv", dv, rdv, bv, regime, report)
    finally:
        _print_report("dense", i, regime, report)


@pytest.mark.parametrize("i", range(16))
def test_fuzz_packed_sequences(eba, i):
    g = torch.Generator().manual_seed(20_000 + i)
    r = np.random.default_rng(20_000 + i)
    d = int(r.choice([64, 128]))
    Hkv = int(r.choice([1, 2]))
    H = Hkv * int(r.choice([1, 2]))
    n = int(r.integers(1, 9))
    pool = [0, 1, 5, 64, 65, 127, 128, 129, 250]
    lq = [int(r.choice(pool)) for _ in range(n)]
    lk = [int(r.choice(pool)) for _ in range(n)]
    if sum(lq) == 0:
        lq[0] = 3
    if sum(lk) == 0:
        lk[-1] = 2
    cu_q, cu_k = [0], [0]
    for a, b in zip(lq, lk):
        cu_q.append(cu_q[-1] + a)
        cu_k.append(cu_k[-1] + b)
    q, do = _bf16(g, (cu_q[-1], H, d)), _bf16(g, (cu_q[-1], H, d))
    k, v = _bf16(g, (cu_k[-1], Hkv, d)), _bf16(g, (cu_k[-1], Hkv, d))
    scale = 1.0 / np.sqrt(d)
    o, lse = eba.fwd_varlen(*(x.cuda() for x in (q, k, v)), cu_q, cu_k, scale)
    dq, dk, dv = eba.bwd_varlen(*(x.cuda() for x in (q, k, v)), o, do.cuda(), lse, cu_q, cu_k,
                                scale)
    torch.cuda.synchronize()
    ro, rl = oracle.varlen_forward(q, k, v, cu_q, cu_k, scale)
    rdq, rdk, rdv = oracle.varlen_backward(q, k, v, do, cu_q, cu_k, scale)
    gl = _np(lse)
    empty = np.isneginf(rl)
    assert (np.isneginf(gl) == empty).all()
    if (~empty).any():
        assert np.abs(gl[~empty] - rl[~empty]).max() <= TOL_LSE
    G = H // Hkv
    qf, kf, vf, dof = (x.double().numpy() for x in (q, k, v, do))
    bo, bq = np.zeros(qf.shape), np.zeros(qf.shape)
    bk, bv = np.zeros(kf.shape), np.zeros(vf.shape)
    for si in range(len(lq)):
        a0, a1, k0, k1 = cu_q[si], cu_q[si + 1], cu_k[si], cu_k[si + 1]
        if a1 == a0 or k1 == k0:
            continue
        for h in range(H):
            eO, q_, k_, v_ = head_bounds(qf[a0:a1, h], kf[k0:k1, h // G], vf[k0:k1, h // G],
                                         dof[a0:a1, h], scale)
            bo[a0:a1, h], bq[a0:a1, h] = eO, q_
            bk[k0:k1, h // G] = np.hypot(bk[k0:k1, h // G], k_)
            bv[k0:k1, h // G] = np.hypot(bv[k0:k1, h // G], v_)
    regime = in_regime(scale, d, list(zip(lq, lk)))
    report = {}
    try:
        check("o", o, ro, bo, regime, report)
        check("dq", dq, rdq, bq, regime, report)
        check("dk", dk, rdk, bk, regime, report)
        check("dv", dv, rdv, bv, regime, report)
    finally:
        _print_report("packed", i, regime, report)


@pytest.mark.parametrize("i", range(12))
def test_fuzz_split_merge(eba, i):
    # Split-KV: random cut points (empty chunks included), every partial
    # against the oracle's partial on its key range, the merge against the
    # unsplit oracle.
    g = torch.Generator().manual_seed(30_000 + i)
    r = np.random.default_rng(30_000 + i)
    d = int(r.choice([64, 128]))
    B, H = int(r.integers(1, 3)), int(r.integers(1, 4))
    Lq = int(r.choice(LENGTHS))
    Lk = int(r.choice(LENGTHS + [500, 777, 1000]))
    C = int(r.integers(1, 9))
    bounds = [0] + sorted(int(x) for x in r.integers(0, Lk + 1, size=C - 1)) + [Lk]
    scale = float(r.choice([1.0 / np.sqrt(d), 0.05, 0.2]))
    q, k, v = _bf16(g, (B, H, Lq, d)), _bf16(g, (B, H, Lk, d)), _bf16(g, (B, H, Lk, d))
    op, lp = eba.split_fwd(*(x.cuda() for x in (q, k, v)), bounds, scale)
    o, lse = eba.merge(op, lp)
    torch.cuda.synchronize()
    qf, kf, vf = (x.double().numpy() for x in (q, k, v))
    zero = np.zeros((Lq, d))
    report = {}
    for c in range(C):
        k0, k1 = bounds[c], bounds[c + 1]
        po, pl = oracle.partial_forward(q, k, v, scale, k0, k1)
        if k0 == k1:
            assert (_np(op[c]) == 0).all() and torch.isneginf(lp[c]).all()
            continue
        assert np.abs(_np(lp[c]) - pl).max() <= TOL_LSE
        # fp32 partials: the bf16 rounding of P only (no output rounding)
        bo = np.zeros(po.shape)
        for b in range(B):
            for h in range(H):
                bo[b, h] = head_bounds(qf[b, h], kf[b, h, k0:k1], vf[b, h, k0:k1], zero, scale)[0]
        # a partial is a forward over its range: in regime by the same rule
        check(f"o_part{c}", op[c], po, bo, in_regime(scale, d, [(Lq, k1 - k0)]), report)
    ro, rl = oracle.forward(q, k, v, scale)
    assert np.abs(_np(lse) - rl).max() <= TOL_LSE
    bo = np.zeros(ro.shape)
    for b in range(B):
        for h in range(H):
            bo[b, h] = head_bounds(qf[b, h], kf[b, h], vf[b, h], zero, scale)[0]
    regime = in_regime(scale, d, [(Lq, Lk)])
    try:
        check("o_merged", o, ro, bo, regime, report)
    finally:
        _print_report("split", i, regime, report)


@pytest.mark.parametrize("i", range(8))
def test_fuzz_fp8(eba, i):
    # e4m3 forward (d = 128, Lk a multiple of 16) against the oracle on the
    # dequantised inputs, under the first-order bound of the e4m3 P rounding.
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("this torch has no float8_e4m3fn")
    from test_gpu_fp8 import check_rows, dequant, quantize

    g = torch.Generator().manual_seed(40_000 + i)
    r = np.random.default_rng(40_000 + i)
    B, H, d = int(r.integers(1, 3)), int(r.integers(1, 3)), 128
    Lq = int(r.choice(LENGTHS))
    Lk = int(r.choice([16, 32, 48, 112, 128, 144, 256, 272, 400]))
    scale = float(r.choice([1.0 / np.sqrt(d), 0.05]))
    q, k, v = _bf16(g, (B, H, Lq, d)), _bf16(g, (B, H, Lk, d)), _bf16(g, (B, H, Lk, d))
    (q8, sq), (k8, sk), (v8, sv) = quantize(q), quantize(k), quantize(v)
    vt8 = v8.transpose(-1, -2).contiguous()
    o, lse = eba.fwd_fp8(q8.cuda(), k8.cuda(), vt8.cuda(), sq, sk, sv, scale)
    torch.cuda.synchronize()
    og, lg = o.float().cpu().numpy(), lse.cpu().numpy()
    qd, kd, vd = dequant(q8, sq).numpy(), dequant(k8, sk).numpy(), dequant(v8, sv).numpy()
    for b in range(B):
        for h in range(H):
            check_rows(og[b, h], lg[b, h], qd[b, h], kd[b, h], vd[b, h], scale)
