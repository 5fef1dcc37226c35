"""Packed variable-length sequences on the GPU against the float64 oracle.

Token-major [T, H, d] tensors with cumulative lengths cu_q, cu_k; every
sequence attends only within itself. Tolerances as in the dense parity tests,
2e-2 on O, dQ, dK, dV and 1e-3 (absolute) on lse, with each element's error
divided by max(1, |oracle value|): a short sequence gives outputs far from unit
scale (one key: dV = the sum of dO over all the sequence's queries, |dV| ~ 40),
where the bf16 rounding of the result alone is above 2e-2 absolute. That
relative form is used only for problems outside the balanced regime (some
sequence with more than 4 queries per key); balanced problems with scale
1/sqrt(d) must meet the flat max-abs 2e-2, and every check prints the flat
max-abs error.
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


def _cu(lengths):
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + n)
    return cu


def _nan(shape, dtype):
    return torch.full(shape, float("nan"), device="cuda", dtype=dtype)


def run_varlen(eba, q, k, v, do, cu_q, cu_k, scale, bwd=True):
    """attn_fwd_varlen / attn_bwd_varlen through the C ABI into NaN-prefilled
    outputs and a NaN-prefilled workspace."""
    import ctypes

    Tq, H, d = q.shape
    n = len(cu_q) - 1
    aq = (ctypes.c_int * len(cu_q))(*cu_q)
    ak = (ctypes.c_int * len(cu_k))(*cu_k)
    stream = torch.cuda.current_stream().cuda_stream
    o, lse = _nan(q.shape, torch.bfloat16), _nan((H, Tq), torch.float32)
    st = eba.lib().attn_fwd_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                   lse.data_ptr(), aq, ak, n, H, d, scale, stream)
    assert st == 0, eba.status_string(st)
    if not bwd:
        return o, lse, None
    dq, dk, dv = _nan(q.shape, torch.bfloat16), _nan(k.shape, torch.bfloat16), _nan(v.shape, torch.bfloat16)
    need = eba.bwd_varlen_workspace_size(Tq, H, d, n)
    ws = torch.full((need // 4,), float("nan"), device="cuda", dtype=torch.float32)
    st = eba.lib().attn_bwd_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                   do.data_ptr(), lse.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                                   dv.data_ptr(), aq, ak, n, H, d, scale, ws.data_ptr(), need,
                                   stream)
    assert st == 0, eba.status_string(st)
    return o, lse, (dq, dk, dv)


def _np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def _rel(g, r):
    """max |g - r| / max(1, |r|), element by element."""
    g = _np(g) if isinstance(g, torch.Tensor) else g
    return float((np.abs(g - r) / np.maximum(1.0, np.abs(r))).max()) if g.size else 0.0


def _flat(g, r):
    """max |g - r| (flat max-abs)."""
    g = _np(g) if isinstance(g, torch.Tensor) else g
    return float(np.abs(g - r).max()) if g.size else 0.0


def balanced(lq, lk):
    """At most 4 queries per key in every sequence that has both."""
    return all(a <= 4 * b for a, b in zip(lq, lk) if a and b)


def _assert_errs(flat, rel, regime, what):
    """Flat bar in the balanced regime, the relative form outside it."""
    print(f"\n{what}: {'balanced' if regime else 'lopsided'}; flat max-abs {flat}")
    for n in flat:
        assert (flat[n] if regime else rel[n]) <= TOL, (what, n, flat, rel)


def _check_all(eba, lq, lk, H, d, seed):
    cu_q, cu_k = _cu(lq), _cu(lk)
    q, k, v, do = W.make_varlen_inputs(cu_q[-1], cu_k[-1], H, d, seed)
    scale = 1.0 / np.sqrt(d)
    o, lse, (dq, dk, dv) = run_varlen(eba, *(x.cuda() for x in (q, k, v, do)), cu_q, cu_k, scale)
    torch.cuda.synchronize()
    ro, rl = oracle.varlen_forward(q, k, v, cu_q, cu_k, scale)
    rdq, rdk, rdv = oracle.varlen_backward(q, k, v, do, cu_q, cu_k, scale)
    go, gl = _np(o), _np(lse)
    for name, g in (("o", go), ("dq", _np(dq)), ("dk", _np(dk)), ("dv", _np(dv))):
        assert np.isfinite(g).all(), f"{name} has unwritten elements"
    # queries of a sequence without keys: O = 0 exactly and lse = -inf
    empty = np.isneginf(rl)
    assert (np.isneginf(gl) == empty).all()
    assert np.abs(gl[~empty] - rl[~empty]).max() <= TOL_LSE
    errs = {"o": _rel(go, ro), "dq": _rel(dq, rdq), "dk": _rel(dk, rdk), "dv": _rel(dv, rdv)}
    flat = {"o": _flat(go, ro), "dq": _flat(dq, rdq), "dk": _flat(dk, rdk), "dv": _flat(dv, rdv)}
    _assert_errs(flat, errs, balanced(lq, lk), f"varlen H{H} d{d} {len(lq)} seqs")
    # exact zeros for the tokens of a sequence without keys (O, dQ) or
    # without queries (dK, dV)
    no_keys = np.repeat([b == 0 for b in lk], lq).astype(bool)
    no_queries = np.repeat([a == 0 for a in lq], lk).astype(bool)
    for g, zero in ((go, no_keys), (_np(dq), no_keys), (_np(dk), no_queries), (_np(dv), no_queries)):
        assert (g[zero] == 0).all()
    return errs


VARLEN_CASES = [
    # query lengths, key lengths, H, d
    ([98], [98], 1, 64),                                   # one sequence
    ([5, 130, 1, 257, 128], [7, 129, 1, 300, 128], 2, 64),  # ragged tiles, sequences inside tiles
    ([100, 0, 300, 129, 1, 257], [50, 70, 0, 400, 1, 128], 2, 64),  # no queries / no keys
    ([0, 0, 64], [10, 0, 64], 1, 64),                      # leading empty sequences
    # runs of sequences without queries (their dK, dV rows are zeroed as one
    # range per run), one in the middle and one at the end, beside sequences
    # long enough for several work items per CTA
    ([0, 0, 300, 0, 0, 0, 129, 700, 0, 0], [40, 200, 300, 1, 0, 130, 129, 650, 64, 3], 2, 64),
    ([0, 0, 300, 0, 0, 129, 0], [40, 200, 300, 1, 130, 129, 7], 2, 128),
    ([384, 3, 200], [384, 500, 17], 3, 64),               # three query tiles (odd pair)
    ([100, 0, 300, 129], [50, 70, 0, 400], 2, 128),
    ([1, 257, 640], [300, 1, 200], 1, 128),
]


@pytest.mark.parametrize("lq,lk,H,d", VARLEN_CASES, ids=lambda x: str(x))
def test_varlen_matches_oracle(eba, lq, lk, H, d):
    _check_all(eba, lq, lk, H, d, seed=3000 + sum(lq) + 7 * sum(lk) + d)


def test_varlen_many_short_sequences(eba):
    # 300 sequences of 1..40 tokens: many sequences per 128-row tile
    g = np.random.default_rng(7)
    lq = [int(x) for x in g.integers(1, 41, size=300)]
    lk = [int(x) for x in g.integers(1, 41, size=300)]
    _check_all(eba, lq, lk, 1, 64, seed=7)


def test_one_sequence_equals_dense(eba):
    # A single packed sequence runs the same tiles as the dense call on the
    # transposed tensors: forward O, lse and backward dK, dV are bit-identical;
    # dQ (fp32 atomic accumulation) agrees within the tolerance.
    B, H, L, d = 1, 4, 1000, 64
    q, k, v, do = W.make_varlen_inputs(L, L, H, d, seed=11)
    qd, kd, vd, dod = (x.cuda() for x in (q, k, v, do))
    scale = 0.125
    o, lse, (dq, dk, dv) = run_varlen(eba, qd, kd, vd, dod, [0, L], [0, L], scale)
    bhld = [x.transpose(0, 1).unsqueeze(0).contiguous() for x in (qd, kd, vd, dod)]
    o2, lse2 = eba.fwd(*bhld[:3], scale)
    dq2, dk2, dv2 = eba.bwd(*bhld[:3], o2, bhld[3], lse2, scale)
    torch.cuda.synchronize()
    assert torch.equal(o, o2[0].transpose(0, 1))
    assert torch.equal(lse, lse2[0])
    assert torch.equal(dk, dk2[0].transpose(0, 1))
    assert torch.equal(dv, dv2[0].transpose(0, 1))
    assert (dq.float() - dq2[0].transpose(0, 1).float()).abs().max().item() <= TOL


def test_varlen_mix_full_size_sampled(eba):
    # The packed image/video mix at full size (25088 tokens, 16 heads), checked
    # against the oracle on sampled sequences and heads.
    w = W.VARLEN_MIX
    cu = w.cu_seqlens()
    q, k, v, do = W.make_varlen_inputs(cu[-1], cu[-1], w.H, w.d, seed=w.seed)
    o, lse, (dq, dk, dv) = run_varlen(eba, *(x.cuda() for x in (q, k, v, do)), cu, cu, w.scale)
    torch.cuda.synchronize()
    g = np.random.default_rng(1)
    n = len(cu) - 1
    for s in sorted(set([0, n - 1] + [int(x) for x in g.integers(0, n, size=4)])):
        a, b = cu[s], cu[s + 1]
        for h in sorted(set([0, w.H - 1, int(g.integers(0, w.H))])):
            sl = (slice(a, b), slice(h, h + 1))
            ro, rl = oracle.varlen_forward(q[sl], k[sl], v[sl], [0, b - a], [0, b - a], w.scale)
            rdq, rdk, rdv = oracle.varlen_backward(q[sl], k[sl], v[sl], do[sl], [0, b - a],
                                                   [0, b - a], w.scale)
            # every sequence of the mix attends to itself (Lq = Lk): balanced
            assert np.abs(_np(lse[h:h + 1, a:b]) - rl).max() <= TOL_LSE
            flat = {"o": _flat(o[sl], ro), "dq": _flat(dq[sl], rdq), "dk": _flat(dk[sl], rdk),
                    "dv": _flat(dv[sl], rdv)}
            _assert_errs(flat, flat, True, f"varlen mix sequence {s} head {h}")


def test_python_binding_varlen(eba):
    lq, lk = [70, 200], [90, 30]
    cu_q, cu_k = _cu(lq), _cu(lk)
    q, k, v, do = W.make_varlen_inputs(cu_q[-1], cu_k[-1], 2, 64, seed=21)
    qd, kd, vd, dod = (x.cuda() for x in (q, k, v, do))
    o, lse = eba.fwd_varlen(qd, kd, vd, torch.tensor(cu_q), cu_k)
    dq, dk, dv = eba.bwd_varlen(qd, kd, vd, o, dod, lse, cu_q, cu_k)
    ro, rl = oracle.varlen_forward(q, k, v, cu_q, cu_k, 0.125)
    rdq, rdk, rdv = oracle.varlen_backward(q, k, v, do, cu_q, cu_k, 0.125)
    assert np.abs(_np(o) - ro).max() <= TOL
    assert np.abs(_np(lse) - rl).max() <= TOL_LSE
    assert np.abs(_np(dq) - rdq).max() <= TOL
    assert np.abs(_np(dk) - rdk).max() <= TOL
    assert np.abs(_np(dv) - rdv).max() <= TOL


@pytest.mark.parametrize("H,Hkv,d", [(4, 2, 64), (6, 1, 64), (4, 2, 128)], ids=lambda x: str(x))
def test_varlen_grouped_query_heads(eba, H, Hkv, d):
    # Packed sequences with K/V shared by groups of query heads (including a
    # sequence without keys and one without queries).
    lq, lk = [100, 0, 300, 129, 1], [50, 70, 0, 400, 1]
    cu_q, cu_k = _cu(lq), _cu(lk)
    g = torch.Generator().manual_seed(41 + H + d)
    mk = lambda T, h: torch.randn((T, h, d), generator=g).to(torch.bfloat16)
    q, do = mk(cu_q[-1], H), mk(cu_q[-1], H)
    k, v = mk(cu_k[-1], Hkv), mk(cu_k[-1], Hkv)
    scale = 1.0 / np.sqrt(d)
    o, lse = eba.fwd_varlen(*(x.cuda() for x in (q, k, v)), cu_q, cu_k, scale)
    dq, dk, dv = eba.bwd_varlen(*(x.cuda() for x in (q, k, v)), o, do.cuda(), lse, cu_q, cu_k,
                                scale)
    torch.cuda.synchronize()
    ro, rl = oracle.varlen_forward(q, k, v, cu_q, cu_k, scale)
    rdq, rdk, rdv = oracle.varlen_backward(q, k, v, do, cu_q, cu_k, scale)
    empty = np.isneginf(rl)
    gl = _np(lse)
    assert (np.isneginf(gl) == empty).all()
    assert np.abs(gl[~empty] - rl[~empty]).max() <= TOL_LSE
    errs = {"o": _rel(o, ro), "dq": _rel(dq, rdq), "dk": _rel(dk, rdk), "dv": _rel(dv, rdv)}
    assert max(errs.values()) <= TOL, errs


def test_autograd_varlen(eba):
    lq, lk = [150, 60, 1], [90, 200, 3]
    cu_q, cu_k = _cu(lq), _cu(lk)
    q, k, v, do = W.make_varlen_inputs(cu_q[-1], cu_k[-1], 2, 64, seed=57)
    qd, kd, vd = (x.cuda().requires_grad_() for x in (q, k, v))
    out = eba.attention_varlen(qd, kd, vd, cu_q, cu_k)
    out.backward(do.cuda())
    ro, _ = oracle.varlen_forward(q, k, v, cu_q, cu_k, 0.125)
    rdq, rdk, rdv = oracle.varlen_backward(q, k, v, do, cu_q, cu_k, 0.125)
    assert _rel(out, ro) <= TOL
    assert _rel(qd.grad, rdq) <= TOL and _rel(kd.grad, rdk) <= TOL and _rel(vd.grad, rdv) <= TOL
