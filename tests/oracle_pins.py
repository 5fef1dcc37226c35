"""Checks that pin the CPU oracle to facts fixed outside itself.

Each check takes an implementation namespace ``impl`` with the oracle's
functions (forward, backward, partial_forward, merge, softmax_weights,
varlen_forward, varlen_backward) so the
same checks can be run against deliberately broken copies (see
test_oracle_mutants.py): a plausible mistake in the oracle must fail at least
one of them.

What pins what:
  * hand-derived closed forms (tests/golden/closed_forms.json),
  * 50-digit brute force with mpmath on tiny inputs,
  * identical keys -> mean of V, one key -> that value, zero query -> mean,
  * invariance to shifting every key and to permuting (K, V) rows together,
  * rows of the softmax sum to one,
  * central finite differences of sum(O * dO) for the gradients,
  * sum over keys of dK is zero,
  * merge of partial ranges equals the unsplit result,
  * torch's float64 CPU scaled_dot_product_attention and its autograd,
  * packed sequences: torch's attention with a block-diagonal mask, sequence
    independence and reordering, one sequence = the dense result,
  * grouped-query heads: torch's attention with enable_gqa (also under the
    block-diagonal mask of packed sequences), one K/V head per query head =
    multi-head attention, finite differences with one K/V head for all.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_forms.json")


def _f(x):
    """Parse JSON numbers, with "-inf" / "inf" strings."""
    return np.vectorize(lambda t: float(t))(np.array(x, dtype=object)).astype(np.float64)


def _head(x):
    """[L, d] -> [1, 1, L, d]."""
    return np.asarray(x, dtype=np.float64)[None, None]


def rng(seed):
    return np.random.default_rng(seed)


def check_golden(impl, tol=1e-12):
    data = json.load(open(GOLDEN))
    for c in data["cases"]:
        q, k, v, do = (_head(_f(c[n])) for n in ("q", "k", "v", "do"))
        s = float(c["scale"])
        o, lse = impl.forward(q, k, v, s)
        assert np.allclose(o[0, 0], _f(c["o"]), atol=tol, rtol=0), (c["name"], "o")
        assert np.allclose(lse[0, 0], _f(c["lse"]), atol=tol, rtol=0), (c["name"], "lse")
        dq, dk, dv = impl.backward(q, k, v, do, s)
        assert np.allclose(dq[0, 0], _f(c["dq"]), atol=tol, rtol=0), (c["name"], "dq")
        assert np.allclose(dk[0, 0], _f(c["dk"]), atol=tol, rtol=0), (c["name"], "dk")
        assert np.allclose(dv[0, 0], _f(c["dv"]), atol=tol, rtol=0), (c["name"], "dv")
    for c in data["merge_cases"]:
        o_parts = _f(c["o_parts"])[:, None, None]        # [C,1,1,Lq,d]
        lse_parts = _f(c["lse_parts"])[:, None, None]    # [C,1,1,Lq]
        o, lse = impl.merge(o_parts, lse_parts)
        assert np.allclose(o[0, 0], _f(c["o"]), atol=tol, rtol=0), (c["name"], "o")
        exp_lse = _f(c["lse"])
        assert np.array_equal(np.isneginf(lse[0, 0]), np.isneginf(exp_lse)), (c["name"], "lse inf")
        fin = ~np.isneginf(exp_lse)
        assert np.allclose(lse[0, 0][fin], exp_lse[fin], atol=tol, rtol=0), (c["name"], "lse")


def check_mpmath_bruteforce(impl, seed=11, Lq=3, Lk=4, d=3, tol=1e-13):
    """Evaluate the definition in 50-digit arithmetic on a tiny random case."""
    import mpmath

    mpmath.mp.dps = 50
    r = rng(seed)
    q, k, v = r.normal(size=(Lq, d)), r.normal(size=(Lk, d)), r.normal(size=(Lk, d))
    s = 0.7
    o, lse = impl.forward(_head(q), _head(k), _head(v), s)
    for i in range(Lq):
        sc = [mpmath.mpf(s) * mpmath.fsum(mpmath.mpf(q[i, t]) * mpmath.mpf(k[j, t]) for t in range(d))
              for j in range(Lk)]
        ex = [mpmath.e ** x for x in sc]
        tot = mpmath.fsum(ex)
        assert abs(float(mpmath.log(tot)) - lse[0, 0, i]) < tol
        for t in range(d):
            oi = mpmath.fsum(ex[j] * mpmath.mpf(v[j, t]) for j in range(Lk)) / tot
            assert abs(float(oi) - o[0, 0, i, t]) < tol


def check_softmax_rows(impl, seed=1):
    r = rng(seed)
    q, k = r.normal(size=(9, 8)) * 2, r.normal(size=(13, 8)) * 2
    P, _ = impl.softmax_weights(q, k, 0.5)
    assert P.shape == (9, 13)
    assert (P >= 0).all()
    assert np.abs(P.sum(axis=1) - 1.0).max() < 1e-12


def check_identical_keys(impl, seed=2, Lq=6, Lk=11, d=5, s=0.3):
    r = rng(seed)
    q = r.normal(size=(Lq, d))
    krow = r.normal(size=(1, d))
    k = np.repeat(krow, Lk, axis=0)
    v = r.normal(size=(Lk, d))
    o, lse = impl.forward(_head(q), _head(k), _head(v), s)
    assert np.abs(o[0, 0] - v.mean(axis=0)[None]).max() < 1e-12
    exp_lse = math.log(Lk) + s * (q @ krow[0])
    assert np.abs(lse[0, 0] - exp_lse).max() < 1e-12


def check_single_key(impl, seed=3):
    r = rng(seed)
    q, k, v = r.normal(size=(4, 6)), r.normal(size=(1, 6)), r.normal(size=(1, 6))
    o, lse = impl.forward(_head(q), _head(k), _head(v), 0.9)
    assert np.abs(o[0, 0] - v).max() < 1e-12
    assert np.abs(lse[0, 0] - 0.9 * (q @ k[0])).max() < 1e-12


def check_zero_query(impl, seed=4):
    r = rng(seed)
    q = np.zeros((3, 4))
    k, v = r.normal(size=(7, 4)), r.normal(size=(7, 4))
    o, lse = impl.forward(_head(q), _head(k), _head(v), 1.3)
    assert np.abs(o[0, 0] - v.mean(axis=0)).max() < 1e-12
    assert np.abs(lse[0, 0] - math.log(7)).max() < 1e-12


def check_key_shift(impl, seed=5, s=0.4):
    """Adding c to every key leaves O unchanged and shifts lse_i by s q_i.c."""
    r = rng(seed)
    q, k, v = r.normal(size=(5, 6)), r.normal(size=(9, 6)), r.normal(size=(9, 6))
    c = r.normal(size=(6,))
    o1, l1 = impl.forward(_head(q), _head(k), _head(v), s)
    o2, l2 = impl.forward(_head(q), _head(k + c), _head(v), s)
    assert np.abs(o1 - o2).max() < 1e-12
    assert np.abs(l2[0, 0] - l1[0, 0] - s * (q @ c)).max() < 1e-12


def check_kv_permutation(impl, seed=6):
    r = rng(seed)
    q, k, v = r.normal(size=(5, 4)), r.normal(size=(8, 4)), r.normal(size=(8, 4))
    perm = r.permutation(8)
    o1, l1 = impl.forward(_head(q), _head(k), _head(v), 0.8)
    o2, l2 = impl.forward(_head(q), _head(k[perm]), _head(v[perm]), 0.8)
    assert np.abs(o1 - o2).max() < 1e-12
    assert np.abs(l1 - l2).max() < 1e-12


def check_finite_differences(impl, seed=7, Lq=5, Lk=7, d=4, s=0.6, h=1e-6, tol=1e-6):
    """Central differences of L = sum(O * dO) against the analytic gradients."""
    r = rng(seed)
    q, k, v, do = (r.normal(size=sh) for sh in ((Lq, d), (Lk, d), (Lk, d), (Lq, d)))

    def loss(args):
        o, _ = impl.forward(_head(args["q"]), _head(args["k"]), _head(args["v"]), s)
        return float((o[0, 0] * do).sum())

    dq, dk, dv = impl.backward(_head(q), _head(k), _head(v), _head(do), s)
    for name, x, g in (("q", q, dq[0, 0]), ("k", k, dk[0, 0]), ("v", v, dv[0, 0])):
        num = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            plus = {"q": q, "k": k, "v": v, name: xp}
            minus = {"q": q, "k": k, "v": v, name: xm}
            num[idx] = (loss(plus) - loss(minus)) / (2 * h)
        rel = np.abs(num - g).max() / max(np.abs(num).max(), 1e-30)
        assert rel < tol, (name, rel)


def check_dk_sums_to_zero(impl, seed=8):
    r = rng(seed)
    q, k, v, do = (r.normal(size=sh) for sh in ((6, 5), (10, 5), (10, 5), (6, 5)))
    _, dk, _ = impl.backward(_head(q), _head(k), _head(v), _head(do), 0.5)
    assert np.abs(dk[0, 0].sum(axis=0)).max() < 1e-12


def check_merge_equals_unsplit(impl, seed=9):
    r = rng(seed)
    B, H, Lq, Lk, d = 2, 3, 7, 29, 8
    q, k, v = (r.normal(size=(B, H, L, d)) for L in (Lq, Lk, Lk))
    s = 0.35
    o_ref, lse_ref = impl.forward(q, k, v, s)
    splits = [
        [(0, Lk)],                                    # C = 1
        [(0, 14), (14, Lk)],                          # C = 2
        [(0, 5), (5, 6), (6, Lk)],                    # C = 3, uneven
        [(0, 3), (3, 3), (3, 10), (10, 11), (11, 11), (11, 20), (20, 28), (28, Lk)],  # C = 8, empties
    ]
    for bounds in splits:
        parts = [impl.partial_forward(q, k, v, s, a, b) for a, b in bounds]
        o, lse = impl.merge(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
        assert np.abs(o - o_ref).max() < 1e-12, bounds
        assert np.abs(lse - lse_ref).max() < 1e-12, bounds


def check_empty_partial(impl):
    q, k, v = np.ones((1, 1, 3, 2)), np.ones((1, 1, 5, 2)), np.ones((1, 1, 5, 2))
    o, lse = impl.partial_forward(q, k, v, 1.0, 2, 2)
    assert (o == 0).all() and np.isneginf(lse).all()


def check_torch_sdpa(impl, seed=10):
    """torch's float64 CPU attention (and autograd) is an independent routine."""
    import torch

    r = rng(seed)
    B, H, Lq, Lk, d = 2, 2, 9, 17, 8
    q, k, v, do = (r.normal(size=(B, H, L, d)) for L in (Lq, Lk, Lk, Lq))
    s = 0.45
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    to = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, scale=s)
    to.backward(torch.tensor(do))
    o, _ = impl.forward(q, k, v, s)
    dq, dk, dv = impl.backward(q, k, v, do, s)
    assert np.abs(o - to.detach().numpy()).max() < 1e-10
    assert np.abs(dq - tq.grad.numpy()).max() < 1e-10
    assert np.abs(dk - tk.grad.numpy()).max() < 1e-10
    assert np.abs(dv - tv.grad.numpy()).max() < 1e-10


def _varlen_case(r, H=2, d=5):
    """Packed sequences with uneven lengths, one without keys and one without
    queries: cu_q, cu_k and token-major q, k, v, dO."""
    lq = [4, 0, 7, 3, 5]
    lk = [6, 3, 5, 0, 9]
    cu_q = [0] + list(np.cumsum(lq))
    cu_k = [0] + list(np.cumsum(lk))
    q = r.normal(size=(cu_q[-1], H, d))
    k = r.normal(size=(cu_k[-1], H, d))
    v = r.normal(size=(cu_k[-1], H, d))
    do = r.normal(size=(cu_q[-1], H, d))
    return cu_q, cu_k, q, k, v, do


def check_varlen_torch_blockmask(impl, seed=12, s=0.5):
    """Packed sequences = attention over all tokens with a block-diagonal
    mask, computed by torch's float64 CPU attention (and its autograd) and
    torch's logsumexp: independent routines."""
    import torch

    r = rng(seed)
    cu_q, cu_k, q, k, v, do = _varlen_case(r)
    Tq, H, d = q.shape
    seq_q = np.repeat(np.arange(len(cu_q) - 1), np.diff(cu_q))
    seq_k = np.repeat(np.arange(len(cu_k) - 1), np.diff(cu_k))
    mask = torch.tensor(seq_q[:, None] == seq_k[None, :])
    has_keys = mask.any(dim=1).numpy()
    tq, tk, tv = (torch.tensor(x.transpose(1, 0, 2)[None], requires_grad=True) for x in (q, k, v))
    to = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask, scale=s)
    tdo = torch.tensor(do.transpose(1, 0, 2)[None])
    # rows without keys are NaN in torch (fully masked); they carry no gradient here
    (torch.nan_to_num(to) * tdo).sum().backward()
    scores = s * (tq.detach() @ tk.detach().transpose(-1, -2))
    tlse = torch.logsumexp(scores.masked_fill(~mask, float("-inf")), dim=-1)[0].numpy()
    o, lse = impl.varlen_forward(q, k, v, cu_q, cu_k, s)
    dq, dk, dv = impl.varlen_backward(q, k, v, do, cu_q, cu_k, s)
    ref_o = to.detach()[0].numpy().transpose(1, 0, 2)
    assert np.abs(o[has_keys] - ref_o[has_keys]).max() < 1e-10
    assert (o[~has_keys] == 0).all()
    assert np.abs(lse[:, has_keys] - tlse[:, has_keys]).max() < 1e-10
    assert np.isneginf(lse[:, ~has_keys]).all()
    for g, tg in ((dq, tq), (dk, tk), (dv, tv)):
        assert np.abs(g - tg.grad[0].numpy().transpose(1, 0, 2)).max() < 1e-10


def check_varlen_independent_sequences(impl, seed=13, s=0.7):
    """Changing one sequence's tokens leaves every other sequence's outputs and
    gradients bit-identical; reordering the sequences reorders the outputs."""
    r = rng(seed)
    cu_q, cu_k, q, k, v, do = _varlen_case(r)
    o, lse = impl.varlen_forward(q, k, v, cu_q, cu_k, s)
    g = impl.varlen_backward(q, k, v, do, cu_q, cu_k, s)
    q2, k2, v2 = q.copy(), k.copy(), v.copy()
    q2[cu_q[2]:cu_q[3]] += 1.0
    k2[cu_k[2]:cu_k[3]] -= 0.5
    v2[cu_k[2]:cu_k[3]] *= 2.0
    o2, lse2 = impl.varlen_forward(q2, k2, v2, cu_q, cu_k, s)
    g2 = impl.varlen_backward(q2, k2, v2, do, cu_q, cu_k, s)
    keep_q = np.ones(q.shape[0], bool)
    keep_q[cu_q[2]:cu_q[3]] = False
    keep_k = np.ones(k.shape[0], bool)
    keep_k[cu_k[2]:cu_k[3]] = False
    assert (o2[keep_q] == o[keep_q]).all() and (lse2[:, keep_q] == lse[:, keep_q]).all()
    assert (g2[0][keep_q] == g[0][keep_q]).all()
    assert (g2[1][keep_k] == g[1][keep_k]).all() and (g2[2][keep_k] == g[2][keep_k]).all()
    # reverse the order of the sequences
    n = len(cu_q) - 1
    segs_q = [slice(cu_q[i], cu_q[i + 1]) for i in range(n)][::-1]
    segs_k = [slice(cu_k[i], cu_k[i + 1]) for i in range(n)][::-1]
    rq = np.concatenate([q[sl] for sl in segs_q])
    rk = np.concatenate([k[sl] for sl in segs_k])
    rv = np.concatenate([v[sl] for sl in segs_k])
    rcu_q = [0] + list(np.cumsum([sl.stop - sl.start for sl in segs_q]))
    rcu_k = [0] + list(np.cumsum([sl.stop - sl.start for sl in segs_k]))
    ro, rlse = impl.varlen_forward(rq, rk, rv, rcu_q, rcu_k, s)
    assert (ro == np.concatenate([o[sl] for sl in segs_q])).all()
    assert (rlse == np.concatenate([lse[:, sl] for sl in segs_q], axis=1)).all()


def check_varlen_one_sequence_is_dense(impl, seed=14, s=0.35):
    """One sequence: the packed forward and backward are the dense ones."""
    r = rng(seed)
    Lq, Lk, H, d = 6, 9, 3, 4
    q, k, v, do = (r.normal(size=(L, H, d)) for L in (Lq, Lk, Lk, Lq))
    o, lse = impl.varlen_forward(q, k, v, [0, Lq], [0, Lk], s)
    dq, dk, dv = impl.varlen_backward(q, k, v, do, [0, Lq], [0, Lk], s)
    bhld = lambda x: x.transpose(1, 0, 2)[None]
    do_, dlse = impl.forward(bhld(q), bhld(k), bhld(v), s)
    ddq, ddk, ddv = impl.backward(bhld(q), bhld(k), bhld(v), bhld(do), s)
    assert np.abs(bhld(o) - do_).max() < 1e-12 and np.abs(lse - dlse[0]).max() < 1e-12
    for a, b in ((dq, ddq), (dk, ddk), (dv, ddv)):
        assert np.abs(bhld(a) - b).max() < 1e-12


def _gqa_case(r, B=2, H=6, H_kv=2, Lq=5, Lk=7, d=4):
    q = r.normal(size=(B, H, Lq, d))
    k = r.normal(size=(B, H_kv, Lk, d))
    v = r.normal(size=(B, H_kv, Lk, d))
    do = r.normal(size=(B, H, Lq, d))
    return q, k, v, do


def check_gqa_torch(impl, seed=15, s=0.45):
    """Grouped-query attention against torch's float64 attention with
    enable_gqa (its own head grouping and autograd) and torch's logsumexp."""
    import torch

    r = rng(seed)
    q, k, v, do = _gqa_case(r)
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    to = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, scale=s, enable_gqa=True)
    (to * torch.tensor(do)).sum().backward()
    o, lse = impl.gqa_forward(q, k, v, s)
    dq, dk, dv = impl.gqa_backward(q, k, v, do, s)
    assert np.abs(o - to.detach().numpy()).max() < 1e-10
    for g, tg in ((dq, tq), (dk, tk), (dv, tv)):
        assert np.abs(g - tg.grad.numpy()).max() < 1e-10
    # lse: torch's logsumexp over each query head's scores against its group's keys
    G = q.shape[1] // k.shape[1]
    for h in range(q.shape[1]):
        sc = s * torch.tensor(q[:, h]) @ torch.tensor(k[:, h // G]).transpose(-1, -2)
        assert np.abs(lse[:, h] - torch.logsumexp(sc, dim=-1).numpy()).max() < 1e-10


def check_gqa_one_group_per_head_is_mha(impl, seed=16, s=0.6):
    """H_kv = H: grouped-query attention is plain multi-head attention."""
    r = rng(seed)
    q, k, v, do = _gqa_case(r, H=3, H_kv=3)
    o, lse = impl.gqa_forward(q, k, v, s)
    g = impl.gqa_backward(q, k, v, do, s)
    o2, lse2 = impl.forward(q, k, v, s)
    g2 = impl.backward(q, k, v, do, s)
    assert np.abs(o - o2).max() < 1e-12 and np.abs(lse - lse2).max() < 1e-12
    for a, b in zip(g, g2):
        assert np.abs(a - b).max() < 1e-12


def check_gqa_single_kv_head_finite_differences(impl, seed=17, s=0.5, h=1e-6):
    """All query heads on one K/V head (H_kv = 1): central finite differences
    of sum(O * dO) in K and V match dK, dV, which sum over every head."""
    r = rng(seed)
    q, k, v, do = _gqa_case(r, B=1, H=3, H_kv=1, Lq=4, Lk=5, d=3)
    dq, dk, dv = impl.gqa_backward(q, k, v, do, s)

    def f(kk, vv):
        return float((impl.gqa_forward(q, kk, vv, s)[0] * do).sum())

    for arr, grad, which in ((k, dk, 0), (v, dv, 1)):
        it = np.nditer(arr, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            a, b = arr.copy(), arr.copy()
            a[idx] += h
            b[idx] -= h
            num = (f(a, v) - f(b, v)) if which == 0 else (f(k, a) - f(k, b))
            num /= 2 * h
            assert abs(num - grad[idx]) < 1e-6 * max(1.0, abs(num))


def check_varlen_gqa_torch_blockmask(impl, seed=18, s=0.55):
    """Packed sequences with grouped K/V heads = torch's float64 attention with
    enable_gqa under the block-diagonal mask (and its autograd)."""
    import torch

    r = rng(seed)
    lq, lk = [4, 0, 7, 3], [6, 3, 5, 0]
    cu_q = [0] + list(np.cumsum(lq))
    cu_k = [0] + list(np.cumsum(lk))
    H, Hkv, d = 6, 2, 4
    q = r.normal(size=(cu_q[-1], H, d))
    k = r.normal(size=(cu_k[-1], Hkv, d))
    v = r.normal(size=(cu_k[-1], Hkv, d))
    do = r.normal(size=(cu_q[-1], H, d))
    seq_q = np.repeat(np.arange(len(lq)), lq)
    seq_k = np.repeat(np.arange(len(lk)), lk)
    mask = torch.tensor(seq_q[:, None] == seq_k[None, :])
    has_keys = mask.any(dim=1).numpy()
    tq, tk, tv = (torch.tensor(x.transpose(1, 0, 2)[None], requires_grad=True) for x in (q, k, v))
    to = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask, scale=s,
                                                          enable_gqa=True)
    (torch.nan_to_num(to) * torch.tensor(do.transpose(1, 0, 2)[None])).sum().backward()
    o, lse = impl.varlen_forward(q, k, v, cu_q, cu_k, s)
    dq, dk, dv = impl.varlen_backward(q, k, v, do, cu_q, cu_k, s)
    ref_o = to.detach()[0].numpy().transpose(1, 0, 2)
    assert np.abs(o[has_keys] - ref_o[has_keys]).max() < 1e-10
    assert (o[~has_keys] == 0).all() and np.isneginf(lse[:, ~has_keys]).all()
    for g, tg in ((dq, tq), (dk, tk), (dv, tv)):
        assert np.abs(g - tg.grad[0].numpy().transpose(1, 0, 2)).max() < 1e-10


ALL_CHECKS = [
    check_golden,
    check_mpmath_bruteforce,
    check_softmax_rows,
    check_identical_keys,
    check_single_key,
    check_zero_query,
    check_key_shift,
    check_kv_permutation,
    check_finite_differences,
    check_dk_sums_to_zero,
    check_merge_equals_unsplit,
    check_empty_partial,
    check_torch_sdpa,
    check_varlen_torch_blockmask,
    check_varlen_independent_sequences,
    check_varlen_one_sequence_is_dense,
    check_gqa_torch,
    check_gqa_one_group_per_head_is_mha,
    check_gqa_single_kv_head_finite_differences,
    check_varlen_gqa_torch_blockmask,
]
