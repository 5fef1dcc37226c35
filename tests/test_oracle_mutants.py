"""Plant plausible mistakes in copies of the oracle and check the pins catch them.

Each mutant replaces one oracle function with a version carrying one typical
slip (a dropped term, a wrong sign, a missing scale, a transposed operand, an
off-by-one range). The pins in oracle_pins.py must reject every mutant: if one
slipped through, the oracle could carry that mistake unnoticed.
"""
import types

import numpy as np
import pytest

import oracle
import oracle_pins as pins
from oracle import attention as A


def _impl(**over):
    base = dict(
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
    base.update(over)
    return types.SimpleNamespace(**base)


def _fwd_with(softmax_fn):
    def forward(q, k, v, scale):
        q, k, v = A._as_f64(q), A._as_f64(k), A._as_f64(v)
        B, H, Lq, _ = q.shape
        o = np.zeros((B, H, Lq, v.shape[3]))
        lse = np.zeros((B, H, Lq))
        for b in range(B):
            for h in range(H):
                P, l = softmax_fn(q[b, h], k[b, h], scale)
                o[b, h] = P @ v[b, h]
                lse[b, h] = l
        return o, lse
    return forward


def _sm_no_scale(q, k, scale):
    return oracle.softmax_weights(q, k, 1.0)


def _sm_wrong_axis(q, k, scale):
    S = scale * (q @ k.T)
    E = np.exp(S - S.max())
    P = E / E.sum(axis=0, keepdims=True)
    return P, np.log(np.exp(S).sum(axis=1))


def _sm_lse_drops_max(q, k, scale):
    S = scale * (q @ k.T)
    m = S.max(axis=1, keepdims=True)
    E = np.exp(S - m)
    l = E.sum(axis=1, keepdims=True)
    return E / l, np.log(l)[:, 0]


def _bwd_with(ds_fn, dq_scale=True, dk_transposed=False, dv_transposed=False):
    def backward(q, k, v, do, scale):
        q, k, v, do = (A._as_f64(x) for x in (q, k, v, do))
        dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
        for b in range(q.shape[0]):
            for h in range(q.shape[1]):
                P, _ = oracle.softmax_weights(q[b, h], k[b, h], scale)
                dv[b, h] = (P @ do[b, h]) if dv_transposed else (P.T @ do[b, h])
                dP = do[b, h] @ v[b, h].T
                dS = ds_fn(P, dP)
                dq[b, h] = (scale if dq_scale else 1.0) * (dS @ k[b, h])
                dk[b, h] = scale * ((dS @ q[b, h]) if dk_transposed else (dS.T @ q[b, h]))
        return dq, dk, dv
    return backward


def _ds_ok(P, dP):
    return P * (dP - (P * dP).sum(axis=1, keepdims=True))


def _merge_unnormalised(o_parts, lse_parts):
    o_parts, lse_parts = A._as_f64(o_parts), A._as_f64(lse_parts)
    M = lse_parts.max(axis=0)
    w = np.exp(lse_parts - M[None])
    lse = M + np.log(w.sum(axis=0))
    return (w[..., None] * o_parts).sum(axis=0), lse


def _merge_plain_mean(o_parts, lse_parts):
    o, lse = oracle.merge(o_parts, lse_parts)
    return A._as_f64(o_parts).mean(axis=0), lse


def _partial_off_by_one(q, k, v, scale, k0, k1):
    return oracle.partial_forward(q, k, v, scale, k0, min(k1 + 1, A._as_f64(k).shape[2]))


def _varlen_fwd_with(key_range, guard_empty=True, lse_token_major=False):
    def varlen_forward(q, k, v, cu_q, cu_k, scale):
        q, k, v = A._as_f64(q), A._as_f64(k), A._as_f64(v)
        Tq, H, _ = q.shape
        o = np.zeros((Tq, H, v.shape[2]))
        lse = np.full((H, Tq), -np.inf)
        for s_ in range(len(cu_q) - 1):
            q0, q1 = cu_q[s_], cu_q[s_ + 1]
            k0, k1 = key_range(cu_q, cu_k, s_)
            if q1 <= q0 or (guard_empty and k1 <= k0):
                continue
            for h in range(H):
                P, l = oracle.softmax_weights(q[q0:q1, h], k[k0:k1, h], scale)
                o[q0:q1, h] = P @ v[k0:k1, h]
                lse[h, q0:q1] = l
        return o, (lse.T.copy() if lse_token_major else lse)
    return varlen_forward


def _varlen_bwd_drops_rowsum(q, k, v, do, cu_q, cu_k, scale):
    q, k, v, do = A._as_f64(q), A._as_f64(k), A._as_f64(v), A._as_f64(do)
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    for s_ in range(len(cu_q) - 1):
        q0, q1, k0, k1 = cu_q[s_], cu_q[s_ + 1], cu_k[s_], cu_k[s_ + 1]
        if q1 <= q0 or k1 <= k0:
            continue
        for h in range(q.shape[1]):
            P, _ = oracle.softmax_weights(q[q0:q1, h], k[k0:k1, h], scale)
            dv[k0:k1, h] = P.T @ do[q0:q1, h]
            dS = P * (do[q0:q1, h] @ v[k0:k1, h].T)
            dq[q0:q1, h] = scale * (dS @ k[k0:k1, h])
            dk[k0:k1, h] = scale * (dS.T @ q[q0:q1, h])
    return dq, dk, dv


def _gqa_fwd_with(kv_head):
    def gqa_forward(q, k, v, scale):
        q, k, v = A._as_f64(q), A._as_f64(k), A._as_f64(v)
        B, H, Lq, _ = q.shape
        Hkv = k.shape[1]
        o = np.zeros((B, H, Lq, v.shape[3]))
        lse = np.zeros((B, H, Lq))
        for b in range(B):
            for h in range(H):
                j = kv_head(h, H, Hkv)
                P, l = oracle.softmax_weights(q[b, h], k[b, j], scale)
                o[b, h] = P @ v[b, j]
                lse[b, h] = l
        return o, lse
    return gqa_forward


def _gqa_bwd_last_head_wins(q, k, v, do, scale):
    # dK, dV of a K/V head taken from the last query head of its group only
    q, k, v, do = A._as_f64(q), A._as_f64(k), A._as_f64(v), A._as_f64(do)
    G = q.shape[1] // k.shape[1]
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    for b in range(q.shape[0]):
        for h in range(q.shape[1]):
            kh, vh = k[b, h // G], v[b, h // G]
            P, _ = oracle.softmax_weights(q[b, h], kh, scale)
            dv[b, h // G] = P.T @ do[b, h]
            dP = do[b, h] @ vh.T
            dS = P * (dP - (P * dP).sum(axis=1, keepdims=True))
            dq[b, h] = scale * (dS @ kh)
            dk[b, h // G] = scale * (dS.T @ q[b, h])
    return dq, dk, dv


_own_keys = lambda cu_q, cu_k, s_: (cu_k[s_], cu_k[s_ + 1])

MUTANTS = {
    "gqa_heads_interleaved": _impl(gqa_forward=_gqa_fwd_with(lambda h, H, Hkv: h % Hkv)),
    "gqa_all_heads_on_first_kv": _impl(gqa_forward=_gqa_fwd_with(lambda h, H, Hkv: 0)),
    "gqa_bwd_last_head_wins": _impl(gqa_backward=_gqa_bwd_last_head_wins),
    "varlen_key_range_off_by_one": _impl(varlen_forward=_varlen_fwd_with(
        lambda cu_q, cu_k, s_: (cu_k[s_], cu_k[s_ + 1] - 1))),
    "varlen_keys_at_query_offsets": _impl(varlen_forward=_varlen_fwd_with(
        lambda cu_q, cu_k, s_: (cu_q[s_], cu_q[s_ + 1]))),
    "varlen_no_empty_guard": _impl(varlen_forward=_varlen_fwd_with(_own_keys, guard_empty=False)),
    "varlen_lse_token_major": _impl(varlen_forward=_varlen_fwd_with(_own_keys, lse_token_major=True)),
    "varlen_bwd_drops_rowsum_term": _impl(varlen_backward=_varlen_bwd_drops_rowsum),
    "fwd_missing_scale": _impl(forward=_fwd_with(_sm_no_scale), softmax_weights=_sm_no_scale),
    "fwd_softmax_wrong_axis": _impl(forward=_fwd_with(_sm_wrong_axis), softmax_weights=_sm_wrong_axis),
    "fwd_lse_drops_max": _impl(forward=_fwd_with(_sm_lse_drops_max)),
    "bwd_drops_rowsum_term": _impl(backward=_bwd_with(lambda P, dP: P * dP)),
    "bwd_wrong_sign": _impl(backward=_bwd_with(lambda P, dP: P * ((P * dP).sum(axis=1, keepdims=True) - dP))),
    "bwd_dq_missing_scale": _impl(backward=_bwd_with(_ds_ok, dq_scale=False)),
    "bwd_dk_transposed": _impl(backward=_bwd_with(_ds_ok, dk_transposed=True)),
    "bwd_dv_transposed": _impl(backward=_bwd_with(_ds_ok, dv_transposed=True)),
    "merge_unnormalised": _impl(merge=_merge_unnormalised),
    "merge_plain_mean": _impl(merge=_merge_plain_mean),
    "partial_off_by_one": _impl(partial_forward=_partial_off_by_one),
}


def _fails_some_pin(impl):
    for check in pins.ALL_CHECKS:
        try:
            with np.errstate(all="ignore"):
                check(impl)
        except ImportError:
            continue
        except Exception:
            return check.__name__
    return None


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    caught_by = _fails_some_pin(MUTANTS[name])
    assert caught_by is not None, f"mutant {name} passed every pin"
