"""CPU oracle for exact softmax attention, in float64. TEST INFRASTRUCTURE ONLY.

Only the tests, the smoke check and the benchmark's CPU-baseline leg may import
this module. The product path (the CUDA library and its Python binding) never
calls it and shares no code with it.

What is computed, per (batch, head), written out from the definition with no
blocking, fusion or reordering:

* Attention is a weighted average of the values whose weights are a softmax of
  query-key dot products ("Training a Large Video Model on a Single Machine in
  a Day", §3 "Flash Attention"). With a softmax scale s:
      S = s * Q K^T,  P = softmax_rows(S),  O = P V,
      lse_i = log sum_j exp(S_ij)   (natural log).
  The blockwise method of that page (§1, §3, §4.1) claims to reach exactly this
  result without storing S, so the plain definition is the oracle.
* Gradients of sum(O * dO) by the softmax Jacobian (the pages do not spell the
  backward out; this is the analytic derivative of the definition above):
      dV = P^T dO,  dP = dO V^T,
      dS_ij = P_ij * (dP_ij - sum_k P_ik dP_ik),
      dQ = s * dS K,  dK = s * dS^T Q.
* Partial attention over a key range [k0, k1) and the exact merge of such
  partials ("LV-XAttn", ICML 2025 poster, Abstract and Lay Summary: key/value
  blocks stay where they are and the split attention is exact, leaving the
  output unchanged). A partial is the definition applied to K[k0:k1],
  V[k0:k1]; its O is that range's own normalised output. Merge:
      M = max_c lse_c,  lse = M + log sum_c exp(lse_c - M),
      O = sum_c exp(lse_c - lse) * O_c.
  An empty range gives O_c = 0 and lse_c = -inf; the merge gives weight 0 to
  such chunks, and O = 0, lse = -inf when every chunk is empty.

* Packed variable-length sequences (the sequence packing of the NeMo video
  foundation-model page, "Sequence packing"): tokens of many sequences lie
  back to back, token-major [T, H, d]; sequence s owns queries
  [cu_q[s], cu_q[s+1]) and keys/values [cu_k[s], cu_k[s+1]) and attends only
  within itself. That is the definition above applied to each sequence; a
  sequence with queries but no keys gives O = 0 and lse = -inf (the empty
  range above), and zero gradients.

* Grouped-query attention (the GQA of the MovieGen Llama architecture named
  on the NeMo video foundation-model page, "Overview of the video diffusion
  pipeline"): H query heads share H_kv key/value heads, G = H / H_kv query
  heads per K/V head, query head h reading K/V head h // G (consecutive query
  heads form a group). Each query head is the definition above with its
  group's K, V; a K/V head's gradients are the sums over the query heads that
  read it (the chain rule through a shared input).

Readings where the pages are silent (scale, no masking, natural-log lse,
normalised fp32 partials, empty chunks) are listed in the design notes.

Every function here is pinned by the CPU tests against closed forms,
invariants, finite differences and an independent library routine.
"""
from __future__ import annotations

import numpy as np


def _as_f64(x) -> np.ndarray:
    """Upcast a torch tensor or array to a float64 numpy array (exact for bf16)."""
    try:
        import torch

        if isinstance(x, torch.Tensor):
            return x.detach().to(torch.float64).cpu().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x, dtype=np.float64)


def _heads(x: np.ndarray):
    """View [B, H, L, d] as an iterable of per-head [L, d] matrices."""
    B, H = x.shape[:2]
    for b in range(B):
        for h in range(H):
            yield b, h


def softmax_weights(q_h: np.ndarray, k_h: np.ndarray, scale: float):
    """One head: S = s Q K^T, P = softmax over keys, lse = log sum exp S.

    Row max subtraction is only there to keep exp() finite; mathematically
    P_ij = exp(S_ij) / sum_j exp(S_ij).
    """
    S = scale * (q_h @ k_h.T)
    m = S.max(axis=1, keepdims=True)
    E = np.exp(S - m)
    l = E.sum(axis=1, keepdims=True)
    P = E / l
    lse = (m + np.log(l))[:, 0]
    return P, lse


def forward(q, k, v, scale: float):
    """O = softmax(s Q K^T) V and lse per row, for [B, H, L, d] inputs.

    Returns (O [B,H,Lq,d], lse [B,H,Lq]) as float64 arrays.
    """
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    B, H, Lq, d = q.shape
    o = np.zeros((B, H, Lq, v.shape[3]))
    lse = np.zeros((B, H, Lq))
    for b, h in _heads(q):
        P, lse_h = softmax_weights(q[b, h], k[b, h], scale)
        o[b, h] = P @ v[b, h]
        lse[b, h] = lse_h
    return o, lse


def backward(q, k, v, do, scale: float):
    """Analytic gradients (dQ, dK, dV) of sum(O * dO) with O = forward(q,k,v).

    Uses the softmax Jacobian directly: dS = P * (dP - rowsum(P * dP)).
    Returns float64 arrays shaped like q, k, v.
    """
    q, k, v, do = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(do)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b, h in _heads(q):
        P, _ = softmax_weights(q[b, h], k[b, h], scale)
        dv[b, h] = P.T @ do[b, h]
        dP = do[b, h] @ v[b, h].T
        dS = P * (dP - (P * dP).sum(axis=1, keepdims=True))
        dq[b, h] = scale * (dS @ k[b, h])
        dk[b, h] = scale * (dS.T @ q[b, h])
    return dq, dk, dv


def partial_forward(q, k, v, scale: float, k0: int, k1: int):
    """Attention of every query over keys [k0, k1) only: (O_c, lse_c).

    O_c is normalised over the range; an empty range gives O_c = 0 and
    lse_c = -inf.
    """
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    B, H, Lq, _ = q.shape
    if k1 <= k0:
        return np.zeros((B, H, Lq, v.shape[3])), np.full((B, H, Lq), -np.inf)
    return forward(q, k[:, :, k0:k1], v[:, :, k0:k1], scale)


def merge(o_parts, lse_parts):
    """Exact merge of C partials: o_parts [C,B,H,Lq,d], lse_parts [C,B,H,Lq].

    Returns (O, lse). Chunks with lse = -inf carry weight 0; if all are -inf the
    row's output is O = 0 and lse = -inf.
    """
    o_parts = _as_f64(o_parts)
    lse_parts = _as_f64(lse_parts)
    M = lse_parts.max(axis=0)
    empty = np.isneginf(M)
    M_safe = np.where(empty, 0.0, M)
    w = np.exp(lse_parts - M_safe[None])            # exp(-inf) = 0 for empty chunks
    tot = w.sum(axis=0)
    with np.errstate(divide="ignore"):
        lse = np.where(empty, -np.inf, M_safe + np.log(np.where(empty, 1.0, tot)))
    lse_safe = np.where(empty, 0.0, lse)
    coef = np.exp(lse_parts - lse_safe[None])        # = w / tot where not empty
    coef = np.where(empty[None], 0.0, coef)
    o = (coef[..., None] * o_parts).sum(axis=0)
    return o, lse


def split_forward(q, k, v, scale: float, bounds):
    """Partial attention per key range followed by the merge."""
    parts = [partial_forward(q, k, v, scale, k0, k1) for (k0, k1) in bounds]
    o_parts = np.stack([p[0] for p in parts])
    lse_parts = np.stack([p[1] for p in parts])
    return merge(o_parts, lse_parts)


def varlen_forward(q, k, v, cu_q, cu_k, scale: float):
    """Packed sequences, token-major q [Tq, H, d], k and v [Tk, H_kv, d]
    (H_kv = H, or a divisor of H for grouped-query attention: query head h
    reads K/V head h // (H / H_kv)).

    Sequence s: queries q[cu_q[s]:cu_q[s+1]] over keys k[cu_k[s]:cu_k[s+1]].
    Returns (O [Tq, H, d], lse [H, Tq]) as float64 arrays.
    """
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    Tq, H, _ = q.shape
    G = H // k.shape[1]
    o = np.zeros((Tq, H, v.shape[2]))
    lse = np.full((H, Tq), -np.inf)
    for s in range(len(cu_q) - 1):
        q0, q1, k0, k1 = cu_q[s], cu_q[s + 1], cu_k[s], cu_k[s + 1]
        if q1 <= q0 or k1 <= k0:
            continue  # no queries, or no keys: O = 0, lse = -inf
        for h in range(H):
            P, lse_h = softmax_weights(q[q0:q1, h], k[k0:k1, h // G], scale)
            o[q0:q1, h] = P @ v[k0:k1, h // G]
            lse[h, q0:q1] = lse_h
    return o, lse


def varlen_backward(q, k, v, do, cu_q, cu_k, scale: float):
    """Gradients (dQ, dK, dV) of sum(O * dO) for varlen_forward, per sequence
    and head by the softmax Jacobian; tokens of a sequence without queries or
    without keys get zero gradients; with grouped K/V heads, dK and dV of a
    K/V head sum over its group."""
    q, k, v, do = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(do)
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    H = q.shape[1]
    G = H // k.shape[1]
    for s in range(len(cu_q) - 1):
        q0, q1, k0, k1 = cu_q[s], cu_q[s + 1], cu_k[s], cu_k[s + 1]
        if q1 <= q0 or k1 <= k0:
            continue
        for h in range(H):
            qh, kh, vh, doh = q[q0:q1, h], k[k0:k1, h // G], v[k0:k1, h // G], do[q0:q1, h]
            P, _ = softmax_weights(qh, kh, scale)
            dv[k0:k1, h // G] += P.T @ doh
            dP = doh @ vh.T
            dS = P * (dP - (P * dP).sum(axis=1, keepdims=True))
            dq[q0:q1, h] = scale * (dS @ kh)
            dk[k0:k1, h // G] += scale * (dS.T @ qh)
    return dq, dk, dv


def gqa_forward(q, k, v, scale: float):
    """Grouped-query attention: q [B, H, Lq, d], k and v [B, H_kv, Lk, d] with
    H a multiple of H_kv; query head h attends with K/V head h // (H / H_kv).
    Returns (O [B, H, Lq, d], lse [B, H, Lq]) as float64 arrays."""
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    B, H, Lq, _ = q.shape
    G = H // k.shape[1]
    o = np.zeros((B, H, Lq, v.shape[3]))
    lse = np.zeros((B, H, Lq))
    for b, h in _heads(q):
        P, lse_h = softmax_weights(q[b, h], k[b, h // G], scale)
        o[b, h] = P @ v[b, h // G]
        lse[b, h] = lse_h
    return o, lse


def gqa_backward(q, k, v, do, scale: float):
    """Gradients (dQ, dK, dV) of sum(O * dO) for gqa_forward; dK and dV of a
    K/V head sum the contributions of every query head in its group."""
    q, k, v, do = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(do)
    G = q.shape[1] // k.shape[1]
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b, h in _heads(q):
        kh, vh = k[b, h // G], v[b, h // G]
        P, _ = softmax_weights(q[b, h], kh, scale)
        dv[b, h // G] += P.T @ do[b, h]
        dP = do[b, h] @ vh.T
        dS = P * (dP - (P * dP).sum(axis=1, keepdims=True))
        dq[b, h] = scale * (dS @ kh)
        dk[b, h // G] += scale * (dS.T @ q[b, h])
    return dq, dk, dv
