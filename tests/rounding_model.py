"""Size of the bf16 roundings the method itself makes, per output element,
computed from float64 oracle quantities only (test infrastructure).

Used where inputs lie outside the unit-variance regime the flat 2e-2 bar is
stated for: there the method's own roundings (P and dS rounded to bf16 as
tensor-core operands, D taken from the stored bf16 O, bf16 outputs) add up
over many terms and can exceed 2e-2 even for an implementation that makes no
other error. Each rounding is at most u = 2^-9 relative and the roundings are
independent, so terms summed over an index add in quadrature:
  O:   bf16 P in P V, sqrt(sum_j P_j^2 (v_j - O)^2) u, plus u |O| (output)
  D = rowsum(dO * O) from the stored bf16 O:  eD_i = sqrt(sum_c (dO_ic eO_ic)^2)
  dS = P (dP - D), rounded to bf16 for the dQ, dK products: w_ij^2 =
       (P_ij eD_i)^2 + (u dS_ij)^2
  dQ_ic = s sqrt(sum_j w_ij^2 K_jc^2) + u |dQ_ic|
  dK_jc = s sqrt(sum_i w_ij^2 Q_ic^2) + u |dK_jc|
  dV_jc = u sqrt(sum_i P_ij^2 dO_ic^2) + u |dV_jc|
The tests accept an element within max(2e-2 relative, 8 R + 1e-3): a CPU model
of exactly these roundings reproduces the kernels' largest errors to two
digits and stays below 3.2 R, measured GPU errors stay below 4 R, and the
factor 8 covers what the model leaves out (fp32 accumulation order, the
exponential's approximation).
"""
import numpy as np


U = 2.0 ** -9  # bf16 unit roundoff


def head_bounds(q, k, v, do, s):
    """Rounding sizes R of (O, dQ, dK, dV) for one head: q, do [Lq, d], k, v
    [Lk, d] float64."""
    S = s * (q @ k.T)
    P = np.exp(S - S.max(axis=1, keepdims=True))
    P /= P.sum(axis=1, keepdims=True)
    O = P @ v
    dP = do @ v.T
    dS = P * (dP - (P * dP).sum(axis=1, keepdims=True))
    P2 = P ** 2  # sum_j P_j^2 (v_j - O)^2, expanded into matrix products
    var = P2 @ v ** 2 - 2.0 * O * (P2 @ v) + O ** 2 * P2.sum(axis=1, keepdims=True)
    eO = U * np.sqrt(np.maximum(var, 0.0)) + U * np.abs(O)
    eD = np.sqrt(((do * eO) ** 2).sum(axis=1))  # [Lq]
    w2 = (P * eD[:, None]) ** 2 + (U * dS) ** 2  # [Lq, Lk]
    bq = s * np.sqrt(w2 @ k ** 2) + U * np.abs(s * dS @ k)
    bk = s * np.sqrt(w2.T @ q ** 2) + U * np.abs(s * dS.T @ q)
    bv = U * np.sqrt((P ** 2).T @ do ** 2) + U * np.abs(P.T @ do)
    return eO, bq, bk, bv


def model_limit(ref, R, tol=2e-2):
    """Per-element acceptance limit outside the flat-bar regime."""
    return np.maximum(tol * np.maximum(1.0, np.abs(ref)), 8.0 * R + 1e-3)
