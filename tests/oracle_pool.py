"""The float64 oracle over many heads at once, in worker processes (test
infrastructure only).

Checking every head of a full-size workload against the oracle takes one
float64 forward and backward per head (about 50 ms each at 1568 tokens). The
heads are independent, so they are spread over a pool of worker processes,
each running the oracle single-threaded. The pool is started with ``spawn``:
the parent process already holds a CUDA context, and a forked child of such a
process can hang.

Inputs and GPU outputs are handed over as .npy files that each worker maps
read-only (bf16 tensors as their raw 16-bit patterns), so nothing large goes
through pipes. Each worker returns, per head, the largest absolute difference
between the GPU output and the oracle for each output tensor; the caller
decides what to accept.
"""
from __future__ import annotations

import multiprocessing as mp
import os

import numpy as np

_ARR: dict = {}
_THREAD_VARS = ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")


def _to_numpy(t) -> np.ndarray:
    """CPU copy of a torch tensor: bf16 as its uint16 bit patterns, float32 as is."""
    import torch

    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def _f64(a: np.ndarray) -> np.ndarray:
    """Exact float64 value of a uint16 bf16 pattern array (or of a float array)."""
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return np.asarray(a, dtype=np.float64)


def _init(paths: dict) -> None:
    for name, p in paths.items():
        _ARR[name] = np.load(p, mmap_mode="r")


def _head_errors(job):
    b, h, scale, bwd, model = job
    import oracle  # the worker's own import; the parent's is not shared

    def head(name):
        return _f64(np.asarray(_ARR[name][b:b + 1, h:h + 1]))

    q, k, v = head("q"), head("k"), head("v")
    ro, rl = oracle.forward(q, k, v, scale)
    errs = {"o": float(np.abs(head("o") - ro).max()), "lse": float(np.abs(head("lse") - rl).max())}
    if bwd:
        rdq, rdk, rdv = oracle.backward(q, k, v, head("do"), scale)
        errs["dq"] = float(np.abs(head("dq") - rdq).max())
        errs["dk"] = float(np.abs(head("dk") - rdk).max())
        errs["dv"] = float(np.abs(head("dv") - rdv).max())
    for name in ("o", "dq", "dk", "dv"):
        if name in errs and not np.isfinite(head(name)).all():
            errs[name] = float("inf")  # an unwritten (NaN-prefilled) element
    if bwd:
        # elements above the flat 2e-2, and, for outputs held to the rounding
        # model instead (inputs outside the unit-variance regime), how many
        # exceed its limit and the largest error / limit
        import rounding_model as rm

        refs = {"dq": rdq, "dk": rdk, "dv": rdv}
        errs.update({f"{n}_n_over_flat": int((np.abs(head(n) - r) > 2e-2).sum())
                     for n, r in refs.items()})
        if model:
            _, bq, bk, bv = rm.head_bounds(q[0, 0], k[0, 0], v[0, 0], head("do")[0, 0], scale)
            for n, R in (("dq", bq), ("dk", bk), ("dv", bv)):
                err = np.abs(head(n)[0, 0] - refs[n][0, 0])
                lim = rm.model_limit(refs[n][0, 0], R)
                errs[f"{n}_n_over_model"] = int((err > lim).sum())
                errs[f"{n}_over_limit"] = float((err / lim).max())
    return b, h, errs


def head_errors(tensors: dict, heads, scale: float, bwd: bool, workdir: str, workers=None,
                model=False):
    """Per-head max-abs errors of GPU outputs against the float64 oracle.

    tensors: q, k, v, o, lse (and do, dq, dk, dv when bwd) as [B, H, ...]
    tensors (any device); heads: (b, h) pairs; workers: pool size (default:
    one per host core); model: also evaluate, per element, the bf16 rounding
    model of rounding_model.py (the bound used for inputs outside the
    unit-variance regime). Returns {(b, h): {name: err}} (plus counts, see
    _head_errors)."""
    paths = {}
    for name, t in tensors.items():
        p = os.path.join(workdir, f"{name}.npy")
        np.save(p, _to_numpy(t))
        paths[name] = p
    jobs = [(b, h, float(scale), bool(bwd), bool(model)) for b, h in heads]
    n = max(1, min(len(jobs), workers or os.cpu_count() or 1))
    ctx = mp.get_context("spawn")
    saved = {v: os.environ.get(v) for v in _THREAD_VARS}
    for var in _THREAD_VARS:  # one BLAS thread per worker; the pool gives the parallelism
        os.environ[var] = "1"
    try:
        pool = ctx.Pool(n, initializer=_init, initargs=(paths,))
    finally:
        for var, val in saved.items():
            if val is None:
                os.environ.pop(var, None)
            else:
                os.environ[var] = val
    with pool:
        out = pool.map(_head_errors, jobs, chunksize=max(1, len(jobs) // (4 * n)))
    return {(b, h): e for b, h, e in out}


def worst(per_head: dict) -> dict:
    """Largest value of each entry over all heads, with the head it came from
    (counts: their total over the heads)."""
    res = {}
    for bh, errs in per_head.items():
        for name, e in errs.items():
            if name.endswith(("_n_over_flat", "_n_over_model")):
                res[name] = res.get(name, 0) + e
            elif name not in res or e > res[name][0]:
                res[name] = (e, bh)
    return res
