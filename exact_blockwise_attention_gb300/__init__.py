"""Exact blockwise attention for long video-token sequences on GB300 (sm_103a).

A thin Python binding over the C ABI of ``libattn.so`` (include/attn.h). Every
step of the computation runs in the library's CUDA kernels; this module only
checks tensors, allocates outputs with PyTorch (device memory and the current
stream are all PyTorch provides here) and passes raw pointers through ctypes.
There is no fallback: if the library is missing, importing the functions
raises.

Entry points (same names as the C ABI):
  fwd(q, k, v, scale=None)                      -> (o, lse)
  bwd(q, k, v, o, do, lse, scale=None)          -> (dq, dk, dv)
  partial_fwd(q, k, v, k0, k1, scale=None)      -> (o_part fp32, lse_part)
  split_fwd(q, k, v, bounds, scale=None)        -> (o_parts fp32, lse_parts)
  merge(o_parts, lse_parts)                     -> (o, lse)
  attention(q, k, v, scale=None)                -> o   (autograd-aware)
  attention_varlen(q, k, v, cu_q, cu_k, scale=None) -> o   (autograd-aware, packed)
  fwd_varlen(q, k, v, cu_q, cu_k, scale=None)   -> (o, lse)      packed sequences
  fwd_fp8(q8, k8, vt8, q_scale, k_scale, v_scale, scale=None) -> (o, lse)   e4m3, d = 128
  bwd_varlen(q, k, v, o, do, lse, cu_q, cu_k, scale=None) -> (dq, dk, dv)
Tensors are CUDA, contiguous, [B, H, L, d] with d in {64, 128}; q, k, v, o,
do are bfloat16, lse and partials float32. The default scale is 1/sqrt(d).
fwd, bwd and attention also take k, v with fewer heads H_kv dividing H
(grouped-query attention: query head h reads K/V head h // (H // H_kv);
attn_fwd_gqa / attn_bwd_gqa).
Packed sequences are token-major [T, H, d] with lse [H, Tq]; cu_q, cu_k are
host-side cumulative lengths (n_seqs + 1 ints, first 0).
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

from . import _build

__all__ = [
    "AttnError", "lib", "fwd", "bwd", "bwd_noalloc", "partial_fwd", "split_fwd", "merge", "attention",
    "bwd_workspace_size", "poll_device_status", "set_wait_limit_ns", "status_string",
    "MAX_CHUNKS", "MAX_SEQS", "fwd_varlen", "bwd_varlen", "bwd_varlen_workspace_size", "fwd_fp8",
    "attention_varlen",
]

ATTN_OK = 0
MAX_CHUNKS = 64
MAX_SEQS = 1024
_LIB = None


class AttnError(RuntimeError):
    """A non-zero status returned by the C ABI."""

    def __init__(self, fn: str, status: int):
        self.status = status
        msg = f"{fn} failed: {status_string(status)} (status {status})"
        if status == 4:
            self.cuda_error = int(lib().attn_last_cuda_error())
            msg += f", cudaError {self.cuda_error}"
        super().__init__(msg)


def _declare(L):
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    L.attn_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, vp]
    L.attn_bwd_workspace_size.argtypes = [i, i, i, i, i]
    L.attn_bwd_workspace_size.restype = sz
    L.attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, vp, sz, vp]
    L.attn_partial_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, vp]
    L.attn_split_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, ctypes.POINTER(i), i, f, vp]
    L.attn_merge.argtypes = [vp, vp, i, vp, vp, i, i, i, i, vp]
    L.attn_status_string.argtypes = [i]
    L.attn_status_string.restype = ctypes.c_char_p
    L.attn_poll_device_status.argtypes = [vp]
    L.attn_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, vp]
    L.attn_bwd_noalloc.restype = ctypes.c_int
    L.attn_last_cuda_error.argtypes = []
    L.attn_last_cuda_error.restype = ctypes.c_int
    L.attn_set_wait_limit_ns.argtypes = [ctypes.c_ulonglong]
    L.attn_set_wait_limit_ns.restype = ctypes.c_ulonglong
    L.attn_fwd_gqa.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, vp]
    L.attn_fwd_fp8.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, f, f, f, vp]
    L.attn_bwd_gqa.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, vp, sz,
                               vp]
    ip = ctypes.POINTER(i)
    L.attn_fwd_varlen.argtypes = [vp, vp, vp, vp, vp, ip, ip, i, i, i, f, vp]
    L.attn_bwd_varlen_workspace_size.argtypes = [i, i, i, i]
    L.attn_bwd_varlen_workspace_size.restype = sz
    L.attn_bwd_varlen.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, ip, ip, i, i, i, f, vp, sz,
                                  vp]
    L.attn_fwd_varlen_gqa.argtypes = [vp, vp, vp, vp, vp, ip, ip, i, i, i, i, f, vp]
    L.attn_bwd_varlen_gqa.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, ip, ip, i, i, i, i, f,
                                      vp, sz, vp]
    for name in ("attn_fwd", "attn_bwd", "attn_partial_fwd", "attn_split_fwd", "attn_merge",
                 "attn_poll_device_status", "attn_fwd_varlen", "attn_bwd_varlen", "attn_fwd_gqa",
                 "attn_bwd_gqa", "attn_fwd_fp8", "attn_fwd_varlen_gqa", "attn_bwd_varlen_gqa"):
        getattr(L, name).restype = ctypes.c_int
    return L


def lib():
    """The loaded libattn.so (raises if it has not been built)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(_build.LIB):
            raise ImportError(
                f"{_build.LIB} is missing: build it with "
                "`python -c 'import exact_blockwise_attention_gb300._build as b; b.build()'`")
        _LIB = _declare(ctypes.CDLL(_build.LIB))
    return _LIB


def status_string(status: int) -> str:
    return lib().attn_status_string(int(status)).decode()


def _check(fn: str, status: int):
    if status != ATTN_OK:
        raise AttnError(fn, status)


def _ptr(t: torch.Tensor) -> int:
    return t.data_ptr()


def _stream() -> int:
    return torch.cuda.current_stream().cuda_stream


def _require(t, name, dtype, ndim=4, device_type="cuda"):
    if not isinstance(t, torch.Tensor):
        raise ValueError(f"{name} must be a torch.Tensor")
    if t.device.type != device_type:
        raise ValueError(f"{name} must be a {device_type.upper()} tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {t.dim()}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _qkv(q, k, v, gqa=False, device_type="cuda"):
    for n, t in (("q", q), ("k", k), ("v", v)):
        _require(t, n, torch.bfloat16, device_type=device_type)
    B, H, Lq, d = q.shape
    Hkv = k.shape[1]
    heads_ok = Hkv == H or (gqa and Hkv >= 1 and H % Hkv == 0)
    if k.shape[0] != B or not heads_ok or k.shape[3] != d or v.shape != k.shape:
        raise ValueError(f"shape mismatch: q {tuple(q.shape)} k {tuple(k.shape)} v {tuple(v.shape)}")
    if not (q.device == k.device == v.device):
        raise ValueError("q, k, v must be on the same device")
    if gqa:
        return B, H, Hkv, Lq, k.shape[2], d
    return B, H, Lq, k.shape[2], d


def _scale(scale, d):
    return 1.0 / math.sqrt(d) if scale is None else float(scale)


def fwd(q, k, v, scale=None):
    """Exact attention forward: returns (o bf16 [B,H,Lq,d], lse fp32 [B,H,Lq]).
    k, v may have H_kv < H heads (grouped-query attention)."""
    B, H, Hkv, Lq, Lk, d = _qkv(q, k, v, gqa=True)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Lq), device=q.device, dtype=torch.float32)
    with torch.cuda.device(q.device):
        if Hkv == H:
            _check("attn_fwd", lib().attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H,
                                              Lq, Lk, d, _scale(scale, d), _stream()))
        else:
            _check("attn_fwd_gqa", lib().attn_fwd_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(o),
                                                      _ptr(lse), B, H, Hkv, Lq, Lk, d,
                                                      _scale(scale, d), _stream()))
    return o, lse


def bwd_workspace_size(B, H, Lq, Lk, d) -> int:
    return int(lib().attn_bwd_workspace_size(B, H, Lq, Lk, d))


def _bwd_inputs(q, k, v, o, do, lse, gqa, device_type="cuda"):
    """Checks shared by the backward entry points: q, k, v as for the forward,
    o and do shaped like q (bf16, contiguous, same device), lse [B, H, Lq] fp32."""
    dims = _qkv(q, k, v, gqa=gqa, device_type=device_type)
    B, H, Lq = q.shape[0], q.shape[1], q.shape[2]
    _require(o, "o", torch.bfloat16, device_type=device_type)
    _require(do, "do", torch.bfloat16, device_type=device_type)
    _require(lse, "lse", torch.float32, ndim=3, device_type=device_type)
    if o.shape != q.shape or do.shape != q.shape or lse.shape != (B, H, Lq):
        raise ValueError("o/do must match q and lse must be [B,H,Lq]")
    if not (o.device == do.device == lse.device == q.device):
        raise ValueError("o, do and lse must be on q's device")
    return dims


def _noalloc_out(q, k, v, out, device_type="cuda"):
    """The caller's (dq, dk, dv) for bwd_noalloc: bf16, contiguous, on q's
    device and shaped like q, k and v, so the kernels never write past them."""
    if not isinstance(out, (tuple, list)) or len(out) != 3:
        raise ValueError("out must be a (dq, dk, dv) tuple")
    for name, t, src, like in zip(("dq", "dk", "dv"), out, "qkv", (q, k, v)):
        _require(t, name, torch.bfloat16, device_type=device_type)
        if t.shape != like.shape or t.device != q.device:
            raise ValueError(f"{name} must be shaped like {src} {tuple(like.shape)} on {q.device}, "
                             f"got {tuple(t.shape)} on {t.device}")
    return tuple(out)


def bwd(q, k, v, o, do, lse, scale=None, workspace=None):
    """Gradients (dq, dk, dv) of sum(o * do); P is recomputed from lse. With
    grouped-query k, v (H_kv < H heads), dk and dv sum over each group."""
    B, H, Hkv, Lq, Lk, d = _bwd_inputs(q, k, v, o, do, lse, gqa=True)
    need = bwd_workspace_size(B, H, Lq, Lk, d)
    if workspace is None:
        workspace = torch.empty(need, device=q.device, dtype=torch.uint8)
    elif workspace.numel() * workspace.element_size() < need or not workspace.is_cuda:
        raise ValueError(f"workspace must be a CUDA tensor of at least {need} bytes")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ptrs = (_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv))
    with torch.cuda.device(q.device):
        if Hkv == H:
            _check("attn_bwd", lib().attn_bwd(*ptrs, B, H, Lq, Lk, d, _scale(scale, d),
                                              _ptr(workspace), need, _stream()))
        else:
            _check("attn_bwd_gqa", lib().attn_bwd_gqa(*ptrs, B, H, Hkv, Lq, Lk, d,
                                                      _scale(scale, d), _ptr(workspace), need,
                                                      _stream()))
    return dq, dk, dv


def bwd_noalloc(q, k, v, o, do, lse, scale=None, out=None):
    """bwd() for callers that cannot allocate device memory: the scratch comes
    from a 64 MiB buffer built into the library (see attn_bwd_noalloc in
    include/attn.h). Pass preallocated ``out=(dq, dk, dv)`` to allocate
    nothing at all from Python either; they are checked (bf16, contiguous,
    on q's device, shaped like q, k, v) before the library is called."""
    B, H, Lq, Lk, d = _bwd_inputs(q, k, v, o, do, lse, gqa=False)
    if out is None:
        out = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v))
    dq, dk, dv = _noalloc_out(q, k, v, out)
    with torch.cuda.device(q.device):
        _check("attn_bwd_noalloc", lib().attn_bwd_noalloc(
            _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv),
            B, H, Lq, Lk, d, _scale(scale, d), _stream()))
    return dq, dk, dv


def partial_fwd(q, k, v, k0, k1, scale=None):
    """Attention over keys [k0, k1): (o_part fp32 [B,H,Lq,d], lse_part fp32 [B,H,Lq])."""
    B, H, Lq, Lk, d = _qkv(q, k, v)
    o = torch.empty((B, H, Lq, d), device=q.device, dtype=torch.float32)
    lse = torch.empty((B, H, Lq), device=q.device, dtype=torch.float32)
    with torch.cuda.device(q.device):
        _check("attn_partial_fwd", lib().attn_partial_fwd(
            _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Lq, Lk, d, int(k0), int(k1),
            _scale(scale, d), _stream()))
    return o, lse


def split_fwd(q, k, v, bounds, scale=None):
    """Partial attention for every chunk [bounds[c], bounds[c+1]) in one launch."""
    B, H, Lq, Lk, d = _qkv(q, k, v)
    bounds = [int(b) for b in bounds]
    C = len(bounds) - 1
    if C < 1:
        raise ValueError("bounds needs at least two entries")
    arr = (ctypes.c_int * len(bounds))(*bounds)
    o = torch.empty((C, B, H, Lq, d), device=q.device, dtype=torch.float32)
    lse = torch.empty((C, B, H, Lq), device=q.device, dtype=torch.float32)
    with torch.cuda.device(q.device):
        _check("attn_split_fwd", lib().attn_split_fwd(
            _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Lq, Lk, d, arr, C,
            _scale(scale, d), _stream()))
    return o, lse


def merge(o_parts, lse_parts):
    """Exact merge of partials: (o bf16 [B,H,Lq,d], lse fp32 [B,H,Lq])."""
    _require(o_parts, "o_parts", torch.float32, ndim=5)
    _require(lse_parts, "lse_parts", torch.float32, ndim=4)
    C, B, H, Lq, d = o_parts.shape
    if lse_parts.shape != (C, B, H, Lq):
        raise ValueError("lse_parts must be [C,B,H,Lq] matching o_parts")
    o = torch.empty((B, H, Lq, d), device=o_parts.device, dtype=torch.bfloat16)
    lse = torch.empty((B, H, Lq), device=o_parts.device, dtype=torch.float32)
    with torch.cuda.device(o_parts.device):
        _check("attn_merge", lib().attn_merge(_ptr(o_parts), _ptr(lse_parts), C, _ptr(o),
                                              _ptr(lse), B, H, Lq, d, _stream()))
    return o, lse


def fwd_fp8(q8, k8, vt8, q_scale, k_scale, v_scale, scale=None):
    """Forward with e4m3 operands (d = 128): q8 [B,H,Lq,128], k8 [B,H,Lk,128] and
    vt8 = V transposed [B,H,128,Lk], torch.float8_e4m3fn, with per-tensor
    dequantisation scales (real value = stored value * scale). Returns
    (o bf16 [B,H,Lq,128], lse fp32 [B,H,Lq])."""
    f8 = getattr(torch, "float8_e4m3fn")
    for n, t in (("q8", q8), ("k8", k8), ("vt8", vt8)):
        _require(t, n, f8)
    B, H, Lq, d = q8.shape
    Lk = k8.shape[2]
    if k8.shape != (B, H, Lk, d) or vt8.shape != (B, H, d, Lk):
        raise ValueError(f"shape mismatch: q8 {tuple(q8.shape)} k8 {tuple(k8.shape)} "
                         f"vt8 {tuple(vt8.shape)} (vt8 is V transposed, [B,H,d,Lk])")
    o = torch.empty((B, H, Lq, d), device=q8.device, dtype=torch.bfloat16)
    lse = torch.empty((B, H, Lq), device=q8.device, dtype=torch.float32)
    with torch.cuda.device(q8.device):
        _check("attn_fwd_fp8", lib().attn_fwd_fp8(
            _ptr(q8), _ptr(k8), _ptr(vt8), _ptr(o), _ptr(lse), B, H, Lq, Lk, d, _scale(scale, d),
            float(q_scale), float(k_scale), float(v_scale), _stream()))
    return o, lse


def _cu(cu, name):
    """Host int array of cumulative lengths (a sequence of ints or a CPU tensor)."""
    if isinstance(cu, torch.Tensor):
        if cu.device.type != "cpu":
            raise ValueError(f"{name} must be on the host (cumulative lengths are read by the CPU)")
        cu = cu.tolist()
    vals = [int(x) for x in cu]
    if len(vals) < 2:
        raise ValueError(f"{name} needs at least two entries")
    return vals, (ctypes.c_int * len(vals))(*vals)


def _varlen_qkv(q, k, v, cu_q, cu_k):
    for n, t in (("q", q), ("k", k), ("v", v)):
        _require(t, n, torch.bfloat16, ndim=3)
    Tq, H, d = q.shape
    Hkv = k.shape[1]
    if k.shape[2] != d or not (Hkv >= 1 and H % Hkv == 0) or v.shape != k.shape:
        raise ValueError(f"shape mismatch: q {tuple(q.shape)} k {tuple(k.shape)} v {tuple(v.shape)}")
    cq, aq = _cu(cu_q, "cu_q")
    ck, ak = _cu(cu_k, "cu_k")
    if len(cq) != len(ck):
        raise ValueError("cu_q and cu_k must have the same length")
    if cq[-1] != Tq or ck[-1] != k.shape[0]:
        raise ValueError("cu_q[-1] / cu_k[-1] must equal the packed token counts")
    return Tq, H, Hkv, d, aq, ak, len(cq) - 1


def fwd_varlen(q, k, v, cu_q, cu_k, scale=None):
    """Exact attention within each packed sequence: (o bf16 [Tq,H,d], lse fp32 [H,Tq]).
    k, v may have H_kv < H heads (grouped-query attention)."""
    Tq, H, Hkv, d, aq, ak, n = _varlen_qkv(q, k, v, cu_q, cu_k)
    o = torch.empty_like(q)
    lse = torch.empty((H, Tq), device=q.device, dtype=torch.float32)
    with torch.cuda.device(q.device):
        _check("attn_fwd_varlen_gqa", lib().attn_fwd_varlen_gqa(
            _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), aq, ak, n, H, Hkv, d, _scale(scale, d),
            _stream()))
    return o, lse


def bwd_varlen_workspace_size(Tq, H, d, n_seqs) -> int:
    return int(lib().attn_bwd_varlen_workspace_size(Tq, H, d, n_seqs))


def bwd_varlen(q, k, v, o, do, lse, cu_q, cu_k, scale=None, workspace=None):
    """Gradients (dq, dk, dv) of sum(o * do) over packed sequences (dk, dv summed
    over each group of query heads when k, v have fewer heads)."""
    Tq, H, Hkv, d, aq, ak, n = _varlen_qkv(q, k, v, cu_q, cu_k)
    _require(o, "o", torch.bfloat16, ndim=3)
    _require(do, "do", torch.bfloat16, ndim=3)
    _require(lse, "lse", torch.float32, ndim=2)
    if o.shape != q.shape or do.shape != q.shape or lse.shape != (H, Tq):
        raise ValueError("o/do must match q and lse must be [H,Tq]")
    need = bwd_varlen_workspace_size(Tq, H, d, n)
    if workspace is None:
        workspace = torch.empty(max(need, 16), device=q.device, dtype=torch.uint8)
    elif workspace.numel() * workspace.element_size() < need or not workspace.is_cuda:
        raise ValueError(f"workspace must be a CUDA tensor of at least {need} bytes")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    with torch.cuda.device(q.device):
        _check("attn_bwd_varlen_gqa", lib().attn_bwd_varlen_gqa(
            _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv),
            aq, ak, n, H, Hkv, d, _scale(scale, d), _ptr(workspace), need, _stream()))
    return dq, dk, dv


def poll_device_status() -> int:
    """Synchronise the current stream; return the status word (0 ok, 5 a wait timed out)."""
    return int(lib().attn_poll_device_status(_stream()))


def set_wait_limit_ns(ns: int) -> int:
    return int(lib().attn_set_wait_limit_ns(int(ns)))


class _Attention(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, scale):
        o, lse = fwd(q, k, v, scale)
        ctx.save_for_backward(q, k, v, o, lse)
        ctx.scale = scale
        return o

    @staticmethod
    def backward(ctx, do):
        q, k, v, o, lse = ctx.saved_tensors
        dq, dk, dv = bwd(q, k, v, o, do.contiguous(), lse, ctx.scale)
        return dq, dk, dv, None


def attention(q, k, v, scale=None):
    """Autograd-aware exact attention; only o and lse are saved for backward."""
    return _Attention.apply(q, k, v, scale)


class _AttentionVarlen(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, cu_q, cu_k, scale):
        o, lse = fwd_varlen(q, k, v, cu_q, cu_k, scale)
        ctx.save_for_backward(q, k, v, o, lse)
        ctx.cu = (cu_q, cu_k)
        ctx.scale = scale
        return o

    @staticmethod
    def backward(ctx, do):
        q, k, v, o, lse = ctx.saved_tensors
        dq, dk, dv = bwd_varlen(q, k, v, o, do.contiguous(), lse, *ctx.cu, ctx.scale)
        return dq, dk, dv, None, None, None


def attention_varlen(q, k, v, cu_q, cu_k, scale=None):
    """Autograd-aware exact attention over packed sequences (token-major
    [T, H, d]; cu_q, cu_k host cumulative lengths)."""
    return _AttentionVarlen.apply(q, k, v, cu_q, cu_k, scale)
