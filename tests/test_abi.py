"""The C ABI without a GPU: the library builds and loads, exports every entry
point include/*.h declares, and rejects invalid arguments before touching CUDA.
"""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w\s\*]*?\b(attn_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return sorted(names)


@pytest.fixture(scope="module")
def L():
    from exact_blockwise_attention_gb300 import _build

    _build.build()
    import exact_blockwise_attention_gb300 as eba

    return eba.lib()


def test_header_declares_the_boundary():
    names = _declared_functions()
    for required in ("attn_fwd", "attn_bwd", "attn_partial_fwd", "attn_merge"):
        assert required in names


def test_every_declared_symbol_is_exported(L):
    for name in _declared_functions():
        assert hasattr(L, name), name
        assert ctypes.cast(getattr(L, name), ctypes.c_void_p).value


def test_status_strings(L):
    import exact_blockwise_attention_gb300 as eba

    for code in range(0, 7):
        s = eba.status_string(code)
        assert s and s != "unknown status"
    assert eba.status_string(99) == "unknown status"


def test_wait_limit_is_kept_positive_as_signed(L):
    # The kernels compare elapsed timer nanoseconds as signed 64-bit values,
    # so a limit above 2^62 is stored as 2^62; 0 restores the 2 s default.
    f = L.attn_set_wait_limit_ns
    f.argtypes = [ctypes.c_ulonglong]
    f.restype = ctypes.c_ulonglong
    old = f(2**64 - 1)
    try:
        assert f(2**63) == 2**62
        assert f(12345) == 2**62
        assert f(0) == 12345
        assert f(0) == 2_000_000_000
    finally:
        f(old)


def test_workspace_size_is_linear_in_length(L):
    import exact_blockwise_attention_gb300 as eba

    # dQ fp32 accumulator + two padded fp32 row vectors; never O(Lq * Lk).
    B, H, d = 16, 16, 64
    for Lq in (128, 1568, 12544):
        pad = -(-Lq // 128) * 128
        assert eba.bwd_workspace_size(B, H, Lq, Lq, d) == B * H * (Lq * d * 4 + 2 * pad * 4)
    assert eba.bwd_workspace_size(1, 1, 100, 100, 96) == 0
    assert eba.bwd_workspace_size(0, 1, 100, 100, 64) == 0


A16 = 1 << 20        # a fake, 16-byte aligned address; never dereferenced
MIS = (1 << 20) + 8  # a fake misaligned address; never dereferenced


@pytest.mark.parametrize(
    "args,code",
    [
        # (q, k, v, o, lse, B, H, Lq, Lk, d, scale)
        ((0, A16, A16, A16, A16, 1, 1, 8, 8, 64, 0.125), 1),
        ((A16, A16, A16, A16, A16, 1, 1, 8, 8, 96, 0.125), 2),
        ((A16, A16, A16, A16, A16, 1, 1, 0, 8, 64, 0.125), 1),
        ((A16, A16, A16, A16, A16, 1, 1, 8, 0, 64, 0.125), 1),
        ((A16, A16, A16, A16, A16, 0, 1, 8, 8, 64, 0.125), 1),
        ((A16, A16, A16, A16, A16, 1, 1, 8, 8, 64, float("nan")), 1),
        ((A16, A16, A16, A16, A16, 1, 1, 8, 8, 64, float("inf")), 1),
        ((A16, A16, A16, A16, A16, 1, 1, 8, 8, 64, 0.0), 1),
        ((A16, A16, A16, A16, A16, 1, 1, 8, 8, 64, -0.125), 1),
        ((MIS, A16, A16, A16, A16, 1, 1, 8, 8, 64, 0.125), 3),
        ((A16, A16, A16, A16, MIS, 1, 1, 8, 8, 64, 0.125), 3),
    ],
)
def test_fwd_rejects_bad_arguments(L, args, code):
    assert L.attn_fwd(*args, None) == code


def test_partial_rejects_bad_ranges(L):
    base = (A16, A16, A16, A16, A16, 1, 1, 8, 10, 64)
    assert L.attn_partial_fwd(*base, -1, 5, 0.125, None) == 1
    assert L.attn_partial_fwd(*base, 6, 5, 0.125, None) == 1
    assert L.attn_partial_fwd(*base, 0, 11, 0.125, None) == 1


def test_split_rejects_bad_bounds(L):
    def call(bounds, n):
        arr = (ctypes.c_int * len(bounds))(*bounds)
        return L.attn_split_fwd(A16, A16, A16, A16, A16, 1, 1, 8, 10, 64, arr, n, 0.125, None)

    assert call([0, 5, 9], 2) == 1            # does not end at Lk
    assert call([1, 5, 10], 2) == 1           # does not start at 0
    assert call([0, 6, 5, 10], 3) == 1        # decreasing
    assert call([0, 10], 0) == 1              # no chunk
    assert call(list(range(0, 66)) + [10], 66) == 2  # too many chunks
    assert L.attn_split_fwd(A16, A16, A16, A16, A16, 1, 1, 8, 10, 64, None, 1, 0.125, None) == 1


def test_bwd_rejects_missing_workspace(L):
    args = [A16] * 9 + [1, 1, 8, 8, 64, 0.125]
    assert L.attn_bwd(*args, None, 0, None) == 6
    need = L.attn_bwd_workspace_size(1, 1, 8, 8, 64)
    assert L.attn_bwd(*args, A16, need - 4, None) == 6
    assert L.attn_bwd(*args, MIS, need, None) == 3
    bad = list(args)
    bad[5] = 0   # lse null
    assert L.attn_bwd(*bad, A16, need, None) == 1


def test_merge_rejects_bad_arguments(L):
    assert L.attn_merge(A16, A16, 0, A16, A16, 1, 1, 8, 64, None) == 1
    assert L.attn_merge(A16, A16, 2, A16, A16, 1, 1, 8, 32, None) == 2
    assert L.attn_merge(A16, MIS, 2, A16, A16, 1, 1, 8, 64, None) == 3


def test_python_binding_rejects_cpu_tensors():
    import torch

    import exact_blockwise_attention_gb300 as eba

    x = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        eba.fwd(x, x, x)
    with pytest.raises(ValueError):
        eba.merge(torch.zeros(2, 1, 1, 8, 64), torch.zeros(2, 1, 1, 8))


def _ints(xs):
    return (ctypes.c_int * len(xs))(*xs)


def test_varlen_rejects_bad_offsets(L):
    def fwd(cu_q, cu_k, n, H=2, d=64, scale=0.125, ptrs=(A16,) * 5):
        q = _ints(cu_q) if cu_q is not None else None
        k = _ints(cu_k) if cu_k is not None else None
        return L.attn_fwd_varlen(*ptrs, q, k, n, H, d, scale, None)

    assert fwd([0, 5, 9], [0, 4, 8], 0) == 1           # no sequence
    assert fwd(None, [0, 4, 8], 2) == 1                # missing offsets
    assert fwd([1, 5, 9], [0, 4, 8], 2) == 1           # does not start at 0
    assert fwd([0, 5, 4], [0, 4, 8], 2) == 1           # decreasing
    assert fwd([0, 5, 9], [0, 9, 8], 2) == 1
    assert fwd([0, 0, 0], [0, 4, 8], 2) == 1           # no query at all
    assert fwd([0, 5, 9], [0, 0, 0], 2) == 1           # no key at all
    assert fwd([0, 5, 9], [0, 4, 8], 2, H=0) == 1
    assert fwd([0, 5, 9], [0, 4, 8], 2, d=96) == 2
    assert fwd([0, 5, 9], [0, 4, 8], 2, scale=float("nan")) == 1
    assert fwd(list(range(1026)), list(range(1026)), 1025) == 2   # over ATTN_MAX_SEQS
    assert fwd([0, 5, 9], [0, 4, 8], 2, ptrs=(A16, A16, A16, MIS, A16)) == 3
    assert fwd([0, 5, 9], [0, 4, 8], 2, ptrs=(A16, 0, A16, A16, A16)) == 1


def test_varlen_bwd_workspace(L):
    # dQ accumulator [Tq, H, d] fp32 + two fp32 values per (head, padded row),
    # at most Tq + 128 * n_seqs rows.
    Tq, H, d, n = 1000, 4, 64, 3
    need = L.attn_bwd_varlen_workspace_size(Tq, H, d, n)
    assert need == Tq * H * d * 4 + 2 * H * (Tq + 128 * n) * 4
    assert L.attn_bwd_varlen_workspace_size(Tq, H, 96, n) == 0
    assert L.attn_bwd_varlen_workspace_size(Tq, H, d, 0) == 0
    assert L.attn_bwd_varlen_workspace_size(Tq, H, d, 1025) == 0
    cu_q, cu_k = _ints([0, 600, 600, 1000]), _ints([0, 300, 700, 700])
    args = [A16] * 9
    assert L.attn_bwd_varlen(*args, cu_q, cu_k, n, H, d, 0.125, None, 0, None) == 6
    assert L.attn_bwd_varlen(*args, cu_q, cu_k, n, H, d, 0.125, A16, need - 4, None) == 6
    assert L.attn_bwd_varlen(*args, cu_q, cu_k, n, H, d, 0.125, MIS, need, None) == 3


def test_gqa_rejects_bad_groups(L):
    # (q, k, v, o, lse, B, H, H_kv, Lq, Lk, d, scale)
    base = [A16] * 5
    assert L.attn_fwd_gqa(*base, 1, 6, 4, 8, 8, 64, 0.125, None) == 1   # 4 does not divide 6
    assert L.attn_fwd_gqa(*base, 1, 6, 0, 8, 8, 64, 0.125, None) == 1
    assert L.attn_fwd_gqa(*base, 1, 6, 3, 8, 8, 96, 0.125, None) == 2
    args = [A16] * 9
    need = L.attn_bwd_workspace_size(1, 6, 8, 8, 64)
    assert L.attn_bwd_gqa(*args, 1, 6, 4, 8, 8, 64, 0.125, A16, need, None) == 1
    assert L.attn_bwd_gqa(*args, 1, 6, 3, 8, 8, 64, 0.125, A16, need - 4, None) == 6


def test_fp8_rejects_bad_arguments(L):
    # (q8, k8, vt8, o, lse, B, H, Lq, Lk, d, scale, q_scale, k_scale, v_scale)
    p5 = [A16] * 5
    assert L.attn_fwd_fp8(*p5, 1, 1, 8, 16, 64, 0.1, 1.0, 1.0, 1.0, None) == 2    # d != 128
    assert L.attn_fwd_fp8(*p5, 1, 1, 8, 20, 128, 0.1, 1.0, 1.0, 1.0, None) == 3   # Lk % 16
    assert L.attn_fwd_fp8(*p5, 1, 1, 8, 16, 128, 0.1, 0.0, 1.0, 1.0, None) == 1   # scale 0
    assert L.attn_fwd_fp8(*p5, 1, 1, 8, 16, 128, 0.1, 1.0, float("nan"), 1.0, None) == 1
    assert L.attn_fwd_fp8(0, A16, A16, A16, A16, 1, 1, 8, 16, 128, 0.1, 1.0, 1.0, 1.0, None) == 1



def test_varlen_gqa_rejects_bad_groups(L):
    cu_q, cu_k = _ints([0, 5, 9]), _ints([0, 4, 8])
    p5 = [A16] * 5
    assert L.attn_fwd_varlen_gqa(*p5, cu_q, cu_k, 2, 6, 4, 64, 0.125, None) == 1   # 4 does not divide 6
    assert L.attn_fwd_varlen_gqa(*p5, cu_q, cu_k, 2, 6, 0, 64, 0.125, None) == 1
    need = L.attn_bwd_varlen_workspace_size(9, 6, 64, 2)
    args = [A16] * 9
    assert L.attn_bwd_varlen_gqa(*args, cu_q, cu_k, 2, 6, 4, 64, 0.125, A16, need, None) == 1


def test_binding_fails_loudly_without_the_library(monkeypatch, tmp_path):
    # No fallback: with the shared library absent, every entry point raises.
    import exact_blockwise_attention_gb300 as eba
    from exact_blockwise_attention_gb300 import _build

    monkeypatch.setattr(_build, "LIB", str(tmp_path / "missing_libattn.so"))
    monkeypatch.setattr(eba, "_LIB", None)
    with pytest.raises(ImportError):
        eba.lib()
    with pytest.raises(ImportError):
        eba.status_string(0)


def test_bwd_noalloc_checks_out_tensors_before_calling_the_library(monkeypatch):
    # A wrong-sized, wrong-dtype or non-contiguous out tensor, or o / do / lse
    # not matching q, must raise ValueError before anything reaches the C ABI
    # (the kernels would write past a too-small dq, dk or dv).
    import torch

    import exact_blockwise_attention_gb300 as eba

    def no_library():
        raise AssertionError("the library was called")

    monkeypatch.setattr(eba, "lib", no_library)
    B, H, L, d = 1, 2, 16, 64
    q, k, v, o, do = (torch.zeros(B, H, L, d, dtype=torch.bfloat16) for _ in range(5))
    lse = torch.zeros(B, H, L)
    good = (torch.zeros_like(q), torch.zeros_like(k), torch.zeros_like(v))
    cpu = dict(device_type="cpu")
    eba._bwd_inputs(q, k, v, o, do, lse, gqa=False, **cpu)
    eba._noalloc_out(q, k, v, good, **cpu)
    bad_outs = [
        (torch.zeros(B, H, L - 1, d, dtype=torch.bfloat16), good[1], good[2]),  # dq too small
        (good[0], torch.zeros(B, H, L, d), good[2]),                            # dk fp32
        (good[0], good[1], torch.zeros(B, H, d, L, dtype=torch.bfloat16).transpose(2, 3)),
        (good[0], good[1]),                                                      # two tensors
    ]
    for out in bad_outs:
        with pytest.raises(ValueError):
            eba._noalloc_out(q, k, v, out, **cpu)
    with pytest.raises(ValueError):
        eba._bwd_inputs(q, k, v, o[:, :, :8], do, lse, gqa=False, **cpu)
    with pytest.raises(ValueError):
        eba._bwd_inputs(q, k, v, o, do, lse[:, :1], gqa=False, **cpu)
    # The public entry point refuses CPU tensors the same way, library untouched.
    with pytest.raises(ValueError):
        eba.bwd_noalloc(q, k, v, o, do, lse, out=good)
