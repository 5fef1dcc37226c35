"""Out-of-bounds writes and determinism, for every entry point.

Every output (and the backward workspace) is a view into a larger buffer whose
guard regions before and after it hold a sentinel; after the call the guards
must be unchanged byte for byte, so a kernel writing one element past (or
before) its output is caught even where that element would not affect parity.
The outputs that do not go through atomic adds (O, lse, dK, dV, partials,
merged O) must also be bit-identical across two runs.
"""
import ctypes
import math

import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu

GUARD = 4096  # elements of sentinel before and after each output (keeps 16-byte alignment)


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


class Guarded:
    """A tensor of `shape` inside a buffer with sentinel guards on both sides."""

    def __init__(self, shape, dtype, fill=float("nan")):
        n = math.prod(shape)
        self.buf = torch.empty(n + 2 * GUARD, device="cuda", dtype=dtype)
        self.buf.view(torch.uint8).fill_(0xA5)  # sentinel bytes
        self.t = self.buf[GUARD:GUARD + n].view(shape)
        self.t.fill_(fill)
        self.before = self.buf[:GUARD].clone()
        self.after = self.buf[GUARD + n:].clone()

    def check(self, name):
        torch.cuda.synchronize()
        n = self.t.numel()
        assert torch.equal(self.buf[:GUARD].view(torch.uint8), self.before.view(torch.uint8)), \
            f"{name}: write before the output"
        assert torch.equal(self.buf[GUARD + n:].view(torch.uint8), self.after.view(torch.uint8)), \
            f"{name}: write past the output"


def _stream():
    return torch.cuda.current_stream().cuda_stream


def _dense(eba, B, H, Lq, Lk, d, Hkv=None, seed=0):
    """attn_fwd(_gqa) + attn_bwd(_gqa) into guarded outputs; returns the outputs."""
    Hkv = Hkv or H
    q, _, _, do = W.make_inputs(W.TINY, seed=seed, B=B, H=H, Lq=Lq, Lk=Lk, d=d)
    _, k, v, _ = W.make_inputs(W.TINY, seed=seed + 1, B=B, H=Hkv, Lq=Lq, Lk=Lk, d=d)
    q, k, v, do = (x.cuda() for x in (q, k, v, do))
    L = eba.lib()
    scale = 1.0 / math.sqrt(d)
    o = Guarded((B, H, Lq, d), torch.bfloat16)
    lse = Guarded((B, H, Lq), torch.float32)
    dq = Guarded((B, H, Lq, d), torch.bfloat16)
    dk = Guarded((B, Hkv, Lk, d), torch.bfloat16)
    dv = Guarded((B, Hkv, Lk, d), torch.bfloat16)
    need = L.attn_bwd_workspace_size(B, H, Lq, Lk, d)
    ws = Guarded((need,), torch.uint8, fill=0)
    ptrs = (q.data_ptr(), k.data_ptr(), v.data_ptr())
    if Hkv == H:
        assert L.attn_fwd(*ptrs, o.t.data_ptr(), lse.t.data_ptr(), B, H, Lq, Lk, d, scale,
                          _stream()) == 0
        assert L.attn_bwd(*ptrs, o.t.data_ptr(), do.data_ptr(), lse.t.data_ptr(), dq.t.data_ptr(),
                          dk.t.data_ptr(), dv.t.data_ptr(), B, H, Lq, Lk, d, scale,
                          ws.t.data_ptr(), need, _stream()) == 0
    else:
        assert L.attn_fwd_gqa(*ptrs, o.t.data_ptr(), lse.t.data_ptr(), B, H, Hkv, Lq, Lk, d, scale,
                              _stream()) == 0
        assert L.attn_bwd_gqa(*ptrs, o.t.data_ptr(), do.data_ptr(), lse.t.data_ptr(),
                              dq.t.data_ptr(), dk.t.data_ptr(), dv.t.data_ptr(), B, H, Hkv, Lq, Lk,
                              d, scale, ws.t.data_ptr(), need, _stream()) == 0
    for g, n in ((o, "o"), (lse, "lse"), (dq, "dq"), (dk, "dk"), (dv, "dv"), (ws, "workspace")):
        g.check(n)
    return o.t.clone(), lse.t.clone(), dk.t.clone(), dv.t.clone()


SHAPES = [
    # B, H, Lq, Lk, d, H_kv
    (2, 3, 200, 333, 64, None),     # ragged tiles
    (1, 2, 1, 1, 64, None),         # single tokens (packed tiles)
    (3, 5, 7, 7, 64, None),         # packed tiles, partial last tile
    (2, 2, 300, 513, 128, None),
    (1, 4, 150, 260, 64, 2),        # grouped-query
    (3, 4, 30, 50, 128, None),      # packed, Lq != Lk
]


@pytest.mark.parametrize("B,H,Lq,Lk,d,Hkv", SHAPES, ids=lambda x: str(x))
def test_dense_guards_and_determinism(eba, B, H, Lq, Lk, d, Hkv):
    a = _dense(eba, B, H, Lq, Lk, d, Hkv, seed=B * 100 + Lq)
    b = _dense(eba, B, H, Lq, Lk, d, Hkv, seed=B * 100 + Lq)
    for x, y, n in zip(a, b, ("o", "lse", "dk", "dv")):
        assert torch.equal(x, y), f"{n} differs between two runs"


def test_varlen_guards_and_determinism(eba):
    lq, lk = [100, 0, 300, 129, 1], [50, 70, 0, 400, 1]
    cu_q, cu_k = [0], [0]
    for a, b in zip(lq, lk):
        cu_q.append(cu_q[-1] + a)
        cu_k.append(cu_k[-1] + b)
    H, d = 2, 64
    q, k, v, do = (x.cuda() for x in W.make_varlen_inputs(cu_q[-1], cu_k[-1], H, d, seed=3))
    aq = (ctypes.c_int * len(cu_q))(*cu_q)
    ak = (ctypes.c_int * len(cu_k))(*cu_k)
    n = len(cu_q) - 1
    L = eba.lib()
    runs = []
    for _ in range(2):
        o = Guarded(tuple(q.shape), torch.bfloat16)
        lse = Guarded((H, cu_q[-1]), torch.float32)
        dq = Guarded(tuple(q.shape), torch.bfloat16)
        dk = Guarded(tuple(k.shape), torch.bfloat16)
        dv = Guarded(tuple(v.shape), torch.bfloat16)
        need = L.attn_bwd_varlen_workspace_size(cu_q[-1], H, d, n)
        ws = Guarded((need,), torch.uint8, fill=0)
        assert L.attn_fwd_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.t.data_ptr(),
                                 lse.t.data_ptr(), aq, ak, n, H, d, 0.125, _stream()) == 0
        assert L.attn_bwd_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.t.data_ptr(),
                                 do.data_ptr(), lse.t.data_ptr(), dq.t.data_ptr(), dk.t.data_ptr(),
                                 dv.t.data_ptr(), aq, ak, n, H, d, 0.125, ws.t.data_ptr(), need,
                                 _stream()) == 0
        for g, nm in ((o, "o"), (lse, "lse"), (dq, "dq"), (dk, "dk"), (dv, "dv"), (ws, "workspace")):
            g.check(nm)
        runs.append((o.t.clone(), lse.t.clone(), dk.t.clone(), dv.t.clone()))
    for x, y in zip(*runs):
        assert torch.equal(x, y)


def test_split_merge_guards_and_determinism(eba):
    B, H, Lq, Lk, d = 2, 3, 130, 700, 128
    q, k, v, _ = (x.cuda() for x in W.make_inputs(W.TINY, seed=5, B=B, H=H, Lq=Lq, Lk=Lk, d=d))
    bounds = [0, 100, 100, 350, 700]
    C = len(bounds) - 1
    arr = (ctypes.c_int * len(bounds))(*bounds)
    L = eba.lib()
    runs = []
    for _ in range(2):
        op = Guarded((C, B, H, Lq, d), torch.float32)
        lp = Guarded((C, B, H, Lq), torch.float32)
        o = Guarded((B, H, Lq, d), torch.bfloat16)
        lse = Guarded((B, H, Lq), torch.float32)
        assert L.attn_split_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), op.t.data_ptr(),
                                lp.t.data_ptr(), B, H, Lq, Lk, d, arr, C, 0.088, _stream()) == 0
        assert L.attn_merge(op.t.data_ptr(), lp.t.data_ptr(), C, o.t.data_ptr(), lse.t.data_ptr(),
                            B, H, Lq, d, _stream()) == 0
        for g, nm in ((op, "o_parts"), (lp, "lse_parts"), (o, "o"), (lse, "lse")):
            g.check(nm)
        runs.append((op.t.clone(), lp.t.clone(), o.t.clone(), lse.t.clone()))
    for x, y in zip(*runs):
        assert torch.equal(x, y)


def test_fp8_guards_and_determinism(eba):
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("this torch has no float8_e4m3fn")
    B, H, Lq, Lk, d = 1, 2, 200, 336, 128
    q, k, v, _ = W.make_inputs(W.TINY, seed=7, B=B, H=H, Lq=Lq, Lk=Lk, d=d)
    f8 = [(x.float() / (float(x.float().abs().max()) / 448.0)).to(torch.float8_e4m3fn).cuda()
          for x in (q, k, v)]
    vt8 = f8[2].transpose(-1, -2).contiguous()
    L = eba.lib()
    runs = []
    for _ in range(2):
        o = Guarded((B, H, Lq, d), torch.bfloat16)
        lse = Guarded((B, H, Lq), torch.float32)
        assert L.attn_fwd_fp8(f8[0].data_ptr(), f8[1].data_ptr(), vt8.data_ptr(), o.t.data_ptr(),
                              lse.t.data_ptr(), B, H, Lq, Lk, d, 0.088, 0.01, 0.01, 0.01,
                              _stream()) == 0
        o.check("o")
        lse.check("lse")
        runs.append((o.t.clone(), lse.t.clone()))
    for x, y in zip(*runs):
        assert torch.equal(x, y)
