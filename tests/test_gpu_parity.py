"""CUDA path against the float64 CPU oracle, element by element, through the C ABI.

Tolerances (stated for unit-variance bf16 inputs with fp32 accumulation):
max |GPU - oracle| <= 2e-2 on O, dQ, dK, dV and <= 1e-3 on lse. Inputs are
seeded bf16 tensors from workloads.py; the oracle sees the same bf16 values
upcast exactly to float64.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
import oracle_pool
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
    """Every test must leave the device status word clean: a bounded in-kernel
    wait that ran out (even one whose outputs happened to be right) fails it."""
    eba.poll_device_status()
    yield
    assert eba.poll_device_status() == 0, "a bounded in-kernel wait gave up"


def _nan(shape, dtype):
    return torch.full(shape, float("nan"), device="cuda", dtype=dtype)


def run_fwd(eba, q, k, v, scale):
    """attn_fwd through the C ABI into NaN-prefilled outputs."""
    B, H, Lq, d = q.shape
    Lk = k.shape[2]
    o = _nan((B, H, Lq, d), torch.bfloat16)
    lse = _nan((B, H, Lq), torch.float32)
    st = eba.lib().attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                            lse.data_ptr(), B, H, Lq, Lk, d, scale,
                            torch.cuda.current_stream().cuda_stream)
    assert st == 0, eba.status_string(st)
    return o, lse


def run_bwd(eba, q, k, v, o, do, lse, scale):
    B, H, Lq, d = q.shape
    Lk = k.shape[2]
    dq, dk, dv = _nan(q.shape, torch.bfloat16), _nan(k.shape, torch.bfloat16), _nan(v.shape, torch.bfloat16)
    need = eba.bwd_workspace_size(B, H, Lq, Lk, d)
    ws = torch.full((need // 4,), float("nan"), device="cuda", dtype=torch.float32)
    st = eba.lib().attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(),
                            lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, Lq,
                            Lk, d, scale, ws.data_ptr(), need,
                            torch.cuda.current_stream().cuda_stream)
    assert st == 0, eba.status_string(st)
    return dq, dk, dv


def _np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def _maxerr(gpu, ref):
    g = _np(gpu)
    assert np.isfinite(g).all(), "GPU output has non-finite (unwritten?) elements"
    return float(np.abs(g - ref).max()) if g.size else 0.0


def _err(gpu, ref, relative):
    err = _maxerr(gpu, ref)
    return err / max(1.0, float(np.abs(ref).max())) if relative else err


def check_heads(eba, q, k, v, do, scale, heads=None, bwd=True, relative=False):
    """Run fwd (+bwd) on the GPU for the whole batch; compare the listed heads.

    relative=True is for inputs that are not unit-variance: each output's
    max-abs error is then divided by max(1, max |oracle value|), since the bf16
    rounding of the result itself grows with its magnitude.
    """
    qd, kd, vd, dod = (x.cuda() for x in (q, k, v, do))
    o, lse = run_fwd(eba, qd, kd, vd, scale)
    if bwd:
        dq, dk, dv = run_bwd(eba, qd, kd, vd, o, dod, lse, scale)
    torch.cuda.synchronize()
    B, H = q.shape[:2]
    heads = heads or [(b, h) for b in range(B) for h in range(H)]
    worst = {}
    for b, h in heads:
        sl = (slice(b, b + 1), slice(h, h + 1))
        ro, rl = oracle.forward(q[sl], k[sl], v[sl], scale)
        errs = {"o": _err(o[sl], ro, relative), "lse": _maxerr(lse[sl], rl)}
        if bwd:
            rdq, rdk, rdv = oracle.backward(q[sl], k[sl], v[sl], do[sl], scale)
            errs.update(dq=_err(dq[sl], rdq, relative), dk=_err(dk[sl], rdk, relative),
                        dv=_err(dv[sl], rdv, relative))
        for n, err in errs.items():
            worst[n] = max(worst.get(n, 0.0), err)
    assert worst["lse"] <= TOL_LSE, worst
    for n in ("o", "dq", "dk", "dv"):
        if n in worst:
            assert worst[n] <= TOL, worst
    return worst


def test_tiny(eba):
    q, k, v, do = W.make_inputs(W.TINY)
    check_heads(eba, q, k, v, do, W.TINY.scale)


RAGGED = [
    # B, H, Lq, Lk, d
    (1, 1, 1, 1, 64),
    (1, 1, 1, 300, 64),
    (1, 2, 17, 129, 64),
    (2, 1, 129, 17, 64),
    (1, 1, 255, 256, 64),
    (1, 1, 384, 384, 64),     # three query tiles: the second CTA holds one tile
    (2, 3, 200, 333, 64),
    (1, 1, 1, 1, 128),
    (1, 2, 100, 257, 128),
    (2, 1, 300, 513, 128),
    (1, 1, 640, 200, 128),
]


@pytest.mark.parametrize("B,H,Lq,Lk,d", RAGGED, ids=lambda x: str(x))
def test_ragged_shapes(eba, B, H, Lq, Lk, d):
    q, k, v, do = W.make_inputs(W.TINY, seed=1000 + Lq + Lk + d, B=B, H=H, Lq=Lq, Lk=Lk, d=d)
    check_heads(eba, q, k, v, do, 1.0 / math.sqrt(d))


def test_scale_and_sharp_softmax(eba):
    # K x 4 and a large scale push the row max far beyond the first tile's
    # maximum, exercising the online rescale path.
    q, k, v, do = W.make_inputs(W.TINY, seed=77, B=1, H=2, Lq=256, Lk=1000, d=64)
    k = (k.float() * torch.linspace(0.1, 4.0, 1000)[None, None, :, None]).to(torch.bfloat16)
    check_heads(eba, q, k, v, do, 0.3, relative=True)


def _pool_workers(bytes_per_head):
    """Worker count for the oracle pool: the host's cores, fewer if each head's
    float64 arrays would not fit in half of the available memory."""
    try:
        with open("/proc/meminfo") as f:
            avail = next(int(l.split()[1]) * 1024 for l in f if l.startswith("MemAvailable"))
    except (OSError, StopIteration):
        avail = 16 << 30
    return max(1, min(os.cpu_count() or 1, avail // 2 // bytes_per_head))


def check_all_heads(eba, w, heads, tmp_path, model_outputs=()):
    """fwd + bwd of the whole workload on the GPU; the listed heads against the
    float64 oracle in a pool of worker processes. Every output is held to the
    flat bar except those in model_outputs (inputs outside the unit-variance
    regime), which are held to the bf16 rounding model's limit. Returns the
    worst error of each output over those heads."""
    q, k, v, do = W.make_inputs(w)
    qd, kd, vd, dod = (x.cuda() for x in (q, k, v, do))
    o, lse = run_fwd(eba, qd, kd, vd, w.scale)
    dq, dk, dv = run_bwd(eba, qd, kd, vd, o, dod, lse, w.scale)
    torch.cuda.synchronize()
    # S, P, dP, dS and temporaries of one head in float64
    per_head = 6 * 8 * w.Lq * w.Lk
    errs = oracle_pool.head_errors(
        dict(q=q, k=k, v=v, do=do, o=o, lse=lse, dq=dq, dk=dk, dv=dv), heads, w.scale, True,
        str(tmp_path), workers=_pool_workers(per_head), model=bool(model_outputs))
    worst = oracle_pool.worst(errs)
    print(f"\n{w.name}: {len(heads)} heads, worst max-abs error (value, (b, h)) and counts: "
          f"{worst}")
    print(f"{w.name}: heads with an element above the flat 2e-2, per output: "
          + str({n: sum(e[n] > TOL for e in errs.values()) for n in ("o", "dq", "dk", "dv")}))

    def over(e):
        flat = [n for n in ("o", "dq", "dk", "dv") if n not in model_outputs and e[n] > TOL]
        model = [n for n in model_outputs if e[f"{n}_n_over_model"] > 0]
        return flat + model + (["lse"] if e["lse"] > TOL_LSE else [])

    bad = {bh: over(e) for bh, e in errs.items() if over(e)}
    assert not bad, f"{len(bad)} of {len(heads)} heads over the bar, e.g. {list(bad.items())[:4]}"
    return worst


def test_vit_b_every_head(eba, tmp_path):
    # Every (batch, head) of the ViT-B workload (384 heads, unit-variance
    # inputs) at full size, in the launch configuration the benchmark times:
    # the flat 2e-2 / 1e-3 bar on every output.
    w = W.VIT_B
    check_all_heads(eba, w, [(b, h) for b in range(w.B) for h in range(w.H)], tmp_path)


def test_vit_l_every_head(eba, tmp_path):
    # Every (batch, head) of the ViT-L workload (256 heads). Its K is doubled,
    # so its inputs are outside the unit-variance regime of the flat bar: the
    # scores have standard deviation 2, the softmax is sharp and |dQ| reaches
    # ~6, where the bf16 rounding of dQ itself is up to 0.0156. An
    # implementation making no error beyond the method's own data formats (O
    # saved in bf16 and D taken from it, dQ written in bf16) already exceeds a
    # flat 2e-2 on some heads (float64 emulation: 3 of 256, worst 0.029), so dQ
    # is held to the bf16 rounding model's limit (rounding_model.py) and its
    # flat error is reported; O, dK, dV and lse keep the flat bar.
    w = W.VIT_L
    check_all_heads(eba, w, [(b, h) for b in range(w.B) for h in range(w.H)], tmp_path,
                    model_outputs=("dq",))


def test_long_video_sampled_heads(eba, tmp_path):
    # 4 of the 32 heads of the 12544-token workload (the float64 oracle holds
    # ~1.3 GB per score-sized matrix of one head), spread over both batches.
    w = W.LONG_VIDEO
    check_all_heads(eba, w, [(0, 0), (0, 11), (1, 7), (1, 15)], tmp_path)


def _ulp_distance(a, b):
    """Distance in bf16 steps between two bf16 tensors (adjacent values: 1)."""
    def ordered(t):
        i = t.contiguous().view(torch.int16).to(torch.int32)
        return torch.where(i < 0, -(i & 0x7FFF), i)
    return (ordered(a) - ordered(b)).abs()


def test_cross_split_merge_full_size(eba):
    w = W.CROSS
    q, k, v, do = W.make_inputs(w)
    qd, kd, vd, dod = (x.cuda() for x in (q, k, v, do))
    bounds = [0] + [b for _, b in W.chunk_bounds(w.Lk, w.n_chunks)]
    o_parts, lse_parts = eba.split_fwd(qd, kd, vd, bounds, w.scale)
    o, lse = eba.merge(o_parts, lse_parts)
    o_ref_gpu, lse_ref_gpu = run_fwd(eba, qd, kd, vd, w.scale)
    dq, dk, dv = run_bwd(eba, qd, kd, vd, o, dod, lse, w.scale)
    torch.cuda.synchronize()
    # Merged split vs unsplit over every head (not just the sampled ones): both
    # round P to bf16 against different reference maxima, so they may differ by
    # that rounding, but never by more than the oracle tolerance.
    assert (o.float() - o_ref_gpu.float()).abs().max().item() <= TOL
    assert (lse - lse_ref_gpu).abs().max().item() <= TOL_LSE
    # Closer than that: the two roundings of P differ by noise of about
    # 2^-10 of O's spread, so wherever |O| exceeds its spread the two bf16
    # results are at most 1 ulp apart (a few exceptions allowed), and nowhere
    # do they differ by a tenth of the spread; the lse values agree to 1e-4.
    sd = o_ref_gpu.float().std().item()
    assert (o.float() - o_ref_gpu.float()).abs().max().item() <= 0.1 * sd
    assert (lse - lse_ref_gpu).abs().max().item() <= 1e-4
    big = o_ref_gpu.float().abs() > sd
    assert (_ulp_distance(o, o_ref_gpu)[big] <= 1).float().mean().item() >= 0.999
    for bb, h in [(0, 0), (0, 19), (1, 5), (1, 31)]:
        sl = (slice(bb, bb + 1), slice(h, h + 1))
        ro, rl = oracle.forward(q[sl], k[sl], v[sl], w.scale)
        assert _maxerr(o[sl], ro) <= TOL
        assert _maxerr(lse[sl], rl) <= TOL_LSE
        # each chunk's partial against the oracle's partial
        for c, (k0, k1) in enumerate(W.chunk_bounds(w.Lk, w.n_chunks)):
            po, pl = oracle.partial_forward(q[sl], k[sl], v[sl], w.scale, k0, k1)
            assert _maxerr(o_parts[c][sl], po) <= TOL
            assert _maxerr(lse_parts[c][sl], pl) <= TOL_LSE
        rdq, rdk, rdv = oracle.backward(q[sl], k[sl], v[sl], do[sl], w.scale)
        assert _maxerr(dq[sl], rdq) <= TOL
        assert _maxerr(dk[sl], rdk) <= TOL
        assert _maxerr(dv[sl], rdv) <= TOL


@pytest.mark.parametrize("k0,k1", [(0, 1), (5, 5), (0, 300), (37, 291), (128, 256), (299, 300)])
@pytest.mark.parametrize("d", [64, 128])
def test_partial_ranges(eba, k0, k1, d):
    q, k, v, _ = W.make_inputs(W.TINY, seed=5 + k0 + k1, B=2, H=2, Lq=140, Lk=300, d=d)
    qd, kd, vd = (x.cuda() for x in (q, k, v))
    o, lse = eba.partial_fwd(qd, kd, vd, k0, k1, 1 / math.sqrt(d))
    torch.cuda.synchronize()
    ro, rl = oracle.partial_forward(q, k, v, 1 / math.sqrt(d), k0, k1)
    assert np.abs(_np(o) - ro).max() <= TOL
    if k0 == k1:
        assert torch.isneginf(lse).all()
    else:
        assert np.abs(_np(lse) - rl).max() <= TOL_LSE


@pytest.mark.parametrize("C", [1, 3, 8, 64])
@pytest.mark.parametrize("d", [64, 128])
def test_split_then_merge_matches_oracle(eba, C, d):
    Lk = 777
    q, k, v, _ = W.make_inputs(W.TINY, seed=C * 10 + d, B=1, H=3, Lq=130, Lk=Lk, d=d)
    rng = np.random.default_rng(C)
    cuts = sorted(rng.integers(0, Lk + 1, size=C - 1).tolist())
    bounds = [0] + cuts + [Lk]
    qd, kd, vd = (x.cuda() for x in (q, k, v))
    o_parts, lse_parts = eba.split_fwd(qd, kd, vd, bounds, 1 / math.sqrt(d))
    o, lse = eba.merge(o_parts, lse_parts)
    torch.cuda.synchronize()
    ro, rl = oracle.forward(q, k, v, 1 / math.sqrt(d))
    assert np.abs(_np(o) - ro).max() <= TOL
    assert np.abs(_np(lse) - rl).max() <= TOL_LSE


@pytest.mark.parametrize("C,d", [(4, 64), (5, 128), (8, 64), (13, 128), (64, 64)])
def test_merge_handles_empty_chunks(eba, C, d):
    # An empty chunk's lse is -inf and its partial O carries no weight, whatever
    # its values (here non-zero); a row whose chunks are all empty gets O = 0,
    # lse = -inf.
    rng = np.random.default_rng(3 + C)
    B, H, Lq = 1, 2, 50
    o_parts = rng.normal(size=(C, B, H, Lq, d))
    lse_parts = rng.normal(size=(C, B, H, Lq)) * 3
    lse_parts[1] = -np.inf                       # one empty chunk everywhere
    lse_parts[:, :, 1, :7] = -np.inf             # rows with every chunk empty
    ro, rl = oracle.merge(o_parts, lse_parts)
    o, lse = eba.merge(torch.tensor(o_parts, dtype=torch.float32).cuda(),
                       torch.tensor(lse_parts, dtype=torch.float32).cuda())
    torch.cuda.synchronize()
    assert np.abs(_np(o) - ro).max() <= TOL
    l = _np(lse)
    assert (np.isneginf(l) == np.isneginf(rl)).all()
    fin = ~np.isneginf(rl)
    assert np.abs(l[fin] - rl[fin]).max() <= TOL_LSE


def test_forward_is_deterministic(eba):
    q, k, v, do = (x.cuda() for x in W.make_inputs(W.VIT_L, B=2, H=4))
    o1, l1 = run_fwd(eba, q, k, v, 0.125)
    o2, l2 = run_fwd(eba, q, k, v, 0.125)
    dq1, dk1, dv1 = run_bwd(eba, q, k, v, o1, do, l1, 0.125)
    dq2, dk2, dv2 = run_bwd(eba, q, k, v, o1, do, l1, 0.125)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert torch.equal(dk1, dk2) and torch.equal(dv1, dv2)
    assert (dq1.float() - dq2.float()).abs().max().item() <= TOL


def test_autograd_function(eba):
    q, k, v, do = W.make_inputs(W.TINY, seed=9, B=2, H=2, Lq=150, Lk=150, d=64)
    qd, kd, vd = (x.cuda().requires_grad_(True) for x in (q, k, v))
    o = eba.attention(qd, kd, vd)
    o.backward(do.cuda())
    ro, _ = oracle.forward(q, k, v, 0.125)
    rdq, rdk, rdv = oracle.backward(q, k, v, do, 0.125)
    assert np.abs(_np(o) - ro).max() <= TOL
    assert np.abs(_np(qd.grad) - rdq).max() <= TOL
    assert np.abs(_np(kd.grad) - rdk).max() <= TOL
    assert np.abs(_np(vd.grad) - rdv).max() <= TOL


def test_calls_from_another_host_thread(eba):
    # The autograd engine runs backward on its own thread; the library must
    # work from any host thread.
    import threading

    q, k, v, do = W.make_inputs(W.TINY, seed=21, B=1, H=2, Lq=130, Lk=140, d=64)
    qd, kd, vd, dod = (x.cuda() for x in (q, k, v, do))
    out = {}

    def work():
        try:
            o, lse = eba.fwd(qd, kd, vd)
            out["g"] = eba.bwd(qd, kd, vd, o, dod, lse)
            torch.cuda.synchronize()
        except Exception as e:  # reported below
            out["err"] = e

    t = threading.Thread(target=work)
    t.start()
    t.join()
    assert "err" not in out, out.get("err")
    rdq, rdk, rdv = oracle.backward(q, k, v, do, 0.125)
    for g, r in zip(out["g"], (rdq, rdk, rdv)):
        assert np.abs(_np(g) - r).max() <= TOL


def test_gpu_rejects_misaligned_and_reports_ok_status(eba):
    x = torch.zeros(1, 1, 64 * 8 + 8, dtype=torch.bfloat16, device="cuda")
    mis = x.data_ptr() + 2
    st = eba.lib().attn_fwd(mis, x.data_ptr(), x.data_ptr(), x.data_ptr(), x.data_ptr(), 1, 1, 8,
                            8, 64, 0.125, None)
    assert st == 3
    assert eba.poll_device_status() == 0
