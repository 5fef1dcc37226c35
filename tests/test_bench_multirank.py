"""bench.py's multi-rank path on CPU: world_size 2 over gloo.

Every rank runs its own replica of the workload; the whole-job value is the
work of all ranks divided by the slowest rank's time (max over ranks), and the
reference arm runs on rank 0 only (other ranks exit 0 without output).
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, ws, port, local_ms, out):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws))
    sys.path.insert(0, ROOT)
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        import bench

        out.put((rank, bench.whole_job(local_ms[rank], 2.0e12, 5, ws, "cpu")))
    finally:
        dist.destroy_process_group()


def test_whole_job_value_is_max_over_ranks():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    local_ms = [10.0, 14.0]
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, local_ms, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank in (0, 1):
        total_ms, value = res[rank]
        assert total_ms == 14.0
        assert value == pytest.approx(2 * 2.0e12 * 5 / 14.0e-3 / 1e12)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.whole_job(8.0, 1.0e12, 4, 1) == (8.0, pytest.approx(1.0e12 * 4 / 8.0e-3 / 1e12))


def _reference(rank, steps=1):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank))
    return subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--gpus", "2",
                           "--steps", str(steps), "--warmup", "0"],
                          cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)


def test_reference_arm_other_ranks_exit_quietly():
    r = _reference(1)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_reference_arm_rank0_prints_one_line():
    r = _reference(0)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference"
    assert line["n_gpus"] == 2 and line["unit"] == "TFLOP/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
