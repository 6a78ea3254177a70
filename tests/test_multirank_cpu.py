"""The N > 1 replica path of bench.py on CPU: two gloo ranks agree on the slowest
rank's timings, the whole-job value counts every rank's tokens, and under
torchrun the reference arm prints one line from rank 0 only.  No GPU."""

import json
import os
import socket
import subprocess
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        vals = [10.0 + rank, 3.0 * (1 - rank), 7.5]
        q.put((rank, bench.max_over_ranks(vals, "cpu", world)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_timings():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert got[0] == got[1] == [11.0, 3.0, 7.5]


def test_single_rank_passes_values_through():
    assert bench.max_over_ranks([1.0, 2.0], "cpu", 1) == [1.0, 2.0]


def test_whole_job_value_counts_every_rank():
    assert bench.replica_value(1, 640, 100.0) == pytest.approx(6400.0)
    assert bench.replica_value(4, 640, 100.0) == pytest.approx(25600.0)


def test_reference_arm_under_torchrun_prints_once_from_rank_zero():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--workload", "toy", "--gpus", "2", "--steps", "1", "--warmup", "3"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["value"] > 0
