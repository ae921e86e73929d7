"""The benchmark's multi-process path on the CPU (gloo, world size 2).

With N GPUs the benchmark runs N independent replicas of the verify step (the
step of one request does not shard here); the job's time is the slowest
replica's, and rank 0 alone prints.  These tests run that host logic with
real gloo process groups on 127.0.0.1, and the reference arm under torchrun.
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


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = bench.max_over_ranks(1.5 + rank, dist, "cpu")   # rank 1 is the slow one
    dist.barrier()
    q.put((rank, ms, bench.job_us_per_step(ms, world)))
    dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [o[1] for o in out] == [2.5, 2.5]          # every rank sees the max
    assert [o[2] for o in out] == [1250.0, 1250.0]    # 2 steps per 2.5 ms


def test_single_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25, None, "cpu") == 3.25
    assert bench.job_us_per_step(3.25, 1) == 3250.0


def test_reference_arm_under_torchrun_prints_once():
    """Two ranks: rank 0 times the oracle and prints one JSON line, rank 1
    exits 0 without work."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--steps", "1", "--warmup", "0"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2 and rec["value"] > 0
    assert rec["cpu_baseline"]["kind"] == "oracle" and rec["e2e"]["h2d_bytes_per_step"] == 0
    # the same metric, unit, direction and workload as the GPU arm's line
    sys.path.insert(0, ROOT)
    import bench
    assert rec["metric"] == bench.METRIC and rec["unit"] == "us/step"
    assert rec["higher_is_better"] is False and rec["scaling"] == "weak"
    assert rec["config"]["workload"] == bench.WORKLOAD
    assert rec["config"]["bytes_per_step"] == bench.step_bytes()
    assert rec["e2e"]["value"] == rec["value"] and rec["e2e"]["unit"] == rec["unit"]
    assert rec["cpu_baseline"]["value"] == rec["value"] and rec["cpu_baseline"]["cores"] >= 1
