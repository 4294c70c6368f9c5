"""The multi-process (N > 1) host path of the bench on CPU with the gloo
backend: ranks are independent replicas, the job rate is all ranks' work over
the slowest rank's time, and only rank 0 prints."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = [1.0 + rank, 10.0 - rank]  # per-rank (ms, e2e ms)
        got = bench.max_over_ranks(torch, dist, mine)
        work = bench.sum_over_ranks(torch, dist, 2.0e12 + 1.0e12 * rank)  # per-rank FLOPs
        dist.barrier()
        q.put((rank, got, work, bench.job_rate(work, got[0] * 1e-3)))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_rate_gloo_world2():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = dict((r, (g, w, v)) for r, g, w, v in (q.get(timeout=120) for _ in range(world)))
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for r in range(world):
        got, work, rate = res[r]
        assert got == [2.0, 10.0]  # max of (1, 2) and (10, 9)
        assert work == 5.0e12  # 2e12 + 3e12: every rank's own work, summed
        assert rate == pytest.approx(5.0e12 / 2.0e-3)


def test_single_rank_is_identity():
    assert bench.max_over_ranks(torch, None, [3, 4.5]) == [3.0, 4.5]
    assert bench.sum_over_ranks(torch, None, 3) == 3.0
    assert bench.job_rate(1.0, 0.5) == 2.0


def test_reference_arm_under_torchrun_world2():
    """torchrun with two ranks: rank 0 alone runs the reference arm (the oracle on
    the host cores) and prints one JSON line; rank 1 exits 0 without work."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--workload", "prefill_tiny", "--gpus", "2", "--steps", "1", "--warmup", "3"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
