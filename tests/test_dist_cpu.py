"""The multi-GPU launch path of the benchmark on CPU processes.

The decode path shards over sequences with no exchange, so N GPUs run N
independent replicas: the only cross-rank steps are the barrier around the
timed region, the maximum of the ranks' times, and the whole-job throughput
rank 0 prints.  Those run here over gloo with two ranks, and the reference
arm runs under torchrun with two processes (rank 0 alone times the oracle and
prints one line; the other rank exits without work)."""

import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = 10.0 + 5.0 * rank            # the ranks' own timed regions
    dist.barrier()
    worst = bench.dist_max(local_ms, dist, "cpu")
    q.put((rank, worst, bench.job_tokens_per_s(world, 16, 100, worst)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time_and_sum_the_replicas():
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = [q.get(timeout=180) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert sorted(r for r, _, _ in got) == [0, 1]
    for _, worst, value in got:
        assert worst == 15.0
        assert value == pytest.approx(2 * 16 * 100 / 0.015)


def test_single_process_helpers():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.dist_max(3.5) == 3.5
    assert bench.job_tokens_per_s(1, 16, 100, 1000.0) == pytest.approx(1600.0)


def test_reference_arm_under_torchrun_prints_one_line():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--config", "tiny_fp32", "--steps", "1", "--warmup", "3", "--gpus", "2"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"
