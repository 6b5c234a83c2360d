"""The benchmark's multi-rank host logic on CPU (gloo, world size 2).

The decode path does not shard: N GPUs run N independent replicas, each its
own requests, with no collective on the data path.  What N > 1 adds is host
bookkeeping: a barrier, the slowest rank's time and the whole-job rate, and
the reference arm running on rank 0 only.  These run here as two gloo
processes, no GPU."""
import io
import os
import socket
import sys
from contextlib import redirect_stdout
from types import SimpleNamespace

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def worker(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        own_ms = 10.0 + 5.0 * rank  # rank 1 is the slower one
        worst = bench.max_over_ranks(own_ms, world, "cpu")
        rate = bench.job_rate(world, 100, worst)
        dist.barrier()
        out.put((rank, worst, rate))
    finally:
        dist.destroy_process_group()


def test_slowest_rank_and_whole_job_rate_over_two_gloo_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[0] for r in results] == [0, 1]
    for _, worst, rate in results:
        assert worst == 15.0                     # every rank sees the slowest time
        assert rate == pytest.approx(2 * 100 / 0.015)  # all units over that time


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.job_rate(1, 10, 5.0) == pytest.approx(2000.0)


def test_reference_arm_runs_on_rank_zero_only():
    sys.path.insert(0, ROOT)
    import bench
    args = SimpleNamespace(steps=3, warmup=3, gpus=2)
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(args, 2, 1)  # a non-zero rank returns without work or output
    assert buf.getvalue() == ""


def test_rank_environment():
    sys.path.insert(0, ROOT)
    import bench
    env = dict(os.environ)
    try:
        os.environ.update(WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
        assert bench.dist_setup() == (2, 1, 1)
        for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
            del os.environ[k]
        assert bench.dist_setup() == (1, 0, 0)
    finally:
        os.environ.clear()
        os.environ.update(env)
