"""bench.py's multi-GPU path (independent replicas) on the CPU: two gloo ranks.

The whole-job time is the slowest replica's, and the whole-job µs per call divides it by
the calls of all ranks.  The reference arm (the oracle on the host cores) runs on rank 0
alone; the other ranks return without work.
"""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out_q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    t = bench.max_over_ranks(times[rank])
    us = bench.whole_job_us_per_call(t, steps=10, world=world)
    dist.barrier()
    dist.destroy_process_group()
    out_q.put((rank, t, us))


def test_two_replicas_take_the_slowest_rank():
    world, times = 2, [3.0, 5.0]          # ms for 10 calls on each rank
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, times, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, t, us in res:
        assert t == 5.0
        assert us == pytest.approx(5.0e3 / 20)   # 5 ms over 2 x 10 calls


def test_single_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(7.5) == 7.5
    assert bench.whole_job_us_per_call(2.0, 100, 1) == pytest.approx(20.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    from mla_tree_verify_gb300 import workloads as W

    class Args:
        steps, warmup = 1, 0
    monkeypatch.setenv("RANK", "1")
    # rank 1 returns before touching the oracle or printing anything
    assert bench.run_reference(Args(), W.shape(1), W.SHAPE_NAMES[1]) is None
