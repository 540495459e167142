"""The N > 1 path of bench.py: independent replicas, one per rank, whose only
cross-rank step is the max of the step times. Run as two gloo processes on CPU."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms, e2e = bench.reduce_over_ranks(1.0 + rank, 10.0 - rank, world)
    q.put((rank, ms, e2e, bench.job_value(1e12, world, ms)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_timing_takes_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, ms, e2e, value in got:
        assert ms == 2.0 and e2e == 10.0           # max over ranks
        assert value == pytest.approx(2 * 1e12 / 2e-3 / 1e12)


def test_single_rank_is_unchanged():
    assert bench.reduce_over_ranks(3.0, 4.0, 1) == (3.0, 4.0)
    assert bench.job_value(2e12, 1, 1.0) == pytest.approx(2000.0)   # 2 TFLOP in 1 ms


def test_step_time_quantiles():
    """The spread reported beside the step time: linear-interpolation quantiles."""
    xs = [1.0, 2.0, 3.0, 4.0, 5.0]
    assert bench.quantile(xs, 0.0) == 1.0 and bench.quantile(xs, 1.0) == 5.0
    assert abs(bench.quantile(xs, 0.1) - 1.4) < 1e-12 and abs(bench.quantile(xs, 0.9) - 4.6) < 1e-12
    assert bench.quantile([7.0], 0.9) == 7.0
