"""Replica aggregation of bench.py on CPU: two gloo ranks, as torchrun starts them.

The branch shards by requests with no exchange step, so several GPUs run
independent replicas; the job's rate is the units all ranks processed over the
slowest rank's time.  These tests run the same helpers bench.py uses, in two
processes on the gloo backend (no GPU).
"""
import multiprocessing as mp
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, elapsed, units, out):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    r, w = bench.dist_init("gloo")
    bench.barrier()
    slowest = bench.max_over_ranks(elapsed[rank])
    rate = bench.job_throughput(units, elapsed[rank], w)
    out.put((r, w, slowest, rate))
    dist.destroy_process_group()


def _run(world, elapsed, units):
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, elapsed, units, out)) for r in range(world)]
    for p in procs:
        p.start()
    results = [out.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return sorted(results)


def test_two_replicas_take_the_slowest_rank_and_sum_the_units():
    elapsed = [2.0, 3.0]       # seconds each rank took for its steps
    units = 1000.0             # tokens each rank processed
    res = _run(2, elapsed, units)
    assert [r[0] for r in res] == [0, 1]
    for rank, world, slowest, rate in res:
        assert world == 2
        assert slowest == pytest.approx(3.0)          # max over ranks
        assert rate == pytest.approx(2 * units / 3.0)  # whole-job rate


def test_single_process_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        os.environ.pop(k, None)
    assert bench.dist_info() == (0, 1, 0)
    assert bench.max_over_ranks(1.5) == 1.5
    assert bench.job_throughput(100.0, 2.0, 1) == pytest.approx(50.0)
