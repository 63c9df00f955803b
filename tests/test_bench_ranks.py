"""The benchmark's multi-rank path on CPU: two gloo ranks, each with its own time.

With N GPUs the benchmark runs N independent replicas (requests shard across ranks with no data
exchange); the only cross-rank step is the timing: every rank's time is reduced to the slowest
one, and the whole-job rate is the units all ranks processed over that time.
"""
import os
import socket

import pytest


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out):
    import torch.distributed as tdist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench

    r, w, local = bench.dist_env()
    tdist.init_process_group("gloo", rank=r, world_size=w)
    try:
        ms = bench.max_over_ranks(times[r], w)
        out.put((r, local, ms, bench.job_throughput(100, w, ms)))
    finally:
        tdist.destroy_process_group()


def test_timing_reduces_to_the_slowest_rank():
    mp = pytest.importorskip("torch.multiprocessing")
    ctx = mp.get_context("spawn")
    world, port = 2, _free_port()
    times = [12.5, 20.0]  # ms of the timed region on each rank
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, times, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r for r, *_ in res] == [0, 1]
    assert [local for _, local, *_ in res] == [0, 1]
    for _, _, ms, value in res:
        assert ms == 20.0                       # the slowest rank's time, on every rank
        assert value == pytest.approx(2 * 100 / 0.020)  # both ranks' 100 units over 20 ms


def test_single_rank_needs_no_process_group():
    import bench

    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.job_throughput(200, 1, 50.0) == pytest.approx(4000.0)
