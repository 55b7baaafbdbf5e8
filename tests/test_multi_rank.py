"""The N > 1 path of bench.py on CPU: two gloo ranks, each a replica of the workload.

bench.py shards nothing on the data path (replicas only); its only cross-rank steps are the
barrier around the timed region and the max-over-ranks of the measured times, from which rank 0
reports units processed by all ranks / slowest rank's time.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        assert (r, w, local) == (rank, world, rank)
        # each replica measured different times; every rank must see the slowest
        times = [10.0 + rank, 3.0 * (1 + rank), 5.0 - rank]
        dist.barrier()
        got = bench.reduce_max(times, world)
        # the job's rate: each rank processed the same units; rank 1 is the slower one on the
        # first time, so the aggregate is twice the units over rank 1's time
        units = 274945015808
        rate = bench.job_rate(units, got[0], world)
        own = bench.job_rate(units, times[0], world)
        q.put((rank, got, rate, own))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_max_times_and_the_job_rate():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = {r: (got, rate, own) for r, got, rate, own in (q.get(timeout=120) for _ in range(world))}
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    expect = [11.0, 6.0, 5.0]
    assert results[0][0] == expect and results[1][0] == expect
    # both ranks report the same job rate, set by the slowest rank's 11 ms
    assert results[0][1] == results[1][1] == 2 * 274945015808 / 11e-3
    # rank 0 alone was faster (10 ms): the aggregate must not use its own time
    assert results[0][1] < results[0][2]


def test_job_rate_is_units_of_all_ranks_over_slowest_time():
    import bench
    # one replica: the rate is just units over time; N replicas multiply the units, not the time
    assert bench.job_rate(1000, 2.0, 1) == 1000 / 2e-3
    assert bench.job_rate(1000, 2.0, 4) == 4 * bench.job_rate(1000, 2.0, 1)
    assert bench.reduce_max([2.0, 3.0], 1) == [2.0, 3.0]
