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
        q.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_max_times():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = dict(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    expect = [11.0, 6.0, 5.0]
    assert results[0] == expect and results[1] == expect


def test_weak_scaling_value_is_units_of_all_ranks_over_slowest_time():
    import bench
    # 2 replicas of 2.7495e11 FLOP each, slowest rank 0.36 ms -> aggregate TFLOPS
    flops, ms, world = 274945015808, 0.36, 2
    assert bench.reduce_max([ms], 1) == [ms]
    value = world * flops / (ms * 1e-3) / 1e12
    assert abs(value - 1527.47) < 0.01
