"""bench.py's multi-rank host logic (replicas only) with two gloo ranks on the
CPU: the barrier, the max over ranks of the timings, and the whole-job value
for N independent replicas."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    import torch
    import torch.distributed as dist

    import bench
    w, r, _ = bench.dist_init()
    assert (w, r) == (world, rank)
    bench.barrier(w)
    per_rank_us = 100.0 + 50.0 * rank           # rank 1 is the slow one
    slowest = bench.max_over_ranks(per_rank_us, w, torch.device("cpu"))
    q.put((rank, slowest, bench.replica_value(slowest, w)))
    dist.destroy_process_group()


def test_two_gloo_ranks_max_and_replica_value():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    got = sorted(q.get(timeout=5) for _ in range(2))
    assert [g[1] for g in got] == [150.0, 150.0]          # both ranks see the slowest rank's time
    assert [g[2] for g in got] == [75.0, 75.0]            # 2 layers per 150 us -> 75 us per layer


def test_single_rank_value_is_the_time():
    import bench
    assert bench.replica_value(123.0, 1) == 123.0
    assert bench.max_over_ranks(5.0, 1, None) == 5.0
