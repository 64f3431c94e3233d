"""The benchmark's multi-rank host logic on CPU with two gloo ranks: each rank
gets its own batch (different seeds), the barrier works, and the timing is the
maximum over ranks; the reference arm runs on rank 0 only."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    w_, r_, l_ = bench.dist_setup()
    assert (w_, r_, l_) == (world, rank, rank)
    bench.barrier(world)
    got = bench.max_over_ranks(1.5 + rank, world)
    import torch.distributed as dist
    dist.destroy_process_group()
    q.put((rank, got, bench.rank_seed(1002, rank)))


def test_two_gloo_ranks_take_the_max_and_use_distinct_batches():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get() for _ in range(world))
    assert [r[1] for r in res] == [2.5, 2.5]
    assert res[0][2] != res[1][2]
