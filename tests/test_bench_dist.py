"""The benchmark's multi-process path (replicas, barrier, max over ranks) on
CPU with the gloo backend, world size 2."""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench

    r, local, w = bench.dist_setup(world)
    assert (r, local, w) == (rank, rank, world)
    bench.barrier(w)
    # each replica measured a different time; every rank must see the largest
    results[rank] = bench.max_over_ranks(10.0 + 5.0 * rank, w)
    bench.barrier(w)
    import torch.distributed as dist

    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    results = manager.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, results)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(100)
        assert p.exitcode == 0
    assert dict(results) == {0: 15.0, 1: 15.0}


def test_single_process_needs_no_process_group():
    import bench

    assert bench.max_over_ranks(3.5, 1) == 3.5
    bench.barrier(1)
