"""bench.py's multi-rank plumbing on CPU: two gloo ranks, barrier, max of the
timings and sum of the work over ranks (replicas: no data-path collective)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    r, w, local = bench.dist_env()
    assert (r, w, local) == (rank, world, rank)
    bench.dist_init(w, "gloo")
    bench.barrier(w)
    times = bench.max_over_ranks([1.0 + rank, 10.0 - rank], w)
    work = bench.sum_over_ranks([100.0 * (rank + 1)], w)
    out[rank] = (times, work)
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_gloo_ranks_reduce_timings_and_work():
    world = 2
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.start_processes(_rank_main, args=(world, port, out), nprocs=world, start_method="spawn", join=True)
    for rank in range(world):
        times, work = out[rank]
        assert times == [2.0, 10.0]
        assert work == [300.0]


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks([3.0, 4.0], 1) == [3.0, 4.0]
    assert bench.sum_over_ranks([5.0], 1) == [5.0]
