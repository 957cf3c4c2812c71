"""The N > 1 bench path is "replicas only": every rank streams its own copy of the
workload and the ranks meet only for a barrier and a max over their step times.
These CPU tests run that host logic on two gloo ranks."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        barrier, reduce_max = bench.replica_helpers(dist, "cpu")
        barrier()
        # each rank's own step time; the job's time is the slowest rank's
        ms = reduce_max(1.0 + rank * 0.5)
        barrier()
        out[rank] = ms
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, _free_port(), out), nprocs=world, join=True)
        got = dict(out)
    assert got == {0: 1.5, 1: 1.5}


def test_replica_value_counts_all_ranks():
    # 13,172,736 bytes per step per rank, 2 ranks, 2 ms for the slowest rank
    assert bench.replica_value(13172736, 2, 2.0) == pytest.approx(13.172736)
    assert bench.replica_value(13172736, 1, 2.0) == pytest.approx(6.586368)
