"""Multi-rank host logic of bench.py on CPU: two gloo ranks, as torchrun
would start them (RANK / WORLD_SIZE / MASTER_* in the environment).

The bench shards by replication: every rank decodes its own copy of the
workload with no collective on the data path, the ranks meet in a barrier
around the timed region, and the job's time is the slowest rank's.
"""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.multiprocessing as mp  # noqa: E402

import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist

    r, w, local = bench.dist_setup(None)
    try:
        assert (r, w, local) == (rank, world, rank)
        assert dist.get_backend() == "gloo"
        bench.barrier(w)
        # each rank "timed" a different interval; every rank sees the max
        ms = bench.reduce_max(10.0 * (rank + 1), w, torch.device("cpu"))
        out[rank] = (ms, bench.job_throughput(1000, w, ms))
        bench.barrier(w)
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_interval():
    world = 2
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert set(res) == {0, 1}
    for ms, value in res.values():
        assert ms == 20.0
        # 1000 units on each of 2 ranks in the slowest rank's 20 ms
        assert value == pytest.approx(2000 / 0.020)


def test_single_rank_helpers_are_local():
    assert bench.reduce_max(3.5, 1, torch.device("cpu")) == 3.5
    bench.barrier(1)
    assert bench.job_throughput(500, 1, 250.0) == pytest.approx(2000.0)
