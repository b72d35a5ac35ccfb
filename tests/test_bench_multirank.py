"""The replica aggregation of bench.py across ranks, on CPU with gloo
(world size 2): the job's time is the slowest rank's and the throughput
counts every rank's tokens."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [10.0, 25.0][rank]
    e2e = [0.5, 0.2][rank]
    got = bench.max_over_ranks([ms, e2e], world, "cpu")
    tput = bench.aggregate_throughput(1000, ms, world, "cpu")
    out[rank] = (got, tput)
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_aggregate_throughput_gloo():
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
    for r in (0, 1):
        got, tput = out[r]
        assert got == [25.0, 0.5]           # the slowest rank bounds the job
        assert tput == pytest.approx(2 * 1000 / 0.025)


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks([3.0, 4.0], 1) == [3.0, 4.0]
    assert bench.aggregate_throughput(100, 50.0, 1) == pytest.approx(2000.0)
