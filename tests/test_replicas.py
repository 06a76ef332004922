"""Replica aggregation of bench.py (one process per GPU, no collective on the
data path): two gloo ranks on the CPU report different byte counts and step
times; the whole-job value is all bytes over the slowest rank's time, the
same on every rank."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      LOCAL_RANK=str(rank), WORLD_SIZE=str(world))
    r, local, w = bench.dist_env()
    assert (r, local, w) == (rank, rank, world)
    d = bench.init_dist(w)
    try:
        seconds = [0.010, 0.025][rank]
        nbytes = [1.0e9, 3.0e9][rank]
        value, t_max, total = bench.replica_throughput(d, nbytes, seconds)
        bench.barrier(d)
        out[rank] = (value, t_max, total)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_aggregate_as_replicas():
    world = 2
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert set(res) == {0, 1}
    for rank in (0, 1):
        value, t_max, total = res[rank]
        assert t_max == pytest.approx(0.025)
        assert total == pytest.approx(4.0e9)
        assert value == pytest.approx(4.0e9 / 0.025 / 1e9)


def test_single_process_has_no_group():
    assert bench.init_dist(1) is None
    value, t_max, total = bench.replica_throughput(None, 2.0e9, 0.5)
    assert (value, t_max, total) == (4.0, 0.5, 2.0e9)
