"""The multi-rank path of bench.py (one independent replica per GPU) on CPU:
two gloo ranks aggregate their timed regions as the maximum over ranks and
report the whole job's tokens per second."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch.distributed as dist
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms_local = 10.0 + 5.0 * rank           # rank 1 is the slower replica
        ms_max, value = bench.job_throughput(ms_local, steps=64, batch=2, world=world, device="cpu")
        out[rank] = (ms_max, value, bench.replica_seed(1000, rank))
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    world, port = 2, _free_port()
    with mp.get_context("spawn").Manager() as mgr:  # no fork of a multi-threaded process
        out = mgr.dict()
        mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert set(res) == {0, 1}
    for r in (0, 1):
        ms_max, value, _ = res[r]
        assert ms_max == pytest.approx(15.0)                        # the slowest rank
        assert value == pytest.approx(2 * 64 * 2 / 15.0e-3)         # tokens of both ranks
    assert res[0][2] != res[1][2]                                   # independent inputs per rank


def test_one_rank_reports_its_own_time():
    import bench
    ms_max, value = bench.job_throughput(8.0, steps=10, batch=1, world=1, device="cpu")
    assert ms_max == 8.0 and value == pytest.approx(10 / 8.0e-3)
