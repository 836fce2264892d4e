"""The multi-GPU path of bench.py is N independent replicas (the layer does
not shard on one node); its host logic -- slowest-rank time over ranks and
whole-job throughput -- checked with two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t = bench.max_over_ranks(times[rank], dist, "cpu")
        out[rank] = (t, bench.job_throughput(world, 4096, 10, t))
    finally:
        dist.destroy_process_group()


def test_slowest_rank_sets_the_job_time():
    world, times = 2, [12.5, 20.0]
    with mp.Manager() as m:
        out = m.dict()
        port = _free_port()
        mp.spawn(_rank, args=(world, port, times, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        t, thr = res[rank]
        assert t == 20.0
        assert thr == pytest.approx(2 * 4096 * 10 / 0.020)


def test_single_rank_throughput():
    assert bench.job_throughput(1, 4096, 100, 200.0) == pytest.approx(4096 * 100 / 0.2)
