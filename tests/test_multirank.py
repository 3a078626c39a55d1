"""The benchmark's multi-rank host logic on CPU: two gloo ranks reduce their
timings to the slowest one and agree on the whole-job rate (the path shards
by independent query rows / replicas, so there is no data exchange)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms, kern = bench.max_over_ranks([10.0 + 5.0 * rank, 3.0 - rank])
        rate = bench.whole_job_rate(131072, 100, world, ms)
        out[rank] = (ms, kern, rate)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world = 2
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_rank_main, args=(world, port, out), nprocs=world, start_method="spawn")
        res = dict(out)
    assert res[0] == res[1]
    ms, kern, rate = res[0]
    assert ms == 15.0 and kern == 3.0
    assert rate == pytest.approx(2 * 131072 * 100 / 15e-3)


def test_single_process_is_identity():
    assert bench.max_over_ranks([1.5, 2.5]) == [1.5, 2.5]
    assert bench.whole_job_rate(10, 4, 1, 2.0) == pytest.approx(20000.0)
