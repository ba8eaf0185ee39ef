"""The N > 1 host path of bench.py (replicas: one process per GPU, the job's
time is the slowest replica's, throughput sums the replicas) run as two gloo
ranks on the CPU. No GPU, no collective in the data path: the only exchange
is the timing reduction."""
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
        local_ms = 10.0 + 5.0 * rank                     # rank 1 is the slower replica
        ms = bench.max_over_ranks(local_ms, dist, torch.device("cpu"))
        value = bench.replica_throughput(1000.0, world, ms)
        out[rank] = (ms, value)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time():
    world, port = 2, _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0] == res[1]                              # every rank reports the same numbers
    ms, value = res[0]
    assert ms == pytest.approx(15.0)                     # the max over ranks
    assert value == pytest.approx(2 * 1000.0 / 0.015)    # both replicas' units over that time


def test_single_process_is_its_own_max():
    assert bench.max_over_ranks(3.5, None, torch.device("cpu")) == 3.5
    assert bench.replica_throughput(100.0, 1, 1000.0) == pytest.approx(100.0)
