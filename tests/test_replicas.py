"""Multi-GPU runs are independent replicas; the benchmark's cross-rank timing
(max over ranks) and whole-job aggregation, checked with two gloo ranks on CPU."""
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


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [1.5, 2.0][rank]
        ms_max = bench.dist_max(local_ms, world)
        out[rank] = (ms_max, bench.replica_value(1e9, ms_max, world))
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_two_rank_max_and_aggregate():
    world, port = 2, _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, start_method="spawn")
    assert out[0][0] == out[1][0] == 2.0
    # 2 replicas x 1 GB in 2 ms (the slower rank) = 1000 GB/s
    assert out[0][1] == pytest.approx(1000.0)


def test_single_rank_is_identity():
    assert bench.dist_max(3.25, 1) == 3.25
    assert bench.replica_value(2e9, 1.0, 1) == pytest.approx(2000.0)
