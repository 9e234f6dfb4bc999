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


def test_spawned_replicas_report_one_aggregated_line(capfd):
    """bench.spawn_replicas starts the ranks itself (torch.distributed.run on
    127.0.0.1); two gloo ranks time a stand-in step and rank 0 alone prints
    the whole-job line, timed by the slower rank."""
    import json
    stub = os.path.join(os.path.dirname(os.path.abspath(__file__)), "replica_stub.py")
    env = dict(os.environ)
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT"):
        env.pop(k, None)
    env["OMP_NUM_THREADS"] = "1"
    rc = bench.spawn_replicas(2, stub, [], env=env)
    assert rc == 0
    lines = [ln for ln in capfd.readouterr().out.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["n_gpus"] == 2
    assert rec["ms_per_step"] >= rec["own_ms"]
    assert rec["value"] == pytest.approx(2 * 1e9 / (rec["ms_per_step"] * 1e-3) / 1e9)


def test_bench_starts_its_own_ranks_without_torchrun(monkeypatch):
    """`bench.py --gpus N` with no WORLD_SIZE in the environment hands itself
    to spawn_replicas with N ranks and its own arguments."""
    calls = []
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    monkeypatch.setattr(bench, "spawn_replicas", lambda n, script, argv: calls.append((n, script, argv)) or 0)
    monkeypatch.setattr(bench.sys, "argv", ["bench.py", "--gpus", "4", "--steps", "7"])
    with pytest.raises(SystemExit) as e:
        bench.main()
    assert e.value.code == 0
    assert calls == [(4, os.path.abspath(bench.__file__), ["--gpus", "4", "--steps", "7"])]
