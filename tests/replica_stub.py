"""One rank of a two-rank CPU run of the benchmark's replica path (launched by
bench.spawn_replicas under torch.distributed.run in tests/test_replicas.py).

A stand-in step (a short CPU matmul loop, no GPU) is timed on every rank;
the ranks then agree on the slowest rank's time and rank 0 prints the
aggregated line, as bench.run_gpu_arm does for its CUDA step."""
import json
import os
import sys
import time

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import torch  # noqa: E402
import torch.distributed as dist  # noqa: E402

import bench  # noqa: E402


def main():
    world = int(os.environ["WORLD_SIZE"])
    rank = int(os.environ["RANK"])
    dist.init_process_group("gloo")
    steps, bytes_per_step = 3, 1e9
    x = torch.ones(64, 64)
    bench.barrier(world)
    t = time.perf_counter()
    for _ in range(steps * (1 + rank)):  # rank 1 is the slow one
        x = x @ x / 64.0
    ms = 1e3 * (time.perf_counter() - t) / steps
    ms_max = bench.dist_max(ms, world)
    bench.barrier(world)
    if rank == 0:
        print(json.dumps({"n_gpus": world, "ms_per_step": ms_max, "own_ms": ms,
                          "value": bench.replica_value(bytes_per_step, ms_max, world)}))
    dist.destroy_process_group()


if __name__ == "__main__":
    main()
