"""A rank started by bench.spawn_ranks in the CPU tests: it reads the rank
environment the launcher set, joins a gloo group, reduces a per-rank time the
way bench.py does, and rank 0 prints one JSON line."""

import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import bench  # noqa: E402

if __name__ == "__main__":
    rank, local, world = bench.dist_env()
    assert local == rank and os.environ["MASTER_ADDR"] == "127.0.0.1"
    bench.dist_init(world, "gloo")
    bench.barrier(world)
    ms = bench.max_over_ranks(10.0 + rank, world, torch.device("cpu"))
    if rank == 0:
        print(json.dumps({"world": world, "ms": ms, "tokens_per_s": bench.job_tokens_per_s(4, world, 100, ms)}),
              flush=True)
    torch.distributed.destroy_process_group()
