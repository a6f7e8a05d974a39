"""The multi-process plumbing of bench.py on CPU: two ranks over gloo (the
path shards by sequence, so ranks run independent replicas and only the
timing is reduced: a barrier around the timed region and the max over ranks),
and `bench.py --gpus 2` starting its two ranks itself."""

import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    os.environ.update({"RANK": str(rank), "LOCAL_RANK": str(rank), "WORLD_SIZE": str(world),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    r, local, w = bench.dist_env()
    assert (r, local, w) == (rank, rank, world)
    bench.dist_init(w, "gloo")
    bench.barrier(w)
    # each rank "timed" a different duration; every rank must see the slowest
    ms = bench.max_over_ranks(10.0 + 5.0 * rank, w, torch.device("cpu"))
    bench.barrier(w)
    out.put((rank, ms, bench.job_tokens_per_s(4, w, 100, ms)))
    torch.distributed.destroy_process_group()


def test_two_ranks_take_the_slowest_time_and_count_every_rank_tokens():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    assert [r for r, _, _ in res] == [0, 1]
    for _, ms, tps in res:
        assert ms == 15.0
        # 4 sequences x 2 ranks x 100 steps in 15 ms
        assert tps == pytest.approx(4 * 2 * 100 / 0.015)


def test_single_process_needs_no_group():
    assert bench.max_over_ranks(3.5, 1, torch.device("cpu")) == 3.5
    bench.barrier(1)
    assert bench.job_tokens_per_s(1, 1, 10, 2.0) == pytest.approx(5000.0)


def test_gpus_flag_starts_that_many_ranks():
    # the reference arm needs no GPU: rank 0 times the oracle on one tiny
    # unit, the other rank leaves at once; the line must count both ranks
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = {k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK")}
    res = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--gpus", "2", "--impl", "reference",
                          "--workload", "sliding_f32_b1_pos40", "--steps", "1", "--warmup", "3"],
                         capture_output=True, text=True, timeout=600, env=env, cwd=root)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [json.loads(x) for x in res.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1, res.stdout
    assert lines[0]["n_gpus"] == 2 and lines[0]["impl"] == "reference"


def test_spawned_ranks_see_their_environment(capfd):
    probe = os.path.join(os.path.dirname(os.path.abspath(__file__)), "rank_probe.py")
    assert bench.spawn_ranks(2, ["--gloo"], script=probe) == 0
    out = [json.loads(x) for x in capfd.readouterr().out.splitlines() if x.startswith("{")]
    assert len(out) == 1                      # rank 1's stdout is dropped
    assert out[0]["world"] == 2 and out[0]["ms"] == 11.0
    assert out[0]["tokens_per_s"] == pytest.approx(4 * 2 * 100 / 0.011)
