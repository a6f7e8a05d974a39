"""The multi-process plumbing of bench.py on CPU: two ranks over gloo (the
path shards by sequence, so ranks run independent replicas and only the
timing is reduced: a barrier around the timed region and the max over ranks)."""

import os
import socket

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
