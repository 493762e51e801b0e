"""The benchmark's multi-rank host logic on CPU ranks (gloo, world size 2): each
rank works on its own bucket, the job's time is the slowest rank's, and the
throughput counts the units of all ranks. No GPU and no data-path
collective are involved."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = 10.0 + 5.0 * rank  # rank 1 is the slow one
        ms = bench.max_over_ranks(local_ms, dist, torch.device("cpu"))
        out.put((rank, ms, bench.rank_seed(rank), bench.job_throughput(24 * 3, world, ms / 1e3)))
    finally:
        dist.destroy_process_group()


def test_two_cpu_ranks_take_the_slowest_time_and_count_all_units():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(out.get(timeout=10) for _ in range(world))
    assert [g[1] for g in got] == [15.0, 15.0]
    assert got[0][2] != got[1][2]  # independent buckets
    assert got[0][3] == got[1][3] == pytest.approx(24 * 3 * 2 / 0.015)


def test_single_rank_is_identity():
    assert bench.max_over_ranks(3.5, None, None) == 3.5
    assert bench.job_throughput(10, 1, 2.0) == 5.0

