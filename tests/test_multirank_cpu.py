"""The multi-rank host logic on CPU ranks (gloo, world size 2): the split of a
bucket into contiguous per-rank chunks, the job's time as the slowest
rank's, and the throughput over the units of all ranks. No GPU and no
data-path collective are involved (the oracle stands in for the per-rank
compute)."""
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
        out.put((rank, ms, bench.rank_chunk(rank, world), bench.job_throughput(24 * 3, world, ms / 1e3)))
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
    assert got[0][2] == (0, 24) and got[1][2] == (24, 24)  # contiguous chunks of one bucket
    assert got[0][3] == got[1][3] == pytest.approx(24 * 3 * 2 / 0.015)


def test_single_rank_is_identity():
    assert bench.max_over_ranks(3.5, None, None) == 3.5
    assert bench.job_throughput(10, 1, 2.0) == 5.0



def _chunk_rank(rank, world, port, G, out):
    import numpy as np
    from inputs import generators as gen
    from newton_schulz_gram_gb300.partition import partition
    from oracle import gram_ns
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        start, count = partition(G, world, rank)
        X = gen.gaussian_bucket(count, 8, 32, seed=31, first=start)
        mine = {start + i: gram_ns.orthogonalize(X[i].astype(np.float64)) for i in range(count)}
        gathered = [None] * world
        dist.all_gather_object(gathered, mine)
        if rank == 0:
            out.put(gathered)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("G", [7, 2, 1])
def test_bucket_chunks_cover_every_matrix_once_and_match_the_single_rank_run(G):
    import numpy as np
    from inputs import generators as gen
    from oracle import gram_ns
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    procs = [ctx.Process(target=_chunk_rank, args=(r, world, port, G, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    gathered = out.get(timeout=10)
    keys = [k for part in gathered for k in part]
    assert sorted(keys) == list(range(G))  # every matrix exactly once
    X = gen.gaussian_bucket(G, 8, 32, seed=31)
    merged = {k: v for part in gathered for k, v in part.items()}
    for g in range(G):
        assert np.array_equal(merged[g], gram_ns.orthogonalize(X[g].astype(np.float64)))


def test_partition_sizes():
    from newton_schulz_gram_gb300.partition import partition
    for G in (0, 1, 5, 24, 100):
        for world in (1, 2, 3, 8):
            spans = [partition(G, world, r) for r in range(world)]
            assert sum(c for _, c in spans) == G
            assert all(spans[r][0] + spans[r][1] == spans[r + 1][0] for r in range(world - 1))
            assert max(c for _, c in spans) - min(c for _, c in spans) <= 1
    with pytest.raises(ValueError):
        partition(4, 2, 2)
