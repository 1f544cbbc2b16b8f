"""The benchmark's multi-process path on CPU: two gloo ranks (CPU only).

bench.py runs one process per GPU with no collective on the data path; the
ranks meet only at a barrier around the timed region and in a max of their
times, and the reported value is world x per-rank FLOPs / that max.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench

    w, r, local = bench.dist_setup()
    assert (w, r, local) == (world, rank, rank)
    ranks = bench.Ranks(world, backend="gloo")
    ranks.barrier()
    # each rank "took" a different time; every rank must see the slowest
    slowest = ranks.max(1.0 + rank)
    value = bench.aggregate_tflops(world, 2.0e12, slowest)
    ranks.barrier()
    ranks.close()
    out.put((rank, slowest, value))


@pytest.mark.parametrize("world", [2])
def test_two_gloo_ranks_agree_on_max_time(world):
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    results = sorted(out.get(timeout=10) for _ in range(world))
    for rank, slowest, value in results:
        assert slowest == float(world)               # max over ranks of 1.0 + rank
        assert value == pytest.approx(world * 2.0e12 / (world * 1e-3) / 1e12)


def test_single_rank_is_a_no_op():
    import bench

    ranks = bench.Ranks(1)
    ranks.barrier()
    assert ranks.max(3.5) == 3.5
    assert bench.aggregate_tflops(1, 1e12, 1.0) == pytest.approx(1000.0)
