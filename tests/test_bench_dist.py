"""The multi-rank host logic of bench.py on CPU: two gloo ranks, barrier, max over ranks of
the elapsed time, whole-job aggregation (each rank quantizes its own batch: weak scaling,
no collective on the data path)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank), PTGQ_BENCH_BACKEND="gloo")
    import torch
    import bench
    w, r, _ = bench.dist_setup(world)
    assert (w, r) == (world, rank)
    bench.barrier(w)
    elapsed = 0.5 + rank          # rank 1 is the slow one
    mx = bench.reduce_max(elapsed, w, torch.device("cpu"))
    value = bench.aggregate(bytes_per_step=1000, steps=10, world=w, max_elapsed_s=mx)
    out[rank] = (mx, value)
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_rank_max_and_aggregate():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    for r in range(world):
        mx, value = out[r]
        assert mx == pytest.approx(1.5)
        assert value == pytest.approx(2 * 10 * 1000 / 1.5 / 1e9)


def test_single_rank_aggregate():
    import bench
    assert bench.aggregate(88_309_760, 100, 1, 0.0015) == pytest.approx(88_309_760 * 100 / 0.0015 / 1e9)
    assert bench.algorithmic_bytes() == 88_309_760
