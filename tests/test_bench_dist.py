"""bench.py's multi-rank host logic (replicas, one process per GPU) on CPU with
world_size-2 gloo: the barrier, the max-over-ranks time and the whole-job
throughput. No GPU and no collective on the data path are involved."""
from __future__ import annotations

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, out):
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        ms_local = 2.0 if rank == 0 else 5.0  # rank 1 is the slow replica
        ms, gbs = bench.aggregate(1_000_000, ms_local, world, "cpu")
        out[rank] = (ms, gbs)
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_two_replicas_report_the_slowest_time_and_the_summed_throughput():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    for r in range(2):
        ms, gbs = res[r]
        assert ms == pytest.approx(5.0)
        assert gbs == pytest.approx(2 * 1_000_000 / 5e-3 / 1e9)


def test_single_rank_is_plain():
    import bench
    ms, gbs = bench.aggregate(1_000_000, 4.0, 1, "cpu")
    assert ms == 4.0 and gbs == pytest.approx(1_000_000 / 4e-3 / 1e9)
