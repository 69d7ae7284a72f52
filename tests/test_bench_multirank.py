"""The bench's multi-rank timing logic on two gloo ranks (CPU, no GPU).

Replicas share no data, so the only cross-rank steps are the barrier and the
max-over-ranks of the step time; the whole-job value counts every rank's
bytes over the slowest rank's time.
"""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, lr = bench.dist_env()
        assert (r, w, lr) == (rank, world, rank)
        bench.barrier(world)
        ms = [2.0, 3.5][rank]                        # rank 1 is the slower replica
        out[rank] = (bench.max_over_ranks(ms, world), bench.whole_job(1e9, world, bench.max_over_ranks(ms, world)))
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_two_ranks():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    for r in range(world):
        slowest, value = out[r]
        assert slowest == pytest.approx(3.5)             # every rank sees the slowest rank's time
        assert value == pytest.approx(2e9 / 3.5e-3)      # 2 ranks x 1e9 units over 3.5 ms


def test_single_rank_helpers_need_no_process_group():
    assert bench.max_over_ranks(1.25, 1) == 1.25
    assert bench.whole_job(10.0, 1, 2.0) == pytest.approx(5000.0)
    bench.barrier(1)
