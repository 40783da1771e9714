"""bench.py's multi-rank bookkeeping on CPU: two gloo ranks, each with its own replica time,
agree on the slowest rank's time and the whole-job throughput (weak scaling)."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench

        ms = bench.max_over_ranks(times[rank], world)
        value = bench.job_throughput(1_000_000_000, ms, world)
        out[rank] = (ms, value)
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("times", [(2.0, 3.0), (5.0, 1.0)])
def test_two_ranks_agree_on_the_slowest_time(times):
    world = 2
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, times, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    slowest = max(times)
    for r in range(world):
        ms, value = out[r]
        assert ms == slowest
        # 2 ranks x 1 GB each over the slowest rank's time
        assert value == pytest.approx(2 * 1.0 / (slowest * 1e-3))



def test_single_rank_is_unchanged():
    import bench

    assert bench.max_over_ranks(4.5, 1) == 4.5
    assert bench.job_throughput(2_000_000_000, 2.0, 1) == pytest.approx(1000.0)
