"""The N > 1 bench path on the CPU: world_size 2 over gloo. Each rank is a replica (tokens
are independent, so no data-path collective); the job time is the slowest rank's and the
job throughput counts every rank's tokens."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    dist.barrier()
    t = bench.reduce_max(times[rank], world, "cpu")
    v = bench.job_tokens_per_s(4096, 10, t, world)
    out[rank] = (t, v)
    dist.destroy_process_group()


@pytest.mark.parametrize("times", [(20.0, 25.0), (31.5, 12.0)])
def test_two_ranks_take_the_slowest_time(times):
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    ctx = mp.get_context("spawn")
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, times, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    slow = max(times)
    for r in range(world):
        t, v = out[r]
        assert t == slow
        assert v == pytest.approx(world * 4096 * 10 / (slow / 1e3))


def test_single_rank_is_unchanged():
    import bench
    assert bench.reduce_max(3.5, 1) == 3.5
    assert bench.job_tokens_per_s(64, 20, 10.0, 1) == pytest.approx(64 * 20 / 0.01)
