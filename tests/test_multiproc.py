"""The N > 1 host path of bench.py (replicas): max-over-ranks timing and the
whole-job rate, run as two gloo ranks on the CPU."""
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


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    # rank r "took" 10 + r ms for 4 steps of 1000 units each
    ms = bench.max_over_ranks(world, 10.0 + rank, device="cpu")
    rate = bench.whole_job_rate(world, 1000, ms, 4)
    dist.barrier()
    q.put((rank, ms, rate))
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, ms, rate in got:
        assert ms == 11.0  # the slower rank's time
        assert rate == pytest.approx(2 * 1000 / (11e-3 / 4))  # all ranks' units / that time


def test_single_rank_is_unchanged():
    import bench
    assert bench.max_over_ranks(1, 3.5) == 3.5
    assert bench.whole_job_rate(1, 65536, 17.5, 10) == pytest.approx(65536 / 1.75e-3)
