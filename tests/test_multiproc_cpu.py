"""The N>1 host path of bench.py (replicas, one rank per GPU) on CPU: two gloo
ranks agree on the slowest rank's time and report the whole-job value."""
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


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ws, r, local = bench.dist_env()
    ms = bench.max_over_ranks(1.0 + 0.5 * rank, ws)  # rank 1 is the slower replica
    q.put((r, ws, local, ms, bench.job_us_per_call(ms, ws)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert [g[0] for g in got] == [0, 1] and all(g[1] == 2 for g in got) and [g[2] for g in got] == [0, 1]
    assert all(g[3] == pytest.approx(1.5) for g in got)  # max over ranks
    assert all(g[4] == pytest.approx(750.0) for g in got)  # 2 calls per 1.5 ms -> 750 us per call for the job


def test_single_rank_is_unchanged():
    import bench
    assert bench.max_over_ranks(2.5, 1) == 2.5
    assert bench.job_us_per_call(2.5, 1) == pytest.approx(2500.0)
