"""The N>1 host path of bench.py on CPU: two gloo ranks partition one batch by
request (balanced on (p_r + n_r) * n_r), each builds its share, and both agree
on the slowest rank's time."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from paged_mla_speculative_tree_gb300 import partition as PT
from paged_mla_speculative_tree_gb300 import workloads as W


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _batch():
    g = torch.Generator().manual_seed(61)
    sizes = [8, 64, 3, 17, 40, 1, 25]
    prefix = [4000, 300, 12000, 77, 2500, 9000, 640]
    return W.custom(prefix, [W.random_parents(n, g) for n in sizes], 32768, seed=62)


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ws, r, local = bench.dist_env()
    wl = _batch()
    parts = PT.partition_requests(wl.prefix_lens, wl.tree_sizes, ws)
    mine = W.sub_workload(wl, parts[r])
    ms = bench.max_over_ranks(1.0 + 0.5 * rank, ws)  # rank 1 is the slower one
    q.put((r, ws, local, ms, parts[r], mine.bs, mine.total_q, int(mine.kv_indptr[-1])))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_partition_the_batch_and_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert [g[0] for g in got] == [0, 1] and all(g[1] == 2 for g in got) and [g[2] for g in got] == [0, 1]
    assert all(g[3] == pytest.approx(1.5) for g in got)  # max over ranks
    wl = _batch()
    union = sorted(got[0][4] + got[1][4])
    assert union == list(range(wl.bs))  # every request exactly once
    assert sum(g[6] for g in got) == wl.total_q and sum(g[7] for g in got) == sum(wl.prefix_lens)


def test_partition_is_balanced_and_exact():
    rng = np.random.default_rng(3)
    for world in (1, 2, 3, 4, 8):
        prefix = rng.integers(0, 70000, size=29).tolist()
        sizes = rng.integers(1, 65, size=29).tolist()
        parts = PT.partition_requests(prefix, sizes, world)
        assert sorted(r for p in parts for r in p) == list(range(29))
        loads = PT.partition_loads(prefix, sizes, parts)
        costs = [PT.request_cost(p, n) for p, n in zip(prefix, sizes)]
        # greedy longest-first: the slowest rank is within the largest request of the average
        assert max(loads) <= sum(costs) / world + max(costs)
        # and within 4/3 of the lower bound max(average, largest request)
        assert max(loads) <= 4.0 / 3.0 * max(sum(costs) / world, max(costs)) + 1


def test_sub_workload_rows_match_the_whole_batch():
    wl = _batch()
    parts = PT.partition_requests(wl.prefix_lens, wl.tree_sizes, 3)
    H = 64
    qop = wl.qo_indptr.numpy()
    for p in parts:
        sub = W.sub_workload(wl, p)
        rows = np.arange(0, sub.total_q * H, 331)
        o1, l1 = oracle.mla_tree_verify(sub, rows=rows)
        full_rows = np.concatenate([np.arange(qop[r] * H, qop[r + 1] * H) for r in p])[rows]
        o2, l2 = oracle.mla_tree_verify(wl, rows=full_rows)
        assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_single_rank_is_unchanged():
    import bench
    assert bench.max_over_ranks(2.5, 1) == 2.5
    assert PT.partition_requests([10, 20], [1, 2], 1) == [[0, 1]]
