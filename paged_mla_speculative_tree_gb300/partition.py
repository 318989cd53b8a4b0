"""Request partition for running one verify-attention batch on several GPUs.

Requests are independent (each attends only over its own prefix and tree), so
a batch shards by request with no exchange step.  The work of request r is
proportional to (p_r + n_r) * n_r: its 64 * n_r query rows each attend over
p_r + n_r keys.  Requests are assigned longest-first to the least-loaded rank
(LPT greedy), which bounds the slowest rank at 4/3 of the optimum.
"""
from __future__ import annotations


def request_cost(prefix_len: int, tree_size: int) -> int:
    return (int(prefix_len) + int(tree_size)) * int(tree_size)


def partition_requests(prefix_lens, tree_sizes, world: int):
    """Returns ``world`` sorted lists of request indices covering the batch once."""
    if world < 1:
        raise ValueError("world must be >= 1")
    costs = [request_cost(p, n) for p, n in zip(prefix_lens, tree_sizes)]
    order = sorted(range(len(costs)), key=lambda r: (-costs[r], r))
    loads = [0] * world
    parts = [[] for _ in range(world)]
    for r in order:
        k = min(range(world), key=lambda i: (loads[i], i))
        parts[k].append(r)
        loads[k] += costs[r]
    return [sorted(p) for p in parts]


def partition_loads(prefix_lens, tree_sizes, parts):
    return [sum(request_cost(prefix_lens[r], tree_sizes[r]) for r in p) for p in parts]
