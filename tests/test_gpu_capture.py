"""CUDA-graph capture safety: the run call takes only static pointers, makes no
host sync and no allocation; a graph captured once and replayed with new data
copied into the same buffers matches the oracle on every replay.

The full-size stress case (16 requests x 131,072-token prefix x 64-node tree on
a 2.2M-slot pool, captured once, replayed 100x with new seeded indices, masks,
q and tree slots) checks every replay on a seeded row sample, and replays 0 and
99 on a larger sample."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from paged_mla_speculative_tree_gb300 import binding
from paged_mla_speculative_tree_gb300 import workloads as W
from tests import gpu_util as G

pytestmark = pytest.mark.gpu

BUFS = ("q", "kv_indices", "kv_indptr", "out_cache_loc", "qo_indptr", "custom_mask", "mask_indptr")


def _static(wl):
    return {k: getattr(wl, k).cuda() for k in BUFS}


def _refresh(static, wl):
    for k in BUFS:
        static[k].copy_(getattr(wl, k), non_blocking=True)


def _capture(m, static, pool, scale, out, lse):
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # warm up on the side stream, as capture requires
        m(static["q"], pool, static["kv_indices"], static["kv_indptr"], static["out_cache_loc"],
          static["qo_indptr"], static["custom_mask"], static["mask_indptr"], scale, out, lse, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    free0 = torch.cuda.mem_get_info()[0]
    with torch.cuda.graph(g):
        m(static["q"], pool, static["kv_indices"], static["kv_indptr"], static["out_cache_loc"],
          static["qo_indptr"], static["custom_mask"], static["mask_indptr"], scale, out, lse)
    torch.cuda.synchronize()
    return g, free0


def _moderate(replay):
    g = torch.Generator().manual_seed(900 + replay)
    parents = [W.random_parents(16, g) for _ in range(4)]
    return parents


@pytest.mark.parametrize("flags", [0, binding.FLAG_SIMT_FLOOR], ids=["tc", "simt"])
def test_capture_replay_moderate(flags):
    pool = W.randn_bf16((40000, W.D_QK), torch.Generator().manual_seed(31))
    wls = [W.build_workload("cap", [3000, 2999, 3001, 3000], _moderate(k), 40000,
                            torch.Generator().manual_seed(700 + k), pool=pool) for k in range(4)]
    # same shapes on every replay (static buffers), different content
    shapes = {tuple(getattr(w, k).shape) for w in wls for k in BUFS}
    assert len(shapes) == len({tuple(getattr(wls[0], k).shape) for k in BUFS})
    wl0 = wls[0]
    static = _static(wl0)
    dpool = pool.cuda()
    m = binding.MlaTreeVerify(wl0.bs, 16, wl0.total_q, 3001, flags=flags)
    out = torch.empty((wl0.total_q, 64, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((wl0.total_q, 64), dtype=torch.float32, device="cuda")
    g, _ = _capture(m, static, dpool, wl0.scale, out, lse)
    for k, wl in enumerate(wls):
        _refresh(static, wl)
        g.replay()
        torch.cuda.synchronize()
        o = out.float().cpu().reshape(-1, 512).numpy()
        l = lse.cpu().reshape(-1).numpy()
        rows = G.sample_rows(wl, 128, seed=k)
        G.compare(wl, o, l, rows=rows, tag=f"replay {k}")
    assert m.device_error() == 0


def test_run_makes_no_allocation():
    wl = W.tiny()
    d = G.to_device(wl)
    m = binding.MlaTreeVerify(wl.bs, wl.max_q_per_req, wl.total_q, wl.max_prefix, nsplit=2)
    out = torch.empty((wl.total_q, 64, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((wl.total_q, 64), dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    a0 = torch.cuda.memory_allocated()
    f0 = torch.cuda.mem_get_info()[0]
    for _ in range(3):
        m(d["q"], d["kv_pool"], d["kv_indices"], d["kv_indptr"], d["out_cache_loc"], d["qo_indptr"],
          d["custom_mask"], d["mask_indptr"], wl.scale, out, lse)
    torch.cuda.synchronize()
    assert torch.cuda.memory_allocated() == a0
    assert torch.cuda.mem_get_info()[0] == f0


def test_stress_capture_100_replays():
    pool = W.stress_pool()
    dpool = pool.cuda()
    wl0 = W.stress(0, pool=pool)
    static = _static(wl0)
    m = binding.MlaTreeVerify(wl0.bs, 64, wl0.total_q, 131072)
    out = torch.empty((wl0.total_q, 64, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((wl0.total_q, 64), dtype=torch.float32, device="cuda")
    g, _ = _capture(m, static, dpool, wl0.scale, out, lse)
    H = 64
    rng = np.random.default_rng(5)
    for k in range(100):
        wl = wl0 if k == 0 else W.stress(k, pool=pool)
        _refresh(static, wl)
        g.replay()
        torch.cuda.synchronize()
        o = out.float().cpu().reshape(-1, 512).numpy()
        l = lse.cpu().reshape(-1).numpy()
        if k in (0, 99):
            rows = G.sample_rows(wl, 192, seed=k, include_all_heads_of=1)
        else:  # every request: one random head of each of 4 distinct tree tokens (4 mask rows per request)
            rows = []
            for r in range(wl.bs):
                for t in rng.choice(64, size=4, replace=False):
                    rows.append((int(wl.qo_indptr[r]) + int(t)) * H + int(rng.integers(0, H)))
            rows = np.array(sorted(rows), dtype=np.int64)
        G.compare(wl, o, l, rows=rows, tag=f"stress replay {k}")
        assert np.all(np.isfinite(l)) and np.all(np.isfinite(o))
    assert m.device_error() == 0
