"""The allocation-free entry point (fixed device scratch instead of a caller
workspace) must give the same result as the workspace entry point.

Kept in a file of its own, collected last, so that a failure here never hides
the other GPU tests; it also passes when run alone in a fresh process."""
import numpy as np
import pytest
import torch

from paged_mla_speculative_tree_gb300 import binding
from paged_mla_speculative_tree_gb300 import workloads as W
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


def _wl(seed):
    g = torch.Generator().manual_seed(seed)
    parents = [W.random_parents(n, g) for n in (16, 11)]
    return W.custom([3000, 1777], parents, 8192, seed=seed)


def test_static_scratch_entry_matches_workspace_entry_twice():
    wls = [_wl(51), _wl(52)]  # two calls in a row, different data, same plan
    T = max(w.total_q for w in wls)
    m = binding.MlaTreeVerify(2, 16, T, 3000, nsplit=3)  # nsplit > 1: the scratch holds partials
    assert m.plan.ws_bytes > 256
    for wl in wls:
        d = G.to_device(wl)
        ref_out = torch.zeros((T, 64, 512), dtype=torch.bfloat16, device="cuda")
        ref_lse = torch.zeros((T, 64), dtype=torch.float32, device="cuda")
        m(d["q"], d["kv_pool"], d["kv_indices"], d["kv_indptr"], d["out_cache_loc"], d["qo_indptr"],
          d["custom_mask"], d["mask_indptr"], wl.scale, ref_out, ref_lse)
        out = torch.zeros_like(ref_out)
        lse = torch.zeros_like(ref_lse)
        binding.run_static(m.plan, d["q"], d["kv_pool"], d["kv_indices"], d["kv_indptr"], d["out_cache_loc"],
                           d["qo_indptr"], d["custom_mask"], d["mask_indptr"], wl.scale, out, lse)
        torch.cuda.synchronize()
        n = wl.total_q
        o_ref = ref_out[:n].float().cpu().reshape(-1, 512).numpy()
        o = out[:n].float().cpu().reshape(-1, 512).numpy()
        l_ref = ref_lse[:n].cpu().reshape(-1).numpy()
        l = lse[:n].cpu().reshape(-1).numpy()
        assert np.abs(o - o_ref).max() <= G.OUT_ATOL
        assert np.abs(l - l_ref).max() <= G.LSE_ATOL
        # and both agree with the oracle on a sample
        rows = G.sample_rows(wl, 64, seed=3)
        G.compare(wl, o, l, rows=rows, tag="static scratch")
        assert binding.read_static_device_error() == 0


def test_static_scratch_reports_its_error_word_and_allocates_nothing():
    wl = _wl(53)
    d = G.to_device(wl)
    m = binding.MlaTreeVerify(2, 16, wl.total_q, 3000, nsplit=3)
    out = torch.zeros((wl.total_q, 64, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((wl.total_q, 64), dtype=torch.float32, device="cuda")
    bad = d["kv_indices"].clone()
    bad[10] = 1 << 40  # far outside the pool: flagged, treated as masked
    args = (m.plan, d["q"], d["kv_pool"], bad, d["kv_indptr"], d["out_cache_loc"], d["qo_indptr"],
            d["custom_mask"], d["mask_indptr"], wl.scale, out, lse)
    binding.run_static(*args)  # first call on this device resolves the scratch address
    torch.cuda.synchronize()
    assert binding.read_static_device_error() & binding.DEVERR_SLOT_RANGE
    a0 = torch.cuda.memory_allocated()
    f0 = torch.cuda.mem_get_info()[0]
    for _ in range(3):
        binding.run_static(*args)
    torch.cuda.synchronize()
    assert torch.cuda.memory_allocated() == a0 and torch.cuda.mem_get_info()[0] == f0
    # each call clears the word first: a clean call reports nothing
    binding.run_static(m.plan, d["q"], d["kv_pool"], d["kv_indices"], d["kv_indptr"], d["out_cache_loc"],
                       d["qo_indptr"], d["custom_mask"], d["mask_indptr"], wl.scale, out, lse)
    assert binding.read_static_device_error() == 0


def test_static_scratch_rejects_oversized_plan():
    # 600 tokens x 16 splits of fp32 partials is far above the 64 MiB scratch
    p = binding.plan(torch.cuda.current_device(), 8, 64, 600, 65536, nsplit=16)
    assert p.ws_bytes > (64 << 20)
    z = torch.zeros(16, dtype=torch.uint8, device="cuda")
    # rejected before any buffer is touched
    rc = binding.run_static(p, z.view(torch.bfloat16), z.view(torch.bfloat16), None, z[:8].view(torch.int32),
                            None, z[:8].view(torch.int64), None, z[:8].view(torch.int64), 1.0,
                            z.view(torch.bfloat16), z.view(torch.float32), check=False)
    assert rc == -4  # MTV_E_WORKSPACE_SMALL
