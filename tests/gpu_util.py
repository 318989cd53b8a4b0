"""Helpers for the GPU parity tests: move a workload to the device, run the
library through the C ABI, compare with the CPU oracle on the same inputs."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from paged_mla_speculative_tree_gb300 import binding

OUT_ATOL = 1.5e-2  # bf16 output vs fp64 oracle (before rounding)
LSE_ATOL = 1e-3    # fp32 LSE vs fp64 oracle


def out_tolerance(ref, atol=OUT_ATOL):
    """Per-element bound on the bf16 output: ``atol`` on the computed value, plus
    half a bf16 ulp where storage alone can miss by that much (|ref| >= 4: the
    half ulp is 2^-6 >= 1.56e-2; bf16 keeps 8 significant bits, so on
    [2^e, 2^(e+1)) the half ulp is 2^(e-8))."""
    mag = np.abs(np.asarray(ref, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(mag, 1e-300)))
    return np.where(mag >= 4.0, atol + np.exp2(e - 8), atol)


def to_device(wl, dev="cuda"):
    return dict(q=wl.q.to(dev), kv_pool=wl.kv_pool.to(dev), kv_indices=wl.kv_indices.to(dev),
                kv_indptr=wl.kv_indptr.to(dev), out_cache_loc=wl.out_cache_loc.to(dev),
                qo_indptr=wl.qo_indptr.to(dev), custom_mask=wl.custom_mask.to(dev),
                mask_indptr=wl.mask_indptr.to(dev))


def run_gpu(wl, flags=0, nsplit=0, dev_tensors=None, total_q_max=None, max_prefix=None, max_q=None,
            return_err=False, lengths=None, plan_from_lengths=False):
    """``lengths``: buffer lengths passed to the run; ``plan_from_lengths``:
    the split count comes from the batch's request lengths (choose_nsplit)."""
    d = dev_tensors or to_device(wl)
    T = total_q_max or wl.total_q
    m = binding.MlaTreeVerify(wl.bs, max_q or wl.max_q_per_req, T, max_prefix or wl.max_prefix,
                              device=torch.cuda.current_device(), mask_layout=wl.mask_layout,
                              flags=flags, nsplit=nsplit,
                              lengths=(wl.prefix_lens, wl.tree_sizes) if plan_from_lengths else None)
    out = torch.full((T, 64, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((T, 64), float("nan"), dtype=torch.float32, device="cuda")
    m(d["q"], d["kv_pool"], d["kv_indices"], d["kv_indptr"], d["out_cache_loc"], d["qo_indptr"],
      d["custom_mask"], d["mask_indptr"], wl.scale, out, lse, **(lengths or {}))
    torch.cuda.synchronize()
    err = m.device_error()
    o = out.float().cpu().reshape(-1, 512).numpy()
    l = lse.cpu().reshape(-1).numpy()
    if return_err:
        return o, l, err, m
    assert err == 0, f"device error word {err:#x}"
    return o, l


def sample_rows(wl, n, seed=0, include_all_heads_of=2):
    """A seeded row sample: every head of a few tokens plus random (token, head)."""
    rng = np.random.default_rng(seed)
    H = wl.num_heads
    rows = set()
    toks = rng.choice(wl.total_q, size=min(include_all_heads_of, wl.total_q), replace=False)
    for t in toks:
        rows.update(range(int(t) * H, int(t) * H + H))
    rows.update(rng.choice(wl.total_q * H, size=min(n, wl.total_q * H), replace=False).tolist())
    # first and last row of every request
    qop = wl.qo_indptr.numpy()
    for r in range(wl.bs):
        if qop[r + 1] > qop[r]:
            rows.add(int(qop[r]) * H)
            rows.add(int(qop[r + 1]) * H - 1)
    return np.array(sorted(rows), dtype=np.int64)


def compare(wl, out, lse, rows=None, out_atol=OUT_ATOL, lse_atol=LSE_ATOL, tag="", ref=None):
    """out/lse: full GPU results [total_q*H, 512] / [total_q*H]."""
    if ref is None:
        ref_out, ref_lse = oracle.mla_tree_verify(wl, rows=rows)
    else:
        ref_out, ref_lse = ref
    got_out = out if rows is None else out[rows]
    got_lse = lse if rows is None else lse[rows]
    assert np.all(np.isfinite(got_out)), f"{tag}: non-finite output"
    empty = np.isneginf(ref_lse)
    assert np.array_equal(np.isneginf(got_lse), empty), f"{tag}: -inf LSE pattern differs"
    assert np.all(got_out[empty] == 0), f"{tag}: rows without keys must be zero"
    diff = np.abs(got_out - ref_out)
    err_o = diff.max() if got_out.size else 0.0
    err_l = np.abs(got_lse[~empty] - ref_lse[~empty]).max() if (~empty).any() else 0.0
    over = diff - out_tolerance(ref_out, out_atol)
    assert not np.any(over > 0), \
        f"{tag}: out max-abs {err_o:.3e} beyond the bound by {over.max():.3e} (bound {out_atol} + bf16 half-ulp)"
    assert err_l <= lse_atol, f"{tag}: lse max-abs {err_l:.3e} > {lse_atol}"
    return err_o, err_l
