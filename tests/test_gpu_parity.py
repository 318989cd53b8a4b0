"""GPU parity: the CUDA library (through the C ABI) against the CPU oracle on
the same seeded inputs.  Small cases are compared on every row; the named
full-size workloads on a seeded row sample (plus properties at any size)."""
from __future__ import annotations

import zlib

import numpy as np
import pytest
import torch

import oracle
from paged_mla_speculative_tree_gb300 import binding
from paged_mla_speculative_tree_gb300 import workloads as W
from tests import gpu_util as G
from tests import pins

pytestmark = pytest.mark.gpu

KERNELS = {"tc": 0, "simt": binding.FLAG_SIMT_FLOOR}


@pytest.fixture(params=sorted(KERNELS))
def flags(request):
    return KERNELS[request.param]


# ------------------------------------------------------------ small, every row

def test_tiny_every_row(flags):
    wl = W.tiny()
    out, lse = G.run_gpu(wl, flags)
    G.compare(wl, out, lse, tag="tiny")


@pytest.mark.parametrize("nsplit", [1, 2, 3, 7])
def test_ragged_batch_every_row(flags, nsplit):
    g = torch.Generator().manual_seed(77)
    parents = [W.random_parents(n, g) for n in (1, 5, 13, 3)]
    wl = W.custom([0, 77, 300, 129], parents, 2048, seed=78)
    out, lse = G.run_gpu(wl, flags, nsplit=nsplit)
    G.compare(wl, out, lse, tag=f"ragged nsplit={nsplit}")


@pytest.mark.parametrize("layout", [W.MASK_FULL_ROW, W.MASK_TREE_ONLY])
def test_hand_derived_worked_example(flags, layout):
    # tests/golden/worked_example.json: outputs in closed form, no oracle involved
    wl, ref_out, ref_lse = pins.worked_example(layout)
    out, lse = G.run_gpu(wl, flags)
    G.compare(wl, out, lse, ref=(ref_out, ref_lse), tag="worked example")


def test_tree_only_layout(flags):
    g = torch.Generator().manual_seed(5)
    parents = [W.random_parents(n, g) for n in (9, 4)]
    wl = W.custom([200, 65], parents, 1024, seed=6, mask_layout=W.MASK_TREE_ONLY)
    out, lse = G.run_gpu(wl, flags, nsplit=2)
    G.compare(wl, out, lse, tag="tree-only")


def test_shapes_chain_star_and_tile_edges(flags):
    # prefix lengths on both sides of tile boundaries, odd tree sizes
    parents = [W.chain_parents(3), W.star_parents(64), W.chain_parents(2), W.random_parents(
        33, torch.Generator().manual_seed(1))]
    wl = W.custom([63, 64, 65, 127], parents, 4096, seed=9)
    out, lse = G.run_gpu(wl, flags, nsplit=3)
    G.compare(wl, out, lse, tag="edges")


def test_empty_request_and_rows_without_keys(flags):
    # request 1 has no tree tokens; request 2 has no prefix and an all-zero mask
    parents = [W.random_parents(4, torch.Generator().manual_seed(2)), [], [W.ROOT, 0, 1]]
    wl = W.custom([40, 10, 0], parents, 512, seed=4)
    mip = wl.mask_indptr.numpy()
    wl.custom_mask[mip[2]:mip[3]] = 0
    out, lse = G.run_gpu(wl, flags, nsplit=2)
    G.compare(wl, out, lse, tag="empty")
    H = 64
    assert np.all(np.isneginf(lse[4 * H:7 * H])) and np.all(out[4 * H:7 * H] == 0)


def test_prefix_mask_columns_ignored(flags):
    wl = W.custom([100], [W.random_parents(6, torch.Generator().manual_seed(3))], 512, seed=8)
    base_o, base_l = G.run_gpu(wl, flags)
    wl.custom_mask.view(6, 106)[:, :100] = 0
    o2, l2 = G.run_gpu(wl, flags)
    assert np.array_equal(base_o, o2) and np.array_equal(base_l, l2)


def test_rows_past_total_q_untouched(flags):
    wl = W.custom([50], [W.chain_parents(4)], 256, seed=12)
    out, lse = G.run_gpu(wl, flags, total_q_max=9)
    H = 64
    assert np.all(np.isnan(out[4 * H:])) and np.all(np.isnan(lse[4 * H:]))
    G.compare(wl, out[:4 * H], lse[:4 * H], tag="capacity")


def test_bad_slot_sets_error_and_is_masked(flags):
    wl = W.custom([70], [W.chain_parents(5)], 512, seed=14)
    bad = wl.kv_indices.clone()
    bad[33] = 10_000_000  # beyond the pool
    d = G.to_device(wl)
    d["kv_indices"] = bad.cuda()
    out, lse, err, _ = G.run_gpu(wl, flags, dev_tensors=d, return_err=True)
    assert err & binding.DEVERR_SLOT_RANGE
    # the offending key is treated as masked: compare with the oracle without it
    keep = torch.cat([wl.kv_indices[:33], wl.kv_indices[34:]])
    wl2 = W.custom([69], [W.chain_parents(5)], 512, seed=14)
    ref = oracle.mla_tree_verify(wl, kv_indices=keep, kv_indptr=torch.tensor([0, 69], dtype=torch.int32),
                                 custom_mask=wl2.custom_mask, mask_indptr=wl2.mask_indptr)
    G.compare(wl, out, lse, ref=ref, tag="bad slot")


@pytest.mark.parametrize("nsplit", [1, 3])
def test_run_steps_partial_then_combine_equals_run(flags, nsplit):
    """The two launches of a pass, enqueued separately with an event between
    them, give the result of one run bit for bit."""
    g = torch.Generator().manual_seed(71)
    wl = W.custom([500, 1300, 64], [W.random_parents(n, g) for n in (7, 16, 2)], 4096, seed=72)
    d = G.to_device(wl)
    m = binding.MlaTreeVerify(wl.bs, wl.max_q_per_req, wl.total_q, wl.max_prefix, flags=flags, nsplit=nsplit)
    outs = []
    for split_steps in (False, True):
        out = torch.full((wl.total_q, 64, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((wl.total_q, 64), float("nan"), dtype=torch.float32, device="cuda")
        args = (m.plan, d["q"], d["kv_pool"], d["kv_indices"], d["kv_indptr"], d["out_cache_loc"], d["qo_indptr"],
                d["custom_mask"], d["mask_indptr"], wl.scale, out, lse, m.workspace)
        if split_steps:
            binding.run(*args, steps=binding.STEP_PARTIAL)
            ev = torch.cuda.Event()
            ev.record()
            binding.run(*args, steps=binding.STEP_COMBINE)
        else:
            binding.run(*args)
        torch.cuda.synchronize()
        outs.append((out.cpu(), lse.cpu()))
    assert torch.equal(outs[0][0].view(torch.int16), outs[1][0].view(torch.int16))
    assert torch.equal(outs[0][1].view(torch.int32), outs[1][1].view(torch.int32))
    assert m.device_error() == 0
    G.compare(wl, outs[1][0].float().reshape(-1, 512).numpy(), outs[1][1].reshape(-1).numpy(), tag="run_steps")


def _padded(t, extra):
    """Device copy of t followed by `extra` zero elements: a declared length
    shorter than the allocation lets a test present offsets past the declared
    end while every byte a kernel could touch is still allocated."""
    buf = torch.zeros(t.numel() + extra, dtype=t.dtype, device="cuda")
    buf[:t.numel()].copy_(t)
    return buf


def _rows_of(wl, reqs):
    H = wl.num_heads
    qop = wl.qo_indptr.numpy()
    return np.concatenate([np.arange(qop[r] * H, qop[r + 1] * H) for r in reqs]).astype(np.int64)


def _three_offset_cases():
    g = torch.Generator().manual_seed(91)
    parents = [W.random_parents(n, g) for n in (5, 7, 3, 6)]
    return W.custom([100, 130, 90, 70], parents, 2048, seed=92)


def test_mask_block_past_custom_mask_end_is_flagged_and_skipped(flags):
    # request 1's mask block starts 3 bytes before the declared end of custom_mask
    wl = _three_offset_cases()
    d = G.to_device(wl)
    d["custom_mask"] = _padded(wl.custom_mask, 1 << 16)
    mip = wl.mask_indptr.clone()
    mip[1] = wl.custom_mask.numel() - 3
    d["mask_indptr"] = mip.cuda()
    out, lse, err, _ = G.run_gpu(wl, flags, nsplit=2, dev_tensors=d, return_err=True,
                                 lengths={"custom_mask_len": wl.custom_mask.numel()})
    assert err & binding.DEVERR_INDPTR
    bad = _rows_of(wl, [1])
    assert np.all(np.isnan(out[bad])) and np.all(np.isnan(lse[bad]))  # skipped: rows untouched
    G.compare(wl, out, lse, rows=_rows_of(wl, [0, 2, 3]), tag="mask past end")


def test_kv_indptr_past_kv_indices_end_is_flagged_and_skipped(flags):
    # kv_indptr[bs] is one past the declared length of kv_indices: the last request is skipped
    wl = _three_offset_cases()
    d = G.to_device(wl)
    d["kv_indices"] = _padded(wl.kv_indices, 4096)
    out, lse, err, _ = G.run_gpu(wl, flags, nsplit=2, dev_tensors=d, return_err=True,
                                 lengths={"kv_indices_len": wl.kv_indices.numel() - 1})
    assert err & binding.DEVERR_INDPTR
    bad = _rows_of(wl, [3])
    assert np.all(np.isnan(out[bad])) and np.all(np.isnan(lse[bad]))
    G.compare(wl, out, lse, rows=_rows_of(wl, [0, 1, 2]), tag="kv_indptr past end")


def test_qo_indptr_past_out_cache_loc_end_is_flagged_and_skipped(flags):
    wl = _three_offset_cases()
    d = G.to_device(wl)
    d["out_cache_loc"] = _padded(wl.out_cache_loc, 256)
    out, lse, err, _ = G.run_gpu(wl, flags, dev_tensors=d, return_err=True,
                                 lengths={"out_cache_loc_len": wl.out_cache_loc.numel() - 2})
    assert err & binding.DEVERR_INDPTR
    bad = _rows_of(wl, [3])
    assert np.all(np.isnan(out[bad])) and np.all(np.isnan(lse[bad]))
    G.compare(wl, out, lse, rows=_rows_of(wl, [0, 1, 2]), tag="qo_indptr past end")


@pytest.mark.parametrize("nsplit", [1, 3])
def test_timeout_path_returns_reports_and_leaves_the_context_usable(nsplit):
    """With the test flag every pipeline wait that has to spin gives up: the
    tensor-core kernel must wind down (MMAs, gathers and score copies drained,
    TMEM freed), report MTV_DEVERR_TIMEOUT and return; a normal call in the
    same process then matches the oracle."""
    g = torch.Generator().manual_seed(77)
    parents = [W.random_parents(n, g) for n in (1, 5, 13, 3)]
    wl = W.custom([0, 77, 300, 129], parents, 2048, seed=78)
    d = G.to_device(wl)
    for _ in range(2):
        _, _, err, _ = G.run_gpu(wl, binding.FLAG_TEST_SHORT_WAITS, nsplit=nsplit, dev_tensors=d,
                                 return_err=True)
        assert err & binding.DEVERR_TIMEOUT
    out, lse = G.run_gpu(wl, 0, nsplit=nsplit, dev_tensors=d)
    G.compare(wl, out, lse, tag="after timeout")


def test_request_beyond_plan_bounds_is_flagged(flags):
    wl = W.custom([300], [W.chain_parents(4)], 1024, seed=15)
    out, lse, err, _ = G.run_gpu(wl, flags, max_prefix=200, return_err=True)
    assert err & binding.DEVERR_INDPTR


# ------------------------------------------------------------ named workloads (sampled)

@pytest.mark.parametrize("name", ["batch4", "long_contig", "long_random", "mixed", "mixed_s2", "mixed_s3"])
def test_named_workload_sampled(flags, name):
    # Mixed is drawn with three seeds: split-K balance across ragged requests is
    # that configuration's point, so one draw of the request sizes is not enough
    wl = {"mixed_s2": lambda: W.mixed(seed=2004), "mixed_s3": lambda: W.mixed(seed=3004)}.get(
        name, W.WORKLOADS.get(name))()
    out, lse = G.run_gpu(wl, flags)
    rows = G.sample_rows(wl, 96, seed=zlib.crc32(name.encode()) % 1000)
    G.compare(wl, out, lse, rows=rows, tag=name)
    assert np.all(np.isfinite(lse)) and np.all(np.isfinite(out))


@pytest.mark.parametrize("seed", [1004, 2004, 3004])
def test_mixed_planned_from_request_lengths(flags, seed):
    """The split count chosen from the batch's request lengths (3, 1 and 4 on
    these draws, where the rule from upper bounds alone picks 3, 3 and 2)
    gives results that match the oracle."""
    wl = W.mixed(seed=seed)
    out, lse, err, m = G.run_gpu(wl, flags, plan_from_lengths=True, return_err=True)
    assert err == 0
    rows = G.sample_rows(wl, 96, seed=seed % 1000)
    G.compare(wl, out, lse, rows=rows, tag=f"mixed {seed}, nsplit {m.plan.nsplit} from lengths")


@pytest.mark.parametrize("name", ["batch4", "long_random"])
def test_large_logits_sampled(flags, name):
    """q scaled by 4.5: the largest scaled logits reach ~30 and one CTA's
    partial scores reach a few hundred raw units, where a score exchange whose
    error grows with the size of the scores would miss the LSE tolerance."""
    wl = W.scaled_q(W.WORKLOADS[name](), 4.5)
    out, lse = G.run_gpu(wl, flags)
    rows = G.sample_rows(wl, 160, seed=zlib.crc32(name.encode()) % 997)
    _, ref_lse = oracle.mla_tree_verify(wl, rows=rows)
    assert ref_lse.max() > 25.0  # the regime this test is about
    G.compare(wl, out, lse, rows=rows, tag=f"{name} large logits")


@pytest.mark.parametrize("name", ["batch4", "long_random"])
def test_large_common_component_sampled(flags, name):
    """Keys and queries sharing one large latent direction: every score carries
    an offset of ~1,740 raw units (~870 in each CTA's half of the dims)."""
    wl = W.common_component(W.WORKLOADS[name]())
    out, lse = G.run_gpu(wl, flags)
    rows = G.sample_rows(wl, 160, seed=zlib.crc32(name.encode()) % 991)
    G.compare(wl, out, lse, rows=rows, tag=f"{name} common component")


def test_long_contiguous_equals_random_slots(flags):
    a, b = W.long_context(True), W.long_context(False)
    oa, la = G.run_gpu(a, flags)
    ob, lb = G.run_gpu(b, flags)
    assert np.array_equal(oa, ob) and np.array_equal(la, lb)


@pytest.mark.parametrize("nsplit", [1, 3])
def test_growing_scores_move_the_reference_every_tile(flags, nsplit):
    """Scores that grow along the keys by more than the lazy-rescale threshold
    (2^8) per 64-key tile, driven through the rope dims: the running max moves
    on every tile, so the O rescale path and the LSE bookkeeping across moves
    run many times (random data moves it almost only on the first tile)."""
    g = torch.Generator().manual_seed(4242)
    wl = W.custom([280, 200], [W.random_parents(6, g), W.chain_parents(3)], 4096, seed=4243)
    u = torch.randn(64, generator=g).to(torch.bfloat16).float()
    thr_raw = 8.0 / (wl.scale * 1.4426950408889634)
    step = 1.1 * thr_raw / float((u * u).sum())  # per 64 keys
    q = wl.q.float()
    q[:, :, :512] = 0.05 * torch.randn(q[:, :, :512].shape, generator=g)
    q[:, :, 512:] = u + 0.05 * torch.randn(q[:, :, 512:].shape, generator=g)
    wl.q = q.to(torch.bfloat16)
    pool = wl.kv_pool.float()
    for r in range(wl.bs):
        p = wl.prefix_lens[r]
        slots = torch.cat([wl.kv_indices[int(wl.kv_indptr[r]):int(wl.kv_indptr[r + 1])],
                           wl.out_cache_loc[int(wl.qo_indptr[r]):int(wl.qo_indptr[r + 1])]])
        pos = torch.arange(slots.numel(), dtype=torch.float32)
        pool[slots, :512] = 0.5 * torch.randn((slots.numel(), 512), generator=g)
        pool[slots, 512:] = (step * pos / 64.0)[:, None] * u[None, :]
        assert p + 0 <= slots.numel()
    wl.kv_pool = pool.to(torch.bfloat16)
    out, lse = G.run_gpu(wl, flags, nsplit=nsplit)
    G.compare(wl, out, lse, tag=f"growing nsplit={nsplit}")
