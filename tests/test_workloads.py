"""The seeded generator draws valid inputs with the stated structure."""
import numpy as np
import torch

from paged_mla_speculative_tree_gb300 import workloads as W
from tests import pins


def _check(wl):
    assert wl.q.dtype == torch.bfloat16 and wl.q.shape == (wl.total_q, 64, 576)
    assert wl.kv_pool.dtype == torch.bfloat16 and wl.kv_pool.shape[1] == 576
    assert wl.kv_indices.dtype == torch.int64 and wl.kv_indptr.dtype == torch.int32
    assert wl.out_cache_loc.dtype == torch.int64 and wl.qo_indptr.dtype == torch.int64
    assert wl.custom_mask.dtype == torch.uint8 and wl.mask_indptr.dtype == torch.int64
    used = torch.cat([wl.kv_indices, wl.out_cache_loc])
    assert used.unique().numel() == used.numel(), "slot collision"
    assert int(used.min()) >= 0 and int(used.max()) < wl.num_slots
    for r in range(wl.bs):
        par = wl.parents[r]
        assert all(p < i for i, p in enumerate(par)), "parent must precede child or be the root"
        p, n = wl.prefix_lens[r], wl.tree_sizes[r]
        mip = wl.mask_indptr.numpy()
        blk = wl.custom_mask[mip[r]:mip[r + 1]].numpy()
        if wl.mask_layout == W.MASK_FULL_ROW:
            blk = blk.reshape(n, p + n)[:, p:]
        else:
            blk = blk.reshape(n, n)
        assert np.array_equal(blk.astype(bool), pins.closure_visibility(par))


def test_tiny_workload():
    wl = W.tiny()
    _check(wl)
    assert wl.prefix_lens == [256] and wl.tree_sizes == [8] and wl.num_slots == 4096


def test_tiny_is_deterministic():
    a, b = W.tiny(), W.tiny()
    assert torch.equal(a.q.view(torch.int16), b.q.view(torch.int16))
    assert torch.equal(a.kv_indices, b.kv_indices) and torch.equal(a.custom_mask, b.custom_mask)


def test_mixed_shapes_and_ranges():
    wl = W.mixed()
    _check(wl)
    assert wl.bs == 8 and all(1024 <= p <= 65536 for p in wl.prefix_lens)
    assert all(8 <= n <= 64 for n in wl.tree_sizes)
    for shape, par in zip(wl.meta["shapes"], wl.parents):
        if shape == "chain":
            assert par == W.chain_parents(len(par))
        if shape == "star":
            assert par == W.star_parents(len(par))


def test_long_variants_hold_same_tokens():
    a, b = W.long_context(True), W.long_context(False)
    _check(a)
    _check(b)
    assert torch.equal(a.kv_indices, torch.arange(32768))
    ka = a.kv_pool[a.kv_indices].view(torch.int16)
    kb = b.kv_pool[b.kv_indices].view(torch.int16)
    assert torch.equal(ka, kb)
    assert torch.equal(a.q.view(torch.int16), b.q.view(torch.int16))


def test_tree_only_layout_small():
    wl = W.custom([5, 9], [W.chain_parents(3), W.star_parents(4)], 64, seed=1,
                  mask_layout=W.MASK_TREE_ONLY)
    _check(wl)


def test_shared_prefix_generator_shares_the_prefix_slots():
    wl = W.shared_prefix(bs=4, prefix=50, tree=3, num_slots=512, seed=1)
    ind = wl.kv_indices.numpy().reshape(4, 50)
    assert (ind == ind[0]).all()  # one prefix, listed once per request
    ocl = wl.out_cache_loc.numpy()
    assert len(set(ocl.tolist())) == ocl.size and not set(ocl.tolist()) & set(ind[0].tolist())
    assert wl.kv_indptr.tolist() == [0, 50, 100, 150, 200] and wl.qo_indptr.tolist() == [0, 3, 6, 9, 12]
