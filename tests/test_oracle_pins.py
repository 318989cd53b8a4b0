"""Pins of the CPU oracle against facts that do not come from the oracle itself.

* a dense brute force over every pool slot with visibility from a transitive
  closure of the parent array (different formulation, library matmul);
* chain trees against torch SDPA (fp64) with a causal tree mask;
* invariants: a masked key never changes the output, prefix columns of the
  FULL_ROW mask are never read, permuting the slot map with the data moved is
  exact, V constant => out constant (weights sum to one), an empty tree row is
  plain decode over the prefix;
* closed forms: p=0 and self-only visibility gives out = v_self and
  lse = scale*q.k_self; identical keys give out = v, lse = s + ln(#visible);
* exhaustive enumeration of every 5-node parent array against the brute force;
* a hand-derived worked example (tests/golden/worked_example.json) whose
  outputs are closed forms in e;
* planted mistakes: copies of the oracle source with one plausible bug each
  must fail at least one pin.
"""
from __future__ import annotations

import itertools
import math
import os
import tempfile

import numpy as np
import pytest
import torch

import oracle
from paged_mla_speculative_tree_gb300 import workloads as W
from tests import pins

RTOL = 1e-10
ATOL = 1e-10


def small_wl(seed=7, prefix=(37, 100), parents=None, slots=512, **kw):
    g = torch.Generator().manual_seed(seed)
    if parents is None:
        parents = [W.random_parents(n, g) for n in (5, 8)][:len(prefix)]
    return W.custom(prefix, parents, slots, seed, **kw)


def check_dense(wl, tag=""):
    out, lse = oracle.mla_tree_verify(wl)
    ref_out, ref_lse = pins.dense_reference(wl)
    np.testing.assert_allclose(lse, ref_lse, rtol=RTOL, atol=ATOL, err_msg=f"lse {tag}")
    np.testing.assert_allclose(out, ref_out, rtol=RTOL, atol=ATOL, err_msg=f"out {tag}")


# ---------------------------------------------------------------- dense brute force

def test_dense_bruteforce_random_trees():
    check_dense(small_wl())


def test_dense_bruteforce_tree_only_layout():
    wl = small_wl(seed=9, mask_layout=W.MASK_TREE_ONLY)
    check_dense(wl)


def test_layouts_agree_bitwise():
    a = small_wl(seed=11)
    b = small_wl(seed=11, mask_layout=W.MASK_TREE_ONLY)
    oa, la = oracle.mla_tree_verify(a)
    ob, lb = oracle.mla_tree_verify(b)
    assert np.array_equal(oa, ob) and np.array_equal(la, lb)


def test_dense_bruteforce_degenerate_requests():
    # zero-length prefix, single-node tree, star, chain, bs=4 ragged
    parents = [[W.ROOT], W.star_parents(6), W.chain_parents(7), [W.ROOT, 0, 1, 0]]
    wl = W.custom([0, 3, 50, 1], parents, 256, seed=3)
    check_dense(wl)


# ---------------------------------------------------------------- library routine

def test_chain_equals_sdpa_causal():
    wl = W.custom([90, 0, 33], [W.chain_parents(9), W.chain_parents(4), W.chain_parents(1)], 512,
                  seed=21)
    out, _ = oracle.mla_tree_verify(wl)
    H = wl.num_heads
    qop = wl.qo_indptr.numpy()
    for r in range(wl.bs):
        ref = pins.sdpa_chain(wl, r)
        got = out[qop[r] * H:qop[r + 1] * H]
        np.testing.assert_allclose(got, ref, rtol=1e-9, atol=1e-11)


# ---------------------------------------------------------------- invariants

def test_masked_key_never_changes_output():
    wl = small_wl(seed=5)
    out, lse = oracle.mla_tree_verify(wl)
    H = wl.num_heads
    qop = wl.qo_indptr.numpy()
    r = 1
    par = wl.parents[r]
    n = len(par)
    leaves = [t for t in range(n) if t not in par]
    t = leaves[0]
    slot = int(wl.out_cache_loc[qop[r] + t])
    pool2 = wl.kv_pool.clone()
    pool2[slot] = torch.randn(pool2.shape[1], generator=torch.Generator().manual_seed(1)).bfloat16() * 8
    out2, lse2 = oracle.mla_tree_verify(wl, kv_pool=pool2)
    row_t = slice((qop[r] + t) * H, (qop[r] + t + 1) * H)
    keep = np.ones(out.shape[0], dtype=bool)
    keep[row_t] = False
    assert np.array_equal(out[keep], out2[keep]) and np.array_equal(lse[keep], lse2[keep])
    assert not np.array_equal(out[row_t], out2[row_t])  # the leaf itself does see it


def test_prefix_columns_of_full_row_mask_are_ignored():
    wl = small_wl(seed=13)
    out, lse = oracle.mla_tree_verify(wl)
    m2 = wl.custom_mask.clone()
    mip = wl.mask_indptr.numpy()
    for r in range(wl.bs):
        p, n = wl.prefix_lens[r], wl.tree_sizes[r]
        blk = m2[mip[r]:mip[r + 1]].view(n, p + n)
        blk[:, :p] = torch.randint(0, 2, (n, p), dtype=torch.uint8)
    out2, lse2 = oracle.mla_tree_verify(wl, custom_mask=m2)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def test_slot_permutation_with_data_moved_is_exact():
    wl = small_wl(seed=17)
    out, lse = oracle.mla_tree_verify(wl)
    g = torch.Generator().manual_seed(99)
    perm = torch.randperm(wl.num_slots, generator=g)
    pool2 = torch.empty_like(wl.kv_pool)
    pool2[perm] = wl.kv_pool
    out2, lse2 = oracle.mla_tree_verify(wl, kv_pool=pool2, kv_indices=perm[wl.kv_indices],
                                        out_cache_loc=perm[wl.out_cache_loc])
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def test_constant_values_give_constant_output():
    wl = small_wl(seed=19)
    pool2 = wl.kv_pool.clone()
    pool2[:, :512] = 0.5
    out, _ = oracle.mla_tree_verify(wl, kv_pool=pool2)
    np.testing.assert_allclose(out, 0.5, rtol=0, atol=1e-14)


def test_empty_tree_row_is_plain_prefix_decode():
    wl = small_wl(seed=23)
    r, i = 0, 2
    m2 = wl.custom_mask.clone()
    mip = wl.mask_indptr.numpy()
    p, n = wl.prefix_lens[r], wl.tree_sizes[r]
    m2[mip[r] + i * (p + n) + p: mip[r] + (i + 1) * (p + n)] = 0
    out, lse = oracle.mla_tree_verify(wl, custom_mask=m2)
    # plain decode: softmax over the prefix keys only, computed by torch SDPA
    pool = torch.from_numpy(pins.bf16_to_f64(wl.kv_pool))
    keys = pool[wl.kv_indices[wl.kv_indptr[r]:wl.kv_indptr[r + 1]].long()]
    qi = torch.from_numpy(pins.bf16_to_f64(wl.q[int(wl.qo_indptr[r]) + i]))  # [H, 576]
    ref = torch.nn.functional.scaled_dot_product_attention(
        qi.unsqueeze(1), keys.unsqueeze(0).expand(64, -1, -1),
        keys[:, :512].unsqueeze(0).expand(64, -1, -1), scale=wl.scale).squeeze(1).numpy()
    ref_lse = torch.logsumexp(wl.scale * qi @ keys.T, dim=1).numpy()
    H = wl.num_heads
    row = slice((int(wl.qo_indptr[r]) + i) * H, (int(wl.qo_indptr[r]) + i + 1) * H)
    np.testing.assert_allclose(out[row], ref, rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(lse[row], ref_lse, rtol=1e-12, atol=1e-12)


def test_no_visible_key_gives_zero_and_minus_inf():
    parents = [[W.ROOT, 0]]
    wl = W.custom([0], parents, 64, seed=29)
    m2 = torch.zeros_like(wl.custom_mask)
    out, lse = oracle.mla_tree_verify(wl, custom_mask=m2)
    assert np.all(out == 0.0) and np.all(np.isneginf(lse))


# ---------------------------------------------------------------- closed forms

def test_self_only_without_prefix_closed_form():
    parents = [[W.ROOT, W.ROOT, W.ROOT]]  # all hang off the root; self only
    wl = W.custom([0], parents, 64, seed=31)
    out, lse = oracle.mla_tree_verify(wl)
    H = wl.num_heads
    pool = pins.bf16_to_f64(wl.kv_pool)
    q = pins.bf16_to_f64(wl.q)
    for i in range(3):
        slot = int(wl.out_cache_loc[i])
        np.testing.assert_array_equal(out[i * H:(i + 1) * H], np.broadcast_to(pool[slot, :512], (H, 512)))
        s = wl.scale * (q[i] @ pool[slot])
        np.testing.assert_allclose(lse[i * H:(i + 1) * H], s, rtol=1e-13, atol=1e-13)


def test_identical_keys_closed_form():
    wl = small_wl(seed=37)
    row = wl.kv_pool[0].clone()
    pool2 = row.unsqueeze(0).expand_as(wl.kv_pool).contiguous()
    out, lse = oracle.mla_tree_verify(wl, kv_pool=pool2)
    H = wl.num_heads
    k = pins.bf16_to_f64(row)
    q = pins.bf16_to_f64(wl.q)
    qop = wl.qo_indptr.numpy()
    for r in range(wl.bs):
        vis = pins.closure_visibility(wl.parents[r])
        for i in range(wl.tree_sizes[r]):
            cnt = wl.prefix_lens[r] + int(vis[i].sum())
            tok = qop[r] + i
            s = wl.scale * (q[tok] @ k)
            np.testing.assert_allclose(lse[tok * H:(tok + 1) * H], s + math.log(cnt), rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(out[tok * H:(tok + 1) * H], np.broadcast_to(k[:512], (H, 512)),
                                       rtol=1e-13, atol=1e-14)


# ---------------------------------------------------------------- exhaustive tiny trees

def test_every_five_node_tree_against_bruteforce():
    g = torch.Generator().manual_seed(41)
    pool = W.randn_bf16((96, W.D_QK), g)
    for choice in itertools.product(*[range(i + 1) for i in range(5)]):
        parents = [c - 1 for c in choice]
        wl = W.build_workload("enum", [11], [parents], 96, torch.Generator().manual_seed(7), pool=pool,
                              num_heads=2)
        check_dense(wl, tag=str(parents))


# ---------------------------------------------------------------- hand-derived worked example

@pytest.mark.parametrize("layout", [W.MASK_FULL_ROW, W.MASK_TREE_ONLY])
def test_hand_derived_worked_example(layout):
    """tests/golden/worked_example.json: small exact scores, outputs in closed
    form; pins the mask offset p_r + t, unread prefix columns, the rope dims,
    the scale and the natural-log LSE on a case checkable by hand."""
    wl, ref_out, ref_lse = pins.worked_example(layout)
    out, lse = oracle.mla_tree_verify(wl)
    np.testing.assert_allclose(lse, ref_lse, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(out, ref_out, rtol=1e-12, atol=1e-12)


def test_hand_derived_worked_example_full_row():
    test_hand_derived_worked_example(W.MASK_FULL_ROW)


# ---------------------------------------------------------------- lse combine

def test_lse_combine_equals_unsplit_softmax():
    rng = np.random.default_rng(3)
    nrows, nkeys, d, ns = 9, 40, 16, 4
    s = rng.normal(size=(nrows, nkeys)) * 3
    v = rng.normal(size=(nkeys, d))
    full_lse = torch.logsumexp(torch.from_numpy(s), 1).numpy()
    full = np.exp(s - full_lse[:, None]) @ v
    assign = rng.integers(0, ns, size=nkeys)
    assign[0] = ns - 1  # make split 0 possibly empty for some shapes
    o = np.zeros((ns, nrows, d))
    l = np.full((ns, nrows), -np.inf)
    for sp in range(ns):
        idx = np.nonzero(assign == sp)[0]
        if idx.size == 0:
            continue
        ls = torch.logsumexp(torch.from_numpy(s[:, idx]), 1).numpy()
        o[sp] = np.exp(s[:, idx] - ls[:, None]) @ v[idx]
        l[sp] = ls
    out, lse = oracle.lse_combine(o, l)
    np.testing.assert_allclose(lse, full_lse, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(out, full, rtol=1e-12, atol=1e-13)


def test_lse_combine_all_empty():
    out, lse = oracle.lse_combine(np.ones((3, 2, 4)), np.full((3, 2), -np.inf))
    assert np.all(out == 0) and np.all(np.isneginf(lse))


# ---------------------------------------------------------------- planted mistakes

MUTANTS = {
    "drop_rope_dims": ("for (int d = 0; d < dqk; ++d) acc +=", "for (int d = 0; d < J->d_latent; ++d) acc +="),
    "mask_offset_without_prefix": ("base + i * (p + n) + p + t", "base + i * (p + n) + t"),
    "mask_transposed": ("tree_visible(J, (int)r, i, t, p, n)", "tree_visible(J, (int)r, t, i, p, n)"),
    "missing_scale": ("scores[k] = J->scale * acc;", "scores[k] = acc;"),
    "lse_without_max": ("*lse_row = m + log(l);", "*lse_row = log(l);"),
    "prefix_of_request_zero": ("J->kv_indices[(int64_t)J->kv_indptr[r] + j]", "J->kv_indices[j]"),
    "values_from_rope_offset": ("out_row[d] += w * bf16_to_double(vrow[d]);",
                                "out_row[d] += w * bf16_to_double(vrow[d + J->d_rope]);"),
    "tree_slots_of_request_zero": ("slots[nk++] = J->out_cache_loc[J->qo_indptr[r] + t]",
                                   "slots[nk++] = J->out_cache_loc[t]"),
    "combine_weight_vs_max": ("double w = exp(lse_in[s * nrows + r] - L);",
                              "double w = exp(lse_in[s * nrows + r] - m);"),
}

PIN_FUNCS = [
    test_dense_bruteforce_random_trees, test_dense_bruteforce_degenerate_requests,
    test_chain_equals_sdpa_causal, test_self_only_without_prefix_closed_form,
    test_identical_keys_closed_form, test_lse_combine_equals_unsplit_softmax,
    test_hand_derived_worked_example_full_row,
]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name):
    src_path = os.path.join(os.path.dirname(oracle.__file__), "mla_tree_verify_oracle.c")
    src = open(src_path).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    with tempfile.TemporaryDirectory() as d:
        mpath = os.path.join(d, "mutant.c")
        open(mpath, "w").write(src.replace(old, new))
        lib = oracle.build(force=True, src=mpath, out=os.path.join(d, "libmutant.so"))
        caught = []
        with oracle.use_library(lib):
            for f in PIN_FUNCS:
                try:
                    f()
                except AssertionError:
                    caught.append(f.__name__)
    assert caught, f"no pin caught the planted mistake {name}"
