"""GPU parity of the tree steps (mask build, acceptance) against oracle/tree_ops.py,
through the C ABI: mask bytes and indptr bit-exact, acceptance results exact."""
import numpy as np
import pytest
import torch

from oracle import tree_ops as T
from paged_mla_speculative_tree_gb300 import binding, workloads as W
import oracle
from tests.gpu_util import compare, run_gpu, to_device
from tests.test_tree_ops_oracle import distinct_sibling_case, flat_golden_mask, random_trees, tree_steps_example

pytestmark = pytest.mark.gpu


def flat_parents(trees):
    return torch.tensor([p for t in trees for p in t], dtype=torch.int32)


def build_on_gpu(trees, prefix, layout, capacity=None, max_q=None):
    sizes = [len(t) for t in trees]
    qo = torch.tensor([0] + list(np.cumsum(sizes)), dtype=torch.int64).cuda()
    kv = torch.tensor([0] + list(np.cumsum(prefix)), dtype=torch.int32).cuda()
    need = sum(n * ((p + n) if layout == T.MASK_FULL_ROW else n) for p, n in zip(prefix, sizes))
    cap = need if capacity is None else capacity
    mask = torch.full((max(cap, 1),), 7, dtype=torch.uint8, device="cuda")[:cap]
    indptr = torch.full((len(trees) + 1,), -5, dtype=torch.int64, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.tree_mask_build(flat_parents(trees).cuda(), qo, kv, len(trees), max_q or max(sizes + [0]), layout,
                            mask, indptr, err)
    torch.cuda.synchronize()
    return mask.cpu().numpy(), indptr.cpu().numpy(), int(err.item())


@pytest.mark.parametrize("layout", [T.MASK_FULL_ROW, T.MASK_TREE_ONLY])
def test_mask_random_trees_bit_exact(layout):
    trees = random_trees(21, 24, 70) + [W.chain_parents(64), W.star_parents(40), [T.ROOT] * 3, [T.ROOT]]
    prefix = [int(x) for x in np.random.default_rng(5).integers(0, 300, len(trees))]
    mask, indptr, err = build_on_gpu(trees, prefix, layout)
    want, want_ip = T.tree_mask(trees, prefix, layout)
    assert err == 0
    np.testing.assert_array_equal(indptr, want_ip)
    np.testing.assert_array_equal(mask, want)


@pytest.mark.parametrize("name", ["tiny", "batch4", "mixed"])
def test_mask_of_named_workloads_equals_generator_mask(name):
    wl = W.WORKLOADS[name]()
    mask, indptr, err = build_on_gpu(wl.parents, wl.prefix_lens, wl.mask_layout)
    assert err == 0
    np.testing.assert_array_equal(indptr, wl.mask_indptr.numpy())
    np.testing.assert_array_equal(mask, wl.custom_mask.numpy())


def test_mask_stress_shape_bit_exact():
    """Stress shape: 16 requests x 64 rows x (131,072 + 64) columns (134 MB)."""
    g = torch.Generator().manual_seed(5005)
    trees = [W.random_parents(64, g) for _ in range(16)]
    prefix = [131072] * 16
    mask, indptr, err = build_on_gpu(trees, prefix, T.MASK_FULL_ROW)
    want, want_ip = T.tree_mask(trees, prefix, T.MASK_FULL_ROW)
    assert err == 0
    np.testing.assert_array_equal(indptr, want_ip)
    np.testing.assert_array_equal(mask, want)


def test_built_mask_drives_verify_attention():
    wl = W.WORKLOADS["mixed"]()
    mask, indptr, err = build_on_gpu(wl.parents, wl.prefix_lens, wl.mask_layout)
    assert err == 0
    d = to_device(wl)
    o_ref, l_ref = run_gpu(wl, dev_tensors=d)
    d["custom_mask"] = torch.from_numpy(mask).cuda()
    d["mask_indptr"] = torch.from_numpy(indptr).cuda()
    o, l = run_gpu(wl, dev_tensors=d)
    np.testing.assert_array_equal(o, o_ref)
    np.testing.assert_array_equal(l, l_ref)


def test_mask_edges_empty_tree_zero_prefix_unaligned_rows():
    trees = [[], [T.ROOT], [T.ROOT, 0, 1], [], [T.ROOT, T.ROOT]]
    prefix = [5, 0, 13, 0, 1]
    for layout in (T.MASK_FULL_ROW, T.MASK_TREE_ONLY):
        mask, indptr, err = build_on_gpu(trees, prefix, layout, max_q=8)
        want, want_ip = T.tree_mask(trees, prefix, layout)
        assert err == 0
        np.testing.assert_array_equal(indptr, want_ip)
        np.testing.assert_array_equal(mask, want)


def test_mask_capacity_and_bad_parent_are_flagged():
    trees = [W.chain_parents(4), W.chain_parents(4)]
    prefix = [3, 3]
    mask, indptr, err = build_on_gpu(trees, prefix, T.MASK_FULL_ROW, capacity=4 * 7 + 5)
    assert err & binding.DEVERR_INDPTR
    np.testing.assert_array_equal(indptr, [0, 28, 56])  # sizes are still published
    want, _ = T.tree_mask(trees[:1], prefix[:1], T.MASK_FULL_ROW)
    np.testing.assert_array_equal(mask[:28], want)  # the request that fits is written
    bad = [[T.ROOT, 5, 0]]  # node 1 names a later node as parent
    mask, indptr, err = build_on_gpu(bad, [2], T.MASK_TREE_ONLY)
    assert err & binding.DEVERR_PARENT
    fixed = [[T.ROOT, T.ROOT, 0]]  # read as hanging off the prefix
    np.testing.assert_array_equal(mask, T.tree_mask(fixed, [2], T.MASK_TREE_ONLY)[0])


def accept_on_gpu(cases, max_q):
    par = torch.tensor([p for c in cases for p in c[0]], dtype=torch.int32).cuda()
    draft = torch.tensor([t for c in cases for t in c[1]], dtype=torch.int32).cuda()
    target = torch.tensor([t for c in cases for t in c[2]], dtype=torch.int32).cuda()
    root = torch.tensor([c[3] for c in cases], dtype=torch.int32).cuda()
    sizes = [len(c[0]) for c in cases]
    qo = torch.tensor([0] + list(np.cumsum(sizes)), dtype=torch.int64).cuda()
    slots = torch.arange(1000, 1000 + int(qo[-1].item()), dtype=torch.int64).cuda() * 3
    bs = len(cases)
    alen = torch.full((bs,), -9, dtype=torch.int32, device="cuda")
    nodes = torch.full((bs, max_q), -9, dtype=torch.int32, device="cuda")
    aslots = torch.full((bs, max_q), -9, dtype=torch.int64, device="cuda")
    bonus = torch.full((bs,), -9, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.tree_accept(par, draft, target, root, slots, qo, bs, max_q, alen, nodes, aslots, bonus, err)
    torch.cuda.synchronize()
    return (alen.cpu().numpy(), nodes.cpu().numpy(), aslots.cpu().numpy(), bonus.cpu().numpy(),
            int(err.item()), slots.cpu().numpy(), qo.cpu().numpy())


def test_accept_matches_oracle():
    cases = [distinct_sibling_case(s, 1 + (7 * s) % 70, hit=0.5 + 0.5 * (s % 3) / 2) for s in range(48)]
    cases.append(([T.ROOT, T.ROOT, 1, 0], [5, 5, 7, 7], [7, 7, 1, 2], 5))  # duplicate sibling tokens
    n = 9
    cases.append((W.chain_parents(n), list(range(10, 10 + n)), list(range(11, 11 + n - 1)) + [99], 10))
    cases.append(([], [], [], 42))  # empty tree
    max_q = max(len(c[0]) for c in cases)
    alen, nodes, aslots, bonus, err, slots, qo = accept_on_gpu(cases, max_q)
    assert err == 0
    for r, (par, draft, target, root) in enumerate(cases):
        s = slots[qo[r]:qo[r + 1]]
        path, b, sl = T.tree_accept(par, draft, target, root, s)
        assert alen[r] == len(path)
        assert list(nodes[r, :len(path)]) == path and np.all(nodes[r, len(path):] == -1)
        assert list(aslots[r, :len(path)]) == sl and np.all(aslots[r, len(path):] == -1)
        assert bonus[r] == b


@pytest.mark.parametrize("layout", [T.MASK_FULL_ROW, T.MASK_TREE_ONLY])
def test_tree_steps_hand_derived_example(layout):
    # tests/golden/tree_steps_example.json: mask rows and the acceptance walk derived by hand
    ex = tree_steps_example()
    mask, indptr, err = build_on_gpu(ex["parents"], ex["prefix_lens"], layout)
    want, want_ip = flat_golden_mask(ex["mask_full_row" if layout == T.MASK_FULL_ROW else "mask_tree_only"])
    assert err == 0
    np.testing.assert_array_equal(indptr, want_ip)
    np.testing.assert_array_equal(mask, want)
    bs, max_q = len(ex["parents"]), max(len(p) for p in ex["parents"])
    flat = lambda key, dt: torch.tensor([v for per in ex[key] for v in per], dtype=dt).cuda()
    sizes = [len(p) for p in ex["parents"]]
    qo = torch.tensor([0] + list(np.cumsum(sizes)), dtype=torch.int64).cuda()
    alen = torch.full((bs,), -9, dtype=torch.int32, device="cuda")
    nodes = torch.full((bs, max_q), -9, dtype=torch.int32, device="cuda")
    aslots = torch.full((bs, max_q), -9, dtype=torch.int64, device="cuda")
    bonus = torch.full((bs,), -9, dtype=torch.int32, device="cuda")
    aerr = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.tree_accept(flat("parents", torch.int32), flat("draft_tokens", torch.int32),
                        flat("target_tokens", torch.int32),
                        torch.tensor(ex["target_root_tokens"], dtype=torch.int32).cuda(),
                        flat("out_cache_loc", torch.int64), qo, bs, max_q, alen, nodes, aslots, bonus, aerr)
    torch.cuda.synchronize()
    assert int(aerr.item()) == 0
    for r, exp in enumerate(ex["expected_accept"]):
        k = len(exp["nodes"])
        assert int(alen[r]) == k and int(bonus[r]) == exp["bonus"]
        assert nodes[r, :k].tolist() == exp["nodes"] and aslots[r, :k].tolist() == exp["slots"]
        assert bool((nodes[r, k:] == -1).all()) and bool((aslots[r, k:] == -1).all())


def test_tree_ops_capture_and_replay():
    wl = W.WORKLOADS["batch4"]()
    trees, prefix = wl.parents, wl.prefix_lens
    sizes = [len(t) for t in trees]
    par = flat_parents(trees).cuda()
    qo = wl.qo_indptr.cuda()
    kv = wl.kv_indptr.cuda()
    mask = torch.zeros(wl.custom_mask.numel(), dtype=torch.uint8, device="cuda")
    indptr = torch.zeros(wl.bs + 1, dtype=torch.int64, device="cuda")
    g = torch.Generator().manual_seed(9)
    draft = torch.randint(0, 3, (sum(sizes),), generator=g, dtype=torch.int32).cuda()
    target = torch.randint(0, 3, (sum(sizes),), generator=g, dtype=torch.int32).cuda()
    root = torch.randint(0, 3, (wl.bs,), generator=g, dtype=torch.int32).cuda()
    ocl = wl.out_cache_loc.cuda()
    mq = max(sizes)
    alen = torch.zeros(wl.bs, dtype=torch.int32, device="cuda")
    nodes = torch.zeros((wl.bs, mq), dtype=torch.int32, device="cuda")
    aslots = torch.zeros((wl.bs, mq), dtype=torch.int64, device="cuda")
    bonus = torch.zeros(wl.bs, dtype=torch.int32, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # warm-up outside capture
        binding.tree_mask_build(par, qo, kv, wl.bs, mq, wl.mask_layout, mask, indptr, stream=s)
        binding.tree_accept(par, draft, target, root, ocl, qo, wl.bs, mq, alen, nodes, aslots, bonus, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        binding.tree_mask_build(par, qo, kv, wl.bs, mq, wl.mask_layout, mask, indptr)
        binding.tree_accept(par, draft, target, root, ocl, qo, wl.bs, mq, alen, nodes, aslots, bonus)
    mask.zero_()
    alen.fill_(-1)
    graph.replay()
    torch.cuda.synchronize()
    np.testing.assert_array_equal(mask.cpu().numpy(), wl.custom_mask.numpy())
    np.testing.assert_array_equal(indptr.cpu().numpy(), wl.mask_indptr.numpy())
    d, t, rt = draft.cpu().tolist(), target.cpu().tolist(), root.cpu().tolist()
    qh = wl.qo_indptr.tolist()
    for r in range(wl.bs):
        path, b, _ = T.tree_accept(trees[r], d[qh[r]:qh[r + 1]], t[qh[r]:qh[r + 1]], rt[r],
                                   wl.out_cache_loc[qh[r]:qh[r + 1]].tolist())
        assert int(alen[r]) == len(path) and int(bonus[r]) == b


def defrag_on_gpu(src, dst, kv_indices, kv_indptr, dst_base, max_prefix, out_alias=False):
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    idx_out = kv_indices if out_alias else torch.full_like(kv_indices, -7)
    binding.kv_defrag(src, dst, kv_indices, kv_indptr, len(dst_base), max_prefix, dst_base, idx_out, err)
    torch.cuda.synchronize()
    return idx_out, int(err.item())


def test_defrag_long_random_bit_exact_and_attention_unchanged():
    wl = W.WORKLOADS["long_random"]()
    d = to_device(wl)
    o_ref, l_ref = run_gpu(wl, dev_tensors=d)
    dst = torch.zeros_like(d["kv_pool"])
    base = 1000
    idx, err = defrag_on_gpu(d["kv_pool"], dst, d["kv_indices"], d["kv_indptr"],
                             torch.tensor([base], dtype=torch.int64, device="cuda"), wl.max_prefix)
    assert err == 0
    src16 = wl.kv_pool.view(torch.int16).numpy()
    want_pool, want_idx = T.kv_defrag(src16, np.zeros_like(src16), wl.kv_indices.numpy(), wl.kv_indptr.numpy(),
                                      [base])
    np.testing.assert_array_equal(idx.cpu().numpy(), want_idx)
    np.testing.assert_array_equal(dst.view(torch.int16).cpu().numpy(), want_pool)
    # move the tree tokens right after the prefix run, then verify reads only the new pool
    p = wl.prefix_lens[0]
    new_ocl = torch.arange(base + p, base + p + wl.total_q, dtype=torch.int64, device="cuda")
    dst[new_ocl] = d["kv_pool"][d["out_cache_loc"]]
    d2 = dict(d, kv_pool=dst, kv_indices=idx, out_cache_loc=new_ocl)
    o, l = run_gpu(wl, dev_tensors=d2)
    np.testing.assert_array_equal(o, o_ref)
    np.testing.assert_array_equal(l, l_ref)


def test_defrag_in_place_ragged_batch_and_aliased_indices():
    g = torch.Generator().manual_seed(31)
    pool = W.randn_bf16((4096, 576), g).cuda()
    prefix = [100, 0, 333, 1]
    slots = torch.randperm(2048, generator=g)[:sum(prefix)].to(torch.int64)  # sources in [0, 2048)
    indptr = torch.tensor([0] + list(np.cumsum(prefix)), dtype=torch.int32)
    starts = [2048, 2500, 3000, 3500]  # destinations in the free half
    before = pool.view(torch.int16).cpu().numpy()
    idx = slots.clone().cuda()
    out_idx, err = defrag_on_gpu(pool, pool, idx, indptr.cuda(), torch.tensor(starts, dtype=torch.int64).cuda(),
                                 max(prefix), out_alias=True)
    assert err == 0
    want_pool, want_idx = T.kv_defrag(before, before, slots.numpy(), indptr.numpy(), starts)
    np.testing.assert_array_equal(out_idx.cpu().numpy(), want_idx)
    np.testing.assert_array_equal(pool.view(torch.int16).cpu().numpy(), want_pool)


def test_defrag_out_of_range_slots_are_flagged():
    pool = torch.randn(64, 576).to(torch.bfloat16).cuda()
    dst = torch.zeros_like(pool)
    idx = torch.tensor([3, 99, 5], dtype=torch.int64, device="cuda")
    indptr = torch.tensor([0, 3], dtype=torch.int32, device="cuda")
    out, err = defrag_on_gpu(pool, dst, idx, indptr, torch.tensor([10], dtype=torch.int64, device="cuda"), 3)
    assert err & binding.DEVERR_SLOT_RANGE
    o = out.cpu().tolist()
    assert o[0] == 10 and o[1] == -7 and o[2] == 12  # the bad row keeps its index slot unwritten
    assert torch.equal(dst[10], pool[3]) and torch.equal(dst[12], pool[5]) and not dst[11].any()


def group_on_gpu(wl, group_indptr):
    dev = "cuda"
    gi = torch.tensor(group_indptr, dtype=torch.int32, device=dev)
    G = len(group_indptr) - 1
    par = flat_parents(wl.parents).to(dev)
    kvp = torch.full((G + 1,), -5, dtype=torch.int32, device=dev)
    lead_total = sum(wl.prefix_lens[group_indptr[g]] for g in range(G) if group_indptr[g + 1] > group_indptr[g])
    idx = torch.full((max(lead_total, 1),), -5, dtype=torch.int64, device=dev)[:lead_total]
    qop = torch.full((G + 1,), -5, dtype=torch.int64, device=dev)
    parout = torch.full_like(par, -9)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    binding.tree_group_prefix(gi, G, max(wl.prefix_lens), wl.kv_indices.to(dev), wl.kv_indptr.to(dev),
                              wl.qo_indptr.to(dev), par, kvp, idx, qop, parout, err)
    torch.cuda.synchronize()
    return kvp, idx, qop, parout, int(err.item())


@pytest.mark.parametrize("groups", [[0, 16], [0, 8, 16], [0, 1, 5, 5, 16], list(range(17))])
def test_group_prefix_matches_oracle(groups):
    wl = W.WORKLOADS["shared_tree3"]()
    kvp, idx, qop, par, err = group_on_gpu(wl, groups)
    want = T.group_prefix(np.array(groups), wl.kv_indices.numpy(), wl.kv_indptr.numpy(), wl.qo_indptr.numpy(),
                          [p for t in wl.parents for p in t])
    assert err == 0 and not want[4]
    np.testing.assert_array_equal(kvp.cpu().numpy(), want[0])
    np.testing.assert_array_equal(idx.cpu().numpy(), want[1])
    np.testing.assert_array_equal(qop.cpu().numpy(), want[2])
    np.testing.assert_array_equal(par.cpu().numpy(), want[3])


@pytest.mark.parametrize("name", ["shared_decode", "shared_tree3"])
def test_grouped_verify_matches_oracle_of_the_original_requests(name):
    """group -> mask build -> verify on the merged requests, against the
    oracle on the original (ungrouped) requests."""
    wl = W.WORKLOADS[name]()
    kvp, idx, qop, par, err = group_on_gpu(wl, [0, wl.bs])
    assert err == 0
    n_merged = wl.total_q
    width = wl.prefix_lens[0] + n_merged
    mask = torch.zeros(n_merged * width, dtype=torch.uint8, device="cuda")
    mip = torch.zeros(2, dtype=torch.int64, device="cuda")
    merr = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.tree_mask_build(par, qop, kvp, 1, n_merged, binding.MASK_FULL_ROW, mask, mip, merr)
    torch.cuda.synchronize()
    assert int(merr.item()) == 0
    d = to_device(wl)
    d.update(kv_indices=idx, kv_indptr=kvp, qo_indptr=qop, custom_mask=mask, mask_indptr=mip)
    merged = W.Workload(name=wl.name + "_merged", bs=1, prefix_lens=[wl.prefix_lens[0]], tree_sizes=[n_merged],
                        parents=[par.cpu().tolist()], q=wl.q, kv_pool=wl.kv_pool, kv_indices=idx.cpu(),
                        kv_indptr=kvp.cpu(), out_cache_loc=wl.out_cache_loc, qo_indptr=qop.cpu(),
                        custom_mask=mask.cpu(), mask_indptr=mip.cpu())
    out, lse = run_gpu(merged, dev_tensors=d)
    rows = np.arange(0, wl.total_q * 64, 7)
    ref = oracle.mla_tree_verify(wl, rows=rows)
    compare(wl, out, lse, rows=rows, ref=ref, tag=name + " grouped")


def test_group_prefix_mismatch_is_flagged():
    wl = W.custom([30, 30, 31], [[T.ROOT], [T.ROOT, 0], [T.ROOT]], 512, seed=3)  # three different prefixes
    kvp, idx, qop, par, err = group_on_gpu(wl, [0, 3])
    assert err & binding.DEVERR_PREFIX
    np.testing.assert_array_equal(kvp.cpu().numpy(), [0, 30])  # the leader's prefix is used
    np.testing.assert_array_equal(idx.cpu().numpy(), wl.kv_indices[:30].numpy())
