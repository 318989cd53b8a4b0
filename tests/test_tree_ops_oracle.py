"""Pins of the tree-step oracle (oracle/tree_ops.py) to things other than itself:
closed forms for chain and star trees, the reflexive-transitive closure of the
parent relation (Warshall), invariants, brute force over all root paths for
acceptance, a hand-derived worked example (tests/golden/tree_steps_example.json)
and planted mistakes that each pin must catch."""

import numpy as np
import pytest
import torch

from oracle import tree_ops as T
from paged_mla_speculative_tree_gb300 import workloads as W


def closure_mask(parents):
    """[n, n] reflexive-transitive closure of child -> parent (Warshall)."""
    n = len(parents)
    a = np.eye(n, dtype=bool)
    for i, p in enumerate(parents):
        if p != T.ROOT:
            a[i, p] = True
    for k in range(n):
        a |= a[:, k:k + 1] & a[k:k + 1, :]
    return a.astype(np.uint8)


def tree_part(mask, indptr, prefix_lens, sizes, layout, r):
    n, p = sizes[r], prefix_lens[r]
    w = p + n if layout == T.MASK_FULL_ROW else n
    blk = mask[indptr[r]:indptr[r + 1]].reshape(n, w)
    return blk[:, (p if layout == T.MASK_FULL_ROW else 0):], blk


def tree_steps_example():
    """tests/golden/tree_steps_example.json (visibility and the acceptance walk derived by hand)."""
    import json
    import os
    return json.load(open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                                       "tree_steps_example.json")))


def flat_golden_mask(rows_per_req):
    mask = np.array([b for rows in rows_per_req for row in rows for b in row], dtype=np.uint8)
    indptr = np.cumsum([0] + [len(rows) * len(rows[0]) for rows in rows_per_req]).astype(np.int64)
    return mask, indptr


def random_trees(seed, count, nmax):
    g = torch.Generator().manual_seed(seed)
    out = []
    for _ in range(count):
        n = int(torch.randint(1, nmax + 1, (1,), generator=g).item())
        out.append(W.random_parents(n, g))
    return out


# ---------------------------------------------------------------- mask pins
def mask_pins_hold(build):
    """Every mask pin, applied to a mask builder with tree_mask's signature."""
    ex = tree_steps_example()  # hand-derived rows
    for layout, key in ((T.MASK_FULL_ROW, "mask_full_row"), (T.MASK_TREE_ONLY, "mask_tree_only")):
        want, want_ip = flat_golden_mask(ex[key])
        got, got_ip = build(ex["parents"], ex["prefix_lens"], layout)
        if not (np.array_equal(got, want) and np.array_equal(got_ip, want_ip)):
            return False
    trees = random_trees(7, 12, 24) + [W.chain_parents(9), W.star_parents(7), [T.ROOT] * 5, [T.ROOT]]
    prefix = [int(x) for x in np.random.default_rng(3).integers(0, 40, len(trees))]
    sizes = [len(t) for t in trees]
    for layout in (T.MASK_FULL_ROW, T.MASK_TREE_ONLY):
        mask, indptr = build(trees, prefix, layout)
        widths = [(p + n) if layout == T.MASK_FULL_ROW else n for p, n in zip(prefix, sizes)]
        if list(np.diff(indptr)) != [n * w for n, w in zip(sizes, widths)]:
            return False
        for r, par in enumerate(trees):
            tp, blk = tree_part(mask, indptr, prefix, sizes, layout, r)
            if not np.array_equal(tp, closure_mask(par)):
                return False
            if layout == T.MASK_FULL_ROW and not np.all(blk[:, :prefix[r]] == 1):
                return False
    # closed forms
    for n in (1, 2, 8, 33):
        m, _ = build([W.chain_parents(n)], [0], T.MASK_TREE_ONLY)
        if not np.array_equal(m.reshape(n, n), np.tril(np.ones((n, n), dtype=np.uint8))):
            return False
        m, _ = build([W.star_parents(n)], [0], T.MASK_TREE_ONLY)
        want = np.eye(n, dtype=np.uint8)
        want[:, 0] = 1
        if not np.array_equal(m.reshape(n, n), want):
            return False
    return True


def test_mask_oracle_meets_its_pins():
    assert mask_pins_hold(T.tree_mask)


def test_mask_invariants_on_random_trees():
    for par in random_trees(11, 20, 40):
        m, _ = T.tree_mask([par], [0], T.MASK_TREE_ONLY)
        n = len(par)
        m = m.reshape(n, n)
        for i, p in enumerate(par):
            assert m[i, i] == 1
            depth = len(T.ancestors_or_self(par, i))
            assert int(m[i].sum()) == depth
            if p != T.ROOT:
                assert np.all(m[i] >= m[p])  # a node sees everything its parent sees
                assert m[i, p] == 1


@pytest.mark.parametrize("mutant", ["no_self", "parent_only", "prefix_zero", "off_by_one_column"])
def test_mask_pins_catch_planted_mistakes(mutant):
    def bad(trees, prefix, layout):
        mask, indptr = T.tree_mask(trees, prefix, layout)
        mask = mask.copy()
        for r, par in enumerate(trees):
            n, p = len(par), prefix[r]
            w = p + n if layout == T.MASK_FULL_ROW else n
            off = p if layout == T.MASK_FULL_ROW else 0
            blk = mask[indptr[r]:indptr[r + 1]].reshape(n, w)
            for i in range(n):
                if mutant == "no_self":
                    blk[i, off + i] = 0
                elif mutant == "parent_only":  # forgets the grand-ancestors
                    row = np.zeros(n, dtype=np.uint8)
                    row[i] = 1
                    if par[i] != T.ROOT:
                        row[par[i]] = 1
                    blk[i, off:] = row
                elif mutant == "prefix_zero" and layout == T.MASK_FULL_ROW and p > 0:
                    blk[i, 0] = 0
                elif mutant == "off_by_one_column" and i + 1 < n:
                    blk[i, off:] = np.roll(blk[i, off:], 1)
        return mask, indptr

    assert not mask_pins_hold(bad)


# ---------------------------------------------------------------- acceptance pins
def brute_force_accept(parents, draft, target, root_tok):
    """Deepest node whose whole root path was predicted token by token (unique
    when siblings carry distinct draft tokens)."""
    best = []
    for v in range(len(parents)):
        path = list(reversed(T.ancestors_or_self(parents, v)))
        want, ok = root_tok, True
        for u in path:
            if draft[u] != want:
                ok = False
                break
            want = target[u]
        if ok and len(path) > len(best):
            best = path
    bonus = target[best[-1]] if best else root_tok
    return best, bonus


def distinct_sibling_case(seed, n, vocab=5, hit=0.7):
    rng = np.random.default_rng(seed)
    g = torch.Generator().manual_seed(seed)
    par = W.random_parents(n, g)
    draft = [0] * n
    used = {}
    for i, p in enumerate(par):  # distinct tokens among siblings
        taken = used.setdefault(p, set())
        choices = [t for t in range(vocab + n) if t not in taken]
        draft[i] = int(rng.choice(choices))
        taken.add(draft[i])
    # the target agrees with some child of each node with probability `hit`
    children = {}
    for i, p in enumerate(par):
        children.setdefault(p, []).append(i)
    def predict(node):
        kids = children.get(node, [])
        if kids and rng.random() < hit:
            return draft[int(rng.choice(kids))]
        return int(rng.integers(1000, 2000))
    target = [predict(i) for i in range(n)]
    return par, draft, target, predict(T.ROOT)


def accept_pins_hold(accept):
    ex = tree_steps_example()  # hand-derived walk
    for r, exp in enumerate(ex["expected_accept"]):
        got = accept(ex["parents"][r], ex["draft_tokens"][r], ex["target_tokens"][r], ex["target_root_tokens"][r],
                     ex["out_cache_loc"][r])
        if list(got[0]) != exp["nodes"] or got[1] != exp["bonus"] or list(got[2]) != exp["slots"]:
            return False
    for seed in range(40):
        par, draft, target, root_tok = distinct_sibling_case(seed, 1 + seed % 17)
        slots = [100 + 3 * i for i in range(len(par))]
        path, bonus, sl = accept(par, draft, target, root_tok, slots)
        want_path, want_bonus = brute_force_accept(par, draft, target, root_tok)
        if path != want_path or bonus != want_bonus or sl != [100 + 3 * c for c in want_path]:
            return False
    # chain, every draft predicted: the whole chain is accepted
    n = 6
    par = W.chain_parents(n)
    draft = list(range(10, 10 + n))
    target = draft[1:] + [77]
    path, bonus, _ = accept(par, draft, target, 10, list(range(n)))
    if path != list(range(n)) or bonus != 77:
        return False
    # first token mispredicted: nothing accepted, bonus = the root prediction
    path, bonus, _ = accept(par, draft, target, 11, list(range(n)))
    if path != [] or bonus != 11:
        return False
    # duplicate sibling tokens: the lowest-index child wins
    par = [T.ROOT, T.ROOT, 1, 0]
    draft = [5, 5, 7, 7]
    target = [7, 7, 1, 2]
    path, bonus, _ = accept(par, draft, target, 5, [0, 1, 2, 3])
    return path == [0, 3] and bonus == 2


def test_accept_oracle_meets_its_pins():
    assert accept_pins_hold(T.tree_accept)


@pytest.mark.parametrize("mutant", ["highest_index", "skip_bonus", "wrong_prediction_index", "stop_after_one"])
def test_accept_pins_catch_planted_mistakes(mutant):
    def bad(parents, draft, target, root_tok, slots):
        n = len(parents)
        cur, want, path = T.ROOT, root_tok, []
        while True:
            order = range(n - 1, -1, -1) if mutant == "highest_index" else range(n)
            nxt = next((c for c in order if parents[c] == cur and draft[c] == want), None)
            if nxt is None:
                break
            path.append(nxt)
            cur = nxt
            want = target[parents[nxt]] if (mutant == "wrong_prediction_index" and parents[nxt] != T.ROOT) \
                else target[nxt]
            if mutant == "stop_after_one":
                break
        bonus = root_tok if mutant == "skip_bonus" else want
        return path, bonus, [slots[c] for c in path]

    assert not accept_pins_hold(bad)


# ---------------------------------------------------------------- defrag pins
def defrag_pins_hold(defrag):
    rng = np.random.default_rng(17)
    slots, width = 400, 6
    src = rng.integers(0, 1 << 16, (slots, width)).astype(np.uint16)
    dst0 = rng.integers(0, 1 << 16, (slots, width)).astype(np.uint16)
    prefix = [30, 0, 55, 7]
    perm = rng.permutation(slots)
    kv_indptr = np.array([0] + list(np.cumsum(prefix)))
    kv_indices = perm[:kv_indptr[-1]].astype(np.int64)
    dst_base = np.array([10, 60, 100, 300])
    out, idx = defrag(src, dst0, kv_indices, kv_indptr, dst_base)
    touched = np.zeros(slots, dtype=bool)
    for r, p in enumerate(prefix):
        k0 = kv_indptr[r]
        run = np.arange(dst_base[r], dst_base[r] + p)
        if not np.array_equal(idx[k0:k0 + p], run):  # indices become the contiguous run
            return False
        for j in range(p):  # each row of the run is the request's j-th prefix row
            if not np.array_equal(out[dst_base[r] + j], src[kv_indices[k0 + j]]):
                return False
        touched[run] = True
    if not np.array_equal(out[~touched], dst0[~touched]):  # nothing else changes
        return False
    # a prefix that already is the run at its base is left as it was (in place)
    same = src.copy()
    o2, i2 = defrag(same, same, np.arange(20, 50, dtype=np.int64), np.array([0, 30]), np.array([20]))
    return np.array_equal(o2, same) and np.array_equal(i2, np.arange(20, 50))


def test_defrag_oracle_meets_its_pins():
    assert defrag_pins_hold(T.kv_defrag)


@pytest.mark.parametrize("mutant", ["shifted_run", "indices_not_rewritten", "reversed_rows"])
def test_defrag_pins_catch_planted_mistakes(mutant):
    def bad(src, dst, kv_indices, kv_indptr, dst_base):
        out, idx = T.kv_defrag(src, dst, kv_indices, kv_indptr, dst_base)
        if mutant == "shifted_run":
            out, idx = T.kv_defrag(src, dst, kv_indices, kv_indptr, np.asarray(dst_base) + 1)
        elif mutant == "indices_not_rewritten":
            idx = np.array(kv_indices, copy=True)
        else:
            for r in range(len(dst_base)):
                k0, k1 = int(kv_indptr[r]), int(kv_indptr[r + 1])
                if k1 - k0 > 1:
                    run = np.arange(dst_base[r], dst_base[r] + k1 - k0)
                    out[run] = out[run[::-1]]
        return out, idx

    assert not defrag_pins_hold(bad)


# ---------------------------------------------------------------- shared-prefix grouping pins
def merged_workload(wl, group_indptr, grouping=None):
    import oracle  # noqa: F401  (fp64 attention oracle, used by the callers)
    grouping = grouping or T.group_prefix
    par_flat = [p for t in wl.parents for p in t]
    kvp, idx, qop, par, bad = grouping(group_indptr, wl.kv_indices.numpy(), wl.kv_indptr.numpy(),
                                       wl.qo_indptr.numpy(), par_flat)
    G = len(group_indptr) - 1
    trees = [list(par[qop[g]:qop[g + 1]]) for g in range(G)]
    prefix = [int(kvp[g + 1] - kvp[g]) for g in range(G)]
    mask, mip = T.tree_mask(trees, prefix, T.MASK_FULL_ROW)
    m = W.Workload(name=wl.name + "_merged", bs=G, prefix_lens=prefix, tree_sizes=[len(t) for t in trees],
                   parents=trees, q=wl.q, kv_pool=wl.kv_pool, kv_indices=torch.from_numpy(idx),
                   kv_indptr=torch.from_numpy(kvp), out_cache_loc=wl.out_cache_loc,
                   qo_indptr=torch.from_numpy(qop), custom_mask=torch.from_numpy(mask),
                   mask_indptr=torch.from_numpy(mip))
    return m, bad


def test_grouping_preserves_the_attention():
    import oracle
    g = torch.Generator().manual_seed(8)
    wl = W.shared_prefix(bs=5, prefix=150, tree=3, num_slots=1024, seed=9)
    ref_o, ref_l = oracle.mla_tree_verify(wl)
    for gi in ([0, 5], [0, 2, 5], [0, 1, 2, 3, 4, 5], [0, 3, 3, 5]):
        m, bad = merged_workload(wl, np.array(gi))
        assert not bad
        o, l = oracle.mla_tree_verify(m)
        assert np.max(np.abs(o - ref_o)) < 1e-9 and np.max(np.abs(l - ref_l)) < 1e-9


def test_grouping_identity_and_mismatch():
    wl = W.shared_prefix(bs=3, prefix=40, tree=2, num_slots=512, seed=10)
    par_flat = [p for t in wl.parents for p in t]
    kvp, idx, qop, par, bad = T.group_prefix(np.arange(4), wl.kv_indices.numpy(), wl.kv_indptr.numpy(),
                                             wl.qo_indptr.numpy(), par_flat)
    assert not bad and np.array_equal(kvp, wl.kv_indptr.numpy()) and np.array_equal(idx, wl.kv_indices.numpy())
    assert np.array_equal(qop, wl.qo_indptr.numpy()) and list(par) == par_flat
    other = W.custom([40, 40], [[T.ROOT], [T.ROOT]], 512, seed=11)  # two different prefixes
    *_, bad = T.group_prefix(np.array([0, 2]), other.kv_indices.numpy(), other.kv_indptr.numpy(),
                             other.qo_indptr.numpy(), [-1, -1])
    assert bad


def test_grouping_pin_catches_unshifted_parents():
    import oracle
    wl = W.shared_prefix(bs=3, prefix=64, tree=4, num_slots=512, seed=12)
    ref_o, _ = oracle.mla_tree_verify(wl)

    def bad(group_indptr, kv_indices, kv_indptr, qo_indptr, parents_flat):
        kvp, idx, qop, par, mis = T.group_prefix(group_indptr, kv_indices, kv_indptr, qo_indptr, parents_flat)
        return kvp, idx, qop, np.array(parents_flat, dtype=np.int32), mis  # forgets the shift

    m, _ = merged_workload(wl, np.array([0, 3]), grouping=bad)
    o, _ = oracle.mla_tree_verify(m)
    assert np.max(np.abs(o - ref_o)) > 1e-3


@pytest.mark.parametrize("layout", [T.MASK_FULL_ROW, T.MASK_TREE_ONLY])
def test_mask_oracle_matches_hand_derived_example(layout):
    ex = tree_steps_example()
    want, want_ip = flat_golden_mask(ex["mask_full_row" if layout == T.MASK_FULL_ROW else "mask_tree_only"])
    got, got_ip = T.tree_mask(ex["parents"], ex["prefix_lens"], layout)
    np.testing.assert_array_equal(got_ip, want_ip)
    np.testing.assert_array_equal(got, want)


def test_accept_oracle_matches_hand_derived_example():
    ex = tree_steps_example()
    for r, exp in enumerate(ex["expected_accept"]):
        path, bonus, slots = T.tree_accept(ex["parents"][r], ex["draft_tokens"][r], ex["target_tokens"][r],
                                           ex["target_root_tokens"][r], ex["out_cache_loc"][r])
        assert path == exp["nodes"] and bonus == exp["bonus"] and slots == exp["slots"]
