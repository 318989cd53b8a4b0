"""Host-side checks of the C ABI (no GPU needed): the library builds, loads and
exports every declared symbol; the plan struct layout matches the header; host
argument checks return the documented codes without touching a device."""
import ctypes
import os
import re
import subprocess
import tempfile

import pytest

from paged_mla_speculative_tree_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mla_tree_verify.h")


def declared_functions():
    names = []
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if h.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", h)).read()
            txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(mla_\w*)\s*\(", txt, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def test_library_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 5
    for n in names:
        assert hasattr(lib, n), n
    assert set(binding.SYMBOLS) <= set(names)


def test_plan_struct_layout_matches_header():
    prog = r'''
#include <stdio.h>
#include <stddef.h>
#include "mla_tree_verify.h"
int main(void) {
  printf("%zu %zu %zu %zu %zu\n", sizeof(mtv_plan_t), offsetof(mtv_plan_t, total_q_max),
         offsetof(mtv_plan_t, split_keys), offsetof(mtv_plan_t, ws_part_lse), offsetof(mtv_plan_t, reserved));
  return 0;
}'''
    with tempfile.TemporaryDirectory() as d:
        src = os.path.join(d, "l.c")
        exe = os.path.join(d, "l")
        open(src, "w").write(prog)
        subprocess.check_call(["gcc", "-I", os.path.join(ROOT, "include"), src, "-o", exe])
        vals = list(map(int, subprocess.check_output([exe]).split()))
    P = binding.MtvPlan
    assert vals == [ctypes.sizeof(P), P.total_q_max.offset, P.split_keys.offset,
                    P.ws_part_lse.offset, P.reserved.offset]


def test_strerror_covers_codes(lib):
    for code in range(0, -9, -1):
        assert binding.strerror(code) != "unknown error code"
    assert binding.strerror(-99) == "unknown error code"


def _plan_rc(lib, **kw):
    a = dict(device=0, bs=1, max_q=8, total_q=8, max_prefix=256, H=64, dl=512, dr=64, layout=0, flags=0,
             nsplit=0)
    a.update(kw)
    p = binding.MtvPlan()
    ws = ctypes.c_uint64()
    return lib.mla_tree_verify_plan(a["device"], a["bs"], a["max_q"], a["total_q"], a["max_prefix"], a["H"],
                                    a["dl"], a["dr"], a["layout"], a["flags"], a["nsplit"], ctypes.byref(p),
                                    ctypes.byref(ws))


def test_plan_rejects_bad_arguments_before_touching_a_device(lib):
    assert _plan_rc(lib, H=32) == -2
    assert _plan_rc(lib, dl=256) == -2
    assert _plan_rc(lib, dr=0) == -2
    assert _plan_rc(lib, layout=7) == -3
    assert _plan_rc(lib, bs=-1) == -3
    assert _plan_rc(lib, flags=0x10) == -3
    assert _plan_rc(lib, flags=0x200) == -3
    assert lib.mla_tree_verify_plan(0, 1, 8, 8, 256, 64, 512, 64, 0, 0, 0, None, None) == -1


def test_run_host_checks(lib):
    P = binding.MtvPlan()
    fake = ctypes.c_void_p(0x100000)  # never dereferenced: checks fail first
    # q, kv_pool, num_slots, kv_indices, len, kv_indptr, out_cache_loc, len, qo_indptr, custom_mask, len,
    # mask_indptr, scale, out, lse
    args = [fake, fake, 4096, fake, 64, fake, fake, 8, fake, fake, 64, fake, 1.0, fake, fake]
    # not a plan
    assert lib.mla_tree_verify_run(ctypes.byref(P), *args, fake, 1 << 20, None) == -6
    assert lib.mla_tree_verify_run(None, *args, fake, 1 << 20, None) == -1
    P.magic, P.version, P.bs, P.total_q_max, P.max_q_per_req, P.ws_bytes = \
        binding.PLAN_MAGIC, binding.ABI_VERSION, 1, 8, 8, 4096
    assert lib.mla_tree_verify_run(ctypes.byref(P), *args, ctypes.c_void_p(0x100010), 1 << 20, None) == -5
    assert lib.mla_tree_verify_run(ctypes.byref(P), *args, fake, 1024, None) == -4
    assert lib.mla_tree_verify_run(ctypes.byref(P), *args, None, 1 << 20, None) == -1
    nulls = list(args)
    nulls[0] = None  # q
    assert lib.mla_tree_verify_run(ctypes.byref(P), *nulls, fake, 1 << 20, None) == -1
    # buffer lengths: negative -> bad argument; NULL with a positive length -> null pointer;
    # NULL with length 0 is allowed (nothing may be read there)
    for i in (4, 7, 10):
        bad = list(args)
        bad[i] = -1
        assert lib.mla_tree_verify_run(ctypes.byref(P), *bad, fake, 1 << 20, None) == -3
        bad = list(args)
        bad[i - 1] = None
        assert lib.mla_tree_verify_run(ctypes.byref(P), *bad, fake, 1 << 20, None) == -1
    big = list(args)
    big[2] = 1 << 31  # num_slots past the 32-bit slot register of the gather
    assert lib.mla_tree_verify_run(ctypes.byref(P), *big, fake, 1 << 20, None) == -3
    assert lib.mla_tree_verify_clear_device_error(None, None) == -1
    v = ctypes.c_uint32()
    assert lib.mla_tree_verify_read_device_error(None, ctypes.byref(v), None) == -1
    assert lib.mla_tree_verify_read_static_device_error(None, None) == -1
    # run_steps: an empty or unknown step mask is a bad argument (checked before anything else runs)
    P.magic = binding.PLAN_MAGIC
    for steps in (0, 4, -1):
        assert lib.mla_tree_verify_run_steps(ctypes.byref(P), *args, fake, 1 << 20, steps, None) == -3
    # the static entry rejects a foreign plan before touching a device
    P.magic = 0
    assert lib.mla_tree_verify_run_static(ctypes.byref(P), *args, None) == -6


def _choose(lib, sms, prefix, tree, flags=0):
    import numpy as np
    pl = np.asarray(prefix, dtype=np.int64)
    ts = np.asarray(tree, dtype=np.int32)
    out = ctypes.c_int(-1)
    rc = lib.mla_tree_verify_choose_nsplit(sms, len(pl), pl.ctypes.data if len(pl) else None,
                                           ts.ctypes.data if len(ts) else None, flags, ctypes.byref(out))
    return rc, out.value


def test_choose_nsplit_argument_checks(lib):
    out = ctypes.c_int()
    assert lib.mla_tree_verify_choose_nsplit(152, 0, None, None, 0, None) == -1
    assert lib.mla_tree_verify_choose_nsplit(152, 1, None, None, 0, ctypes.byref(out)) == -1
    assert lib.mla_tree_verify_choose_nsplit(1, 0, None, None, 0, ctypes.byref(out)) == -3
    assert lib.mla_tree_verify_choose_nsplit(152, -1, None, None, 0, ctypes.byref(out)) == -3
    assert _choose(lib, 152, [100], [4], flags=0x10)[0] == -3
    assert _choose(lib, 152, [-1], [4])[0] == -3
    assert _choose(lib, 152, [100], [-4])[0] == -3
    assert _choose(lib, 152, [], []) == (0, 1)            # nothing to split
    assert _choose(lib, 152, [5000, 7000], [0, 0]) == (0, 1)  # no query rows


def test_choose_nsplit_uniform_batches_keep_the_plan_rule(lib):
    # the counts the plan's automatic rule gives these shapes on 152 SMs (the
    # measured best of split-count sweeps on a GB300)
    assert _choose(lib, 152, [32768], [32]) == (0, 9)            # Long
    assert _choose(lib, 152, [5760] * 4, [16] * 4) == (0, 2)     # Batch-4
    assert _choose(lib, 152, [131072] * 16, [64] * 16) == (0, 4)  # Stress
    assert _choose(lib, 152, [131072] * 2, [64] * 2) == (0, 7)   # the Stress request shape, 2 requests


def test_choose_nsplit_ragged_batches(lib):
    from paged_mla_speculative_tree_gb300 import workloads as W
    got = {}
    for seed in (1004, 2004, 3004):
        wl = W.mixed(seed=seed)
        rc, ns = _choose(lib, 152, wl.prefix_lens, wl.tree_sizes)
        assert rc == 0 and 1 <= ns <= 64
        got[seed] = ns
    # seeds 2004 and 3004 measured fastest at 1 and 4-6 splits (the rule from
    # upper bounds alone picks 3 and 2)
    assert got == {1004: 3, 2004: 1, 3004: 4}
    # a lone long request among short ones is split to spread its keys
    rc, ns = _choose(lib, 152, [200000] + [2000] * 15, [8] * 16)
    assert rc == 0 and ns > 1
    # the SIMT floor keeps its own rule
    assert _choose(lib, 152, [32768], [32], flags=0x1)[0] == 0


def test_tree_ops_host_checks(lib):
    fake = ctypes.c_void_p(0x100000)  # never dereferenced: checks fail first
    # mla_tree_mask_build(parents, qo_indptr, kv_indptr, bs, max_q, layout, mask, cap, mask_indptr, err, stream)
    assert lib.mla_tree_mask_build(fake, fake, fake, -1, 8, 0, fake, 64, fake, None, None) == -3
    assert lib.mla_tree_mask_build(fake, fake, fake, 1, -1, 0, fake, 64, fake, None, None) == -3
    assert lib.mla_tree_mask_build(fake, fake, fake, 1, 8, 7, fake, 64, fake, None, None) == -3
    assert lib.mla_tree_mask_build(fake, fake, fake, 1, 8, 0, fake, 64, None, None, None) == -1
    assert lib.mla_tree_mask_build(fake, fake, fake, 1, 1 << 16, 0, fake, 64, fake, None, None) == -2
    assert lib.mla_tree_mask_build(fake, None, fake, 1, 8, 0, fake, 64, fake, None, None) == -1
    assert lib.mla_tree_mask_build(fake, fake, None, 1, 8, 0, fake, 64, fake, None, None) == -1  # FULL_ROW needs p
    # mla_tree_accept(parents, draft, target, root, ocl, qo_indptr, bs, max_q, len, nodes, slots, bonus, err, s)
    args = [fake] * 6
    outs = [fake] * 4
    assert lib.mla_tree_accept(*args, -1, 8, *outs, None, None) == -3
    assert lib.mla_tree_accept(*args, 1, -2, *outs, None, None) == -3
    assert lib.mla_tree_accept(*args, 0, 8, *outs, None, None) == 0  # nothing to do, nothing launched
    assert lib.mla_tree_accept(fake, fake, fake, None, fake, fake, 1, 8, *outs, None, None) == -1
    assert lib.mla_tree_accept(*args, 1, 8, fake, None, fake, fake, None, None) == -1


def test_kv_defrag_host_checks(lib):
    fake = ctypes.c_void_p(0x100000)
    odd = ctypes.c_void_p(0x100008)
    # mla_kv_defrag(src, dst, num_slots, kv_indices, kv_indptr, bs, max_prefix, dst_base, out, err, stream)
    assert lib.mla_kv_defrag(fake, fake, 10, fake, fake, -1, 8, fake, fake, None, None) == -3
    assert lib.mla_kv_defrag(fake, fake, 10, fake, fake, 1, -1, fake, fake, None, None) == -3
    assert lib.mla_kv_defrag(fake, fake, 10, fake, fake, 0, 8, fake, fake, None, None) == 0
    assert lib.mla_kv_defrag(None, fake, 10, fake, fake, 1, 8, fake, fake, None, None) == -1
    assert lib.mla_kv_defrag(fake, fake, 10, fake, fake, 1, 8, None, fake, None, None) == -1
    assert lib.mla_kv_defrag(odd, fake, 10, fake, fake, 1, 8, fake, fake, None, None) == -3


def test_group_prefix_host_checks(lib):
    fake = ctypes.c_void_p(0x100000)
    # mla_tree_group_prefix(group_indptr, G, max_prefix, kv_indices, kv_indptr, qo_indptr, parents,
    #                       kv_indptr_out, kv_indices_out, qo_indptr_out, parents_out, err, stream)
    f7 = [fake] * 4
    assert lib.mla_tree_group_prefix(fake, -1, 8, *f7, *f7, None, None) == -3
    assert lib.mla_tree_group_prefix(fake, 1, -1, *f7, *f7, None, None) == -3
    assert lib.mla_tree_group_prefix(fake, 0, 8, *f7, *f7, None, None) == 0
    assert lib.mla_tree_group_prefix(None, 1, 8, *f7, *f7, None, None) == -1
    assert lib.mla_tree_group_prefix(fake, 1, 8, *f7, fake, fake, fake, None, None, None) == -1
