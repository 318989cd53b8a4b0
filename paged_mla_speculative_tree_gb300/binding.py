"""ctypes binding of the C ABI in ``include/mla_tree_verify.h``.

Argument marshalling only: every step of the verify attention runs in the CUDA
library.  There is no fallback -- if the library is missing this raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

MTV_OK = 0
MASK_FULL_ROW = 0
MASK_TREE_ONLY = 1
FLAG_SIMT_FLOOR = 0x1
FLAG_TEST_SHORT_WAITS = 0x100  # test only: pipeline waits give up at once (timeout path)
STEP_PARTIAL = 0x1
STEP_COMBINE = 0x2
DEVERR_SLOT_RANGE = 0x1
DEVERR_INDPTR = 0x2
DEVERR_TIMEOUT = 0x4
DEVERR_PARENT = 0x8
DEVERR_PREFIX = 0x10
PLAN_MAGIC = 0x4D545650
ABI_VERSION = 2


class MtvPlan(ctypes.Structure):
    _fields_ = [
        ("magic", ctypes.c_uint32), ("version", ctypes.c_uint32),
        ("device", ctypes.c_int32), ("num_sms", ctypes.c_int32),
        ("cc_major", ctypes.c_int32), ("cc_minor", ctypes.c_int32),
        ("bs", ctypes.c_int32), ("max_q_per_req", ctypes.c_int32), ("num_heads", ctypes.c_int32),
        ("d_latent", ctypes.c_int32), ("d_rope", ctypes.c_int32), ("mask_layout", ctypes.c_int32),
        ("flags", ctypes.c_int32), ("row_tile", ctypes.c_int32), ("key_tile", ctypes.c_int32),
        ("nsplit", ctypes.c_int32), ("grid_rows", ctypes.c_int32), ("reserved0", ctypes.c_int32),
        ("total_q_max", ctypes.c_int64), ("max_prefix", ctypes.c_int64),
        ("split_keys", ctypes.c_int64), ("ws_bytes", ctypes.c_uint64),
        ("ws_part_o", ctypes.c_uint64), ("ws_part_lse", ctypes.c_uint64),
        ("reserved", ctypes.c_int64 * 6),
    ]

    def as_dict(self):
        return {f: getattr(self, f) for f, _ in self._fields_ if not f.startswith("reserved")}


class MtvError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {strerror(code)} (code {code})")
        self.code = code


_lib = None
SYMBOLS = ("mla_tree_verify_plan", "mla_tree_verify_choose_nsplit", "mla_tree_verify_run", "mla_tree_verify_run_steps", "mla_tree_verify_strerror",
           "mla_tree_verify_clear_device_error", "mla_tree_verify_read_device_error",
           "mla_tree_verify_run_static", "mla_tree_verify_read_static_device_error", "mla_tree_mask_build", "mla_tree_accept", "mla_kv_defrag",
           "mla_tree_group_prefix")


def library_path() -> str:
    return _build.LIB


def load(path: str | None = None):
    """Loads the CUDA library (building it first if sources are newer)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    path = path or library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library not built: {path} (run __graft_entry__.build())")
    lib = ctypes.CDLL(path)
    P, I32, I64, U64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_uint64
    lib.mla_tree_verify_plan.argtypes = [I32, I32, I32, I64, I64, I32, I32, I32, I32, I32, I32,
                                         ctypes.POINTER(MtvPlan), ctypes.POINTER(U64)]
    lib.mla_tree_verify_plan.restype = I32
    lib.mla_tree_verify_choose_nsplit.argtypes = [I32, I32, P, P, I32, ctypes.POINTER(I32)]
    lib.mla_tree_verify_choose_nsplit.restype = I32
    lib.mla_tree_verify_run.argtypes = [ctypes.POINTER(MtvPlan), P, P, I64, P, I64, P, P, I64, P, P, I64, P,
                                        ctypes.c_float, P, P, P, U64, P]
    lib.mla_tree_verify_run.restype = I32
    lib.mla_tree_verify_run_steps.argtypes = [ctypes.POINTER(MtvPlan), P, P, I64, P, I64, P, P, I64, P, P, I64, P,
                                              ctypes.c_float, P, P, P, U64, I32, P]
    lib.mla_tree_verify_run_steps.restype = I32
    lib.mla_tree_verify_strerror.argtypes = [I32]
    lib.mla_tree_verify_strerror.restype = ctypes.c_char_p
    lib.mla_tree_verify_clear_device_error.argtypes = [P, P]
    lib.mla_tree_verify_clear_device_error.restype = I32
    lib.mla_tree_verify_read_device_error.argtypes = [P, ctypes.POINTER(ctypes.c_uint32), P]
    lib.mla_tree_verify_read_device_error.restype = I32
    lib.mla_tree_verify_run_static.argtypes = [ctypes.POINTER(MtvPlan), P, P, I64, P, I64, P, P, I64, P, P,
                                               I64, P, ctypes.c_float, P, P, P]
    lib.mla_tree_verify_run_static.restype = I32
    lib.mla_tree_verify_read_static_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint32), P]
    lib.mla_tree_verify_read_static_device_error.restype = I32
    lib.mla_tree_mask_build.argtypes = [P, P, P, I32, I32, I32, P, U64, P, P, P]
    lib.mla_tree_mask_build.restype = I32
    lib.mla_tree_accept.argtypes = [P, P, P, P, P, P, I32, I32, P, P, P, P, P, P]
    lib.mla_tree_accept.restype = I32
    lib.mla_kv_defrag.argtypes = [P, P, I64, P, P, I32, I64, P, P, P, P]
    lib.mla_kv_defrag.restype = I32
    lib.mla_tree_group_prefix.argtypes = [P, I32, I64, P, P, P, P, P, P, P, P, P, P]
    lib.mla_tree_group_prefix.restype = I32
    if path == library_path():
        _lib = lib
    return lib


def strerror(code: int) -> str:
    return load().mla_tree_verify_strerror(int(code)).decode()


def plan(device: int, bs: int, max_q_per_req: int, total_q_max: int, max_prefix: int,
         mask_layout: int = MASK_FULL_ROW, flags: int = 0, nsplit: int = 0,
         num_heads: int = 64, d_latent: int = 512, d_rope: int = 64) -> MtvPlan:
    p = MtvPlan()
    ws = ctypes.c_uint64(0)
    rc = load().mla_tree_verify_plan(int(device), int(bs), int(max_q_per_req), int(total_q_max),
                                      int(max_prefix), int(num_heads), int(d_latent), int(d_rope),
                                      int(mask_layout), int(flags), int(nsplit), ctypes.byref(p),
                                      ctypes.byref(ws))
    if rc != MTV_OK:
        raise MtvError(rc, "mla_tree_verify_plan")
    return p


def choose_nsplit(num_sms: int, prefix_lens, tree_sizes, flags: int = 0) -> int:
    """Split count for a batch with these request lengths (host lists or
    arrays), to pass as ``nsplit`` to ``plan``."""
    import numpy as np
    pl = np.ascontiguousarray(np.asarray(list(prefix_lens), dtype=np.int64))
    ts = np.ascontiguousarray(np.asarray(list(tree_sizes), dtype=np.int32))
    if pl.shape != ts.shape:
        raise ValueError("prefix_lens and tree_sizes differ in length")
    out = ctypes.c_int(0)
    rc = load().mla_tree_verify_choose_nsplit(int(num_sms), int(pl.size), pl.ctypes.data if pl.size else None,
                                              ts.ctypes.data if ts.size else None, int(flags), ctypes.byref(out))
    if rc != MTV_OK:
        raise MtvError(rc, "mla_tree_verify_choose_nsplit")
    return int(out.value)


def _ptr(t, dtype, name, empty=None):
    """Device address of a tensor.  An empty tensor maps to ``empty`` (a valid
    device address that is never dereferenced because its size is zero)."""
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        return int(t)  # raw device address
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr() if t.numel() else empty


def _stream_handle(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _numel(t, given):
    """Element count of a buffer argument: ``given`` if set, else the tensor's
    numel (0 for None).  A raw address needs an explicit count."""
    if given is not None:
        return int(given)
    if t is None:
        return 0
    if isinstance(t, torch.Tensor):
        return t.numel()
    raise ValueError("a raw device address needs an explicit length")


def run(p: MtvPlan, q, kv_pool, kv_indices, kv_indptr, out_cache_loc, qo_indptr, custom_mask,
        mask_indptr, scale: float, out, lse, workspace, stream=None, check: bool = True,
        kv_indices_len=None, out_cache_loc_len=None, custom_mask_len=None, steps=None) -> int:
    """Enqueues one verify-attention pass (or, with ``steps``, only the given
    launches of it); returns the ABI code (raises if check).  Buffer lengths
    default to the tensors' element counts."""
    num_slots = kv_pool.shape[0] if isinstance(kv_pool, torch.Tensor) else 0
    ws_bytes = workspace.numel() * workspace.element_size() if isinstance(workspace, torch.Tensor) else 0
    wsp = _ptr(workspace, torch.uint8, "workspace")
    args = (ctypes.byref(p), _ptr(q, torch.bfloat16, "q", wsp), _ptr(kv_pool, torch.bfloat16, "kv_pool", wsp),
            int(num_slots), _ptr(kv_indices, torch.int64, "kv_indices", wsp), _numel(kv_indices, kv_indices_len),
            _ptr(kv_indptr, torch.int32, "kv_indptr"), _ptr(out_cache_loc, torch.int64, "out_cache_loc", wsp),
            _numel(out_cache_loc, out_cache_loc_len), _ptr(qo_indptr, torch.int64, "qo_indptr"),
            _ptr(custom_mask, torch.uint8, "custom_mask", wsp), _numel(custom_mask, custom_mask_len),
            _ptr(mask_indptr, torch.int64, "mask_indptr"), float(scale),
            _ptr(out, torch.bfloat16, "out", wsp), _ptr(lse, torch.float32, "lse", wsp),
            wsp, int(ws_bytes))
    if steps is None:
        rc = load().mla_tree_verify_run(*args, _stream_handle(stream))
        what = "mla_tree_verify_run"
    else:
        rc = load().mla_tree_verify_run_steps(*args, int(steps), _stream_handle(stream))
        what = "mla_tree_verify_run_steps"
    if check and rc != MTV_OK:
        raise MtvError(rc, what)
    return rc


def run_static(p: MtvPlan, q, kv_pool, kv_indices, kv_indptr, out_cache_loc, qo_indptr, custom_mask,
               mask_indptr, scale: float, out, lse, stream=None, check: bool = True,
               kv_indices_len=None, out_cache_loc_len=None, custom_mask_len=None) -> int:
    """The allocation-free entry point: like ``run`` without a workspace (the
    library's fixed device scratch is used; see the header for its limits)."""
    num_slots = kv_pool.shape[0] if isinstance(kv_pool, torch.Tensor) else 0
    anyp = _ptr(out, torch.bfloat16, "out")
    rc = load().mla_tree_verify_run_static(
        ctypes.byref(p), _ptr(q, torch.bfloat16, "q", anyp), _ptr(kv_pool, torch.bfloat16, "kv_pool", anyp),
        int(num_slots), _ptr(kv_indices, torch.int64, "kv_indices", anyp), _numel(kv_indices, kv_indices_len),
        _ptr(kv_indptr, torch.int32, "kv_indptr"), _ptr(out_cache_loc, torch.int64, "out_cache_loc", anyp),
        _numel(out_cache_loc, out_cache_loc_len), _ptr(qo_indptr, torch.int64, "qo_indptr"),
        _ptr(custom_mask, torch.uint8, "custom_mask", anyp), _numel(custom_mask, custom_mask_len),
        _ptr(mask_indptr, torch.int64, "mask_indptr"), float(scale), anyp,
        _ptr(lse, torch.float32, "lse"), _stream_handle(stream))
    if check and rc != MTV_OK:
        raise MtvError(rc, "mla_tree_verify_run_static")
    return rc


def read_static_device_error(stream=None) -> int:
    """Error word of the fixed scratch of ``run_static`` on the current device (syncs)."""
    v = ctypes.c_uint32(0)
    rc = load().mla_tree_verify_read_static_device_error(ctypes.byref(v), _stream_handle(stream))
    if rc != MTV_OK:
        raise MtvError(rc, "mla_tree_verify_read_static_device_error")
    return int(v.value)


def clear_device_error(workspace, stream=None):
    rc = load().mla_tree_verify_clear_device_error(_ptr(workspace, torch.uint8, "workspace"),
                                                   _stream_handle(stream))
    if rc != MTV_OK:
        raise MtvError(rc, "mla_tree_verify_clear_device_error")


def read_device_error(workspace, stream=None) -> int:
    v = ctypes.c_uint32(0)
    rc = load().mla_tree_verify_read_device_error(_ptr(workspace, torch.uint8, "workspace"),
                                                  ctypes.byref(v), _stream_handle(stream))
    if rc != MTV_OK:
        raise MtvError(rc, "mla_tree_verify_read_device_error")
    return int(v.value)


def tree_mask_build(parents, qo_indptr, kv_indptr, bs: int, max_q_per_req: int, mask_layout: int,
                    custom_mask, mask_indptr, err=None, stream=None, check: bool = True) -> int:
    """Enqueues the custom_mask + mask_indptr build from int32 parent arrays."""
    cap = custom_mask.numel() if isinstance(custom_mask, torch.Tensor) else 0
    ip = _ptr(mask_indptr, torch.int64, "mask_indptr")
    rc = load().mla_tree_mask_build(
        _ptr(parents, torch.int32, "parents", ip), _ptr(qo_indptr, torch.int64, "qo_indptr"),
        _ptr(kv_indptr, torch.int32, "kv_indptr") if kv_indptr is not None else None, int(bs),
        int(max_q_per_req), int(mask_layout), _ptr(custom_mask, torch.uint8, "custom_mask", ip), int(cap), ip,
        _ptr(err, torch.int32, "err") if err is not None else None, _stream_handle(stream))
    if check and rc != MTV_OK:
        raise MtvError(rc, "mla_tree_mask_build")
    return rc


def tree_accept(parents, draft_tokens, target_tokens, target_root_tokens, out_cache_loc, qo_indptr, bs: int,
                max_q_per_req: int, accept_len, accept_nodes, accept_slots, bonus_tokens, err=None, stream=None,
                check: bool = True) -> int:
    """Enqueues the greedy acceptance walk of every request's verified tree."""
    any_p = _ptr(accept_len, torch.int32, "accept_len")
    rc = load().mla_tree_accept(
        _ptr(parents, torch.int32, "parents", any_p), _ptr(draft_tokens, torch.int32, "draft_tokens", any_p),
        _ptr(target_tokens, torch.int32, "target_tokens", any_p),
        _ptr(target_root_tokens, torch.int32, "target_root_tokens"),
        _ptr(out_cache_loc, torch.int64, "out_cache_loc", any_p), _ptr(qo_indptr, torch.int64, "qo_indptr"),
        int(bs), int(max_q_per_req), any_p, _ptr(accept_nodes, torch.int32, "accept_nodes", any_p),
        _ptr(accept_slots, torch.int64, "accept_slots", any_p), _ptr(bonus_tokens, torch.int32, "bonus_tokens"),
        _ptr(err, torch.int32, "err") if err is not None else None, _stream_handle(stream))
    if check and rc != MTV_OK:
        raise MtvError(rc, "mla_tree_accept")
    return rc


def kv_defrag(kv_src, kv_dst, kv_indices, kv_indptr, bs: int, max_prefix: int, dst_base, kv_indices_out,
              err=None, stream=None, check: bool = True) -> int:
    """Enqueues the copy of each request's prefix rows into one contiguous run
    of slots starting at dst_base[r], and the rewrite of their indices."""
    num_slots = kv_src.shape[0] if isinstance(kv_src, torch.Tensor) else 0
    rc = load().mla_kv_defrag(
        _ptr(kv_src, torch.bfloat16, "kv_src"), _ptr(kv_dst, torch.bfloat16, "kv_dst"), int(num_slots),
        _ptr(kv_indices, torch.int64, "kv_indices"), _ptr(kv_indptr, torch.int32, "kv_indptr"), int(bs),
        int(max_prefix), _ptr(dst_base, torch.int64, "dst_base"), _ptr(kv_indices_out, torch.int64, "kv_indices_out"),
        _ptr(err, torch.int32, "err") if err is not None else None, _stream_handle(stream))
    if check and rc != MTV_OK:
        raise MtvError(rc, "mla_kv_defrag")
    return rc


def tree_group_prefix(group_indptr, num_groups: int, max_group_prefix: int, kv_indices, kv_indptr, qo_indptr,
                      parents, kv_indptr_out, kv_indices_out, qo_indptr_out, parents_out, err=None, stream=None,
                      check: bool = True) -> int:
    """Enqueues the merge of runs of requests sharing a prefix (see the header)."""
    rc = load().mla_tree_group_prefix(
        _ptr(group_indptr, torch.int32, "group_indptr"), int(num_groups), int(max_group_prefix),
        _ptr(kv_indices, torch.int64, "kv_indices"), _ptr(kv_indptr, torch.int32, "kv_indptr"),
        _ptr(qo_indptr, torch.int64, "qo_indptr"), _ptr(parents, torch.int32, "parents"),
        _ptr(kv_indptr_out, torch.int32, "kv_indptr_out"), _ptr(kv_indices_out, torch.int64, "kv_indices_out"),
        _ptr(qo_indptr_out, torch.int64, "qo_indptr_out"), _ptr(parents_out, torch.int32, "parents_out"),
        _ptr(err, torch.int32, "err") if err is not None else None, _stream_handle(stream))
    if check and rc != MTV_OK:
        raise MtvError(rc, "mla_tree_group_prefix")
    return rc


class MlaTreeVerify:
    """Owns a plan and a torch-allocated workspace for fixed upper bounds.

    ``__call__`` takes device tensors (the SGLang-style buffers) and writes
    ``out``/``lse``; it never synchronises, so it can be captured in a graph."""

    def __init__(self, bs, max_q_per_req, total_q_max, max_prefix, device=0,
                 mask_layout=MASK_FULL_ROW, flags=0, nsplit=0, lengths=None):
        """``lengths``: optional (prefix_lens, tree_sizes) of the batch the
        plan is for; with ``nsplit == 0`` the split count then comes from
        ``choose_nsplit`` instead of the upper bounds alone."""
        if nsplit == 0 and lengths is not None:
            sms = torch.cuda.get_device_properties(device).multi_processor_count
            nsplit = choose_nsplit(sms, lengths[0], lengths[1], flags)
        self.plan = plan(device, bs, max_q_per_req, total_q_max, max_prefix, mask_layout, flags, nsplit)
        self.device = torch.device("cuda", device)
        self.workspace = torch.empty(max(int(self.plan.ws_bytes), 256), dtype=torch.uint8, device=self.device)
        clear_device_error(self.workspace)

    def __call__(self, q, kv_pool, kv_indices, kv_indptr, out_cache_loc, qo_indptr, custom_mask,
                 mask_indptr, scale, out=None, lse=None, stream=None, **lengths):
        """``lengths``: optional kv_indices_len / out_cache_loc_len /
        custom_mask_len (default: the tensors' element counts)."""
        T = self.plan.total_q_max
        if out is None:
            out = torch.empty((T, 64, 512), dtype=torch.bfloat16, device=self.device)
        if lse is None:
            lse = torch.empty((T, 64), dtype=torch.float32, device=self.device)
        run(self.plan, q, kv_pool, kv_indices, kv_indptr, out_cache_loc, qo_indptr, custom_mask,
            mask_indptr, scale, out, lse, self.workspace, stream, **lengths)
        return out, lse

    def device_error(self, stream=None) -> int:
        return read_device_error(self.workspace, stream)
