"""CPU fp64 oracle for MLA tree-verify attention -- test infrastructure.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  It shares no
code with the CUDA library: the arithmetic lives in ``mla_tree_verify_oracle.c``
(plain C, fp64, pthreads), compiled here with gcc.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mla_tree_verify_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB) -> str:
    """Compile the oracle with gcc (-O2, no fast-math).  ``src``/``out`` let the
    tests compile deliberately broken copies to check that the pins catch them."""
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src):
        tmp = out + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                               "-fno-fast-math", "-o", tmp, src, "-lm"])
        os.replace(tmp, out)
    return out


def open_library(path: str):
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    I64, I32, F64 = ctypes.c_int64, ctypes.c_int, ctypes.c_double
    lib.oracle_mla_tree_verify_rows.argtypes = [
        P, P, I64, P, P, P, P, P, P, I32, I32, I32, I32, I32, F64, P, I64, P, P, I32]
    lib.oracle_mla_tree_verify_rows.restype = I32
    lib.oracle_lse_combine.argtypes = [P, P, I32, I64, I32, P, P]
    lib.oracle_lse_combine.restype = I32
    return lib


_override = threading.local()


def _load():
    global _lib
    lib = getattr(_override, "lib", None)
    if lib is not None:
        return lib
    with _lock:
        if _lib is None:
            _lib = open_library(build())
    return _lib


class use_library:
    """Context manager: route this thread's oracle calls to another compiled copy."""

    def __init__(self, path: str):
        self.lib = open_library(path)

    def __enter__(self):
        self.prev = getattr(_override, "lib", None)
        _override.lib = self.lib
        return self

    def __exit__(self, *exc):
        _override.lib = self.prev


def default_threads() -> int:
    return len(os.sched_getaffinity(0))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _np(t: torch.Tensor, dtype) -> np.ndarray:
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        t = t.view(torch.int16)
    a = t.numpy()
    return np.ascontiguousarray(a.view(dtype))


def mla_tree_verify(wl, rows=None, num_threads: int | None = None, *, q=None, kv_pool=None,
                    kv_indices=None, out_cache_loc=None, custom_mask=None, mask_indptr=None,
                    kv_indptr=None, qo_indptr=None, mask_layout=None):
    """Runs the oracle on a workload (any tensor may be overridden).

    rows: None for every (token, head) row, else an int64 array of token*H + h.
    Returns (out [nrows, 512] float64, lse [nrows] float64)."""
    lib = _load()
    qa = _np(wl.q if q is None else q, np.uint16)
    pool = _np(wl.kv_pool if kv_pool is None else kv_pool, np.uint16)
    kvi = _np(wl.kv_indices if kv_indices is None else kv_indices, np.int64)
    kvp = _np(wl.kv_indptr if kv_indptr is None else kv_indptr, np.int32)
    ocl = _np(wl.out_cache_loc if out_cache_loc is None else out_cache_loc, np.int64)
    qop = _np(wl.qo_indptr if qo_indptr is None else qo_indptr, np.int64)
    msk = _np(wl.custom_mask if custom_mask is None else custom_mask, np.uint8)
    mip = _np(wl.mask_indptr if mask_indptr is None else mask_indptr, np.int64)
    layout = wl.mask_layout if mask_layout is None else mask_layout
    H = wl.num_heads
    d_qk = pool.shape[1]
    d_lat, d_rope = 512, d_qk - 512
    if rows is None:
        nrows = int(qop[-1]) * H
        rows_a = None
    else:
        rows_a = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        nrows = rows_a.shape[0]
    out = np.zeros((nrows, d_lat), dtype=np.float64)
    lse = np.zeros((nrows,), dtype=np.float64)
    # keep empty arrays addressable
    kvi = kvi if kvi.size else np.zeros(1, np.int64)
    ocl = ocl if ocl.size else np.zeros(1, np.int64)
    msk = msk if msk.size else np.zeros(1, np.uint8)
    rc = lib.oracle_mla_tree_verify_rows(
        _ptr(qa), _ptr(pool), pool.shape[0], _ptr(kvi), _ptr(kvp), _ptr(ocl), _ptr(qop),
        _ptr(msk), _ptr(mip), int(layout), int(wl.bs), H, d_lat, d_rope, float(wl.scale),
        _ptr(rows_a) if rows_a is not None else None, nrows, _ptr(out), _ptr(lse),
        int(num_threads or default_threads()))
    if rc != 0:
        raise RuntimeError(f"oracle failed with code {rc}")
    return out, lse


def lse_combine(o: np.ndarray, lse_in: np.ndarray):
    """o: [nsplit, nrows, d], lse_in: [nsplit, nrows] -> (out [nrows, d], lse [nrows])."""
    lib = _load()
    o = np.ascontiguousarray(o, dtype=np.float64)
    lse_in = np.ascontiguousarray(lse_in, dtype=np.float64)
    ns, nr, d = o.shape
    out = np.zeros((nr, d), np.float64)
    lse = np.zeros((nr,), np.float64)
    rc = lib.oracle_lse_combine(_ptr(o), _ptr(lse_in), ns, nr, d, _ptr(out), _ptr(lse))
    if rc != 0:
        raise RuntimeError(f"oracle combine failed with code {rc}")
    return out, lse
