"""fp64 CPU oracle for fork decode attention (test infrastructure only).

Only ``tests/``, the smoke check and the benchmark's CPU-baseline leg import this package.
The definition it computes is stated in ``fork_attn_oracle.c``.

Parity pins (what checks the oracle against something other than itself) live in
``tests/test_oracle_pins.py``.  No absolute attention value is printed on the source pages, so
beyond closed forms, library special cases, brute force and invariants the values are
"parity unpinned".
"""
import ctypes
import os

import numpy as np
import torch

from . import build as _build


class _Problem(ctypes.Structure):
    _fields_ = [
        ("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32), ("page_size", ctypes.c_int32),
        ("scale", ctypes.c_double),
        ("page_ids", ctypes.c_void_p), ("num_page_ids", ctypes.c_int64),
        ("segs", ctypes.c_void_p), ("num_segs", ctypes.c_int32),
        ("branch_seg_off", ctypes.c_void_p), ("branch_segs", ctypes.c_void_p),
        ("num_branches", ctypes.c_int32),
        ("branch_q_off", ctypes.c_void_p),
        ("vis_bits", ctypes.c_void_p), ("vis_word_off", ctypes.c_void_p),
        ("num_pages_pool", ctypes.c_int64),
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
    ]


_LIB = None


def _lib():
    global _LIB
    if _LIB is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        lib.oracle_fork_attn.restype = ctypes.c_int
        lib.oracle_fork_attn.argtypes = [ctypes.POINTER(_Problem), ctypes.c_void_p,
                                         ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                                         ctypes.c_int]
        lib.oracle_unique_slots.restype = ctypes.c_int
        lib.oracle_unique_slots.argtypes = [ctypes.POINTER(_Problem),
                                            ctypes.POINTER(ctypes.c_int64),
                                            ctypes.POINTER(ctypes.c_int64)]
        _LIB = lib
    return _LIB


def _bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)


def _problem(w, keep):
    def arr(x, dt):
        a = np.ascontiguousarray(x, dtype=dt)
        keep.append(a)
        return a.ctypes.data

    q, k, v = _bf16_bits(w.q), _bf16_bits(w.k_pages), _bf16_bits(w.v_pages)
    keep.extend([q, k, v])
    pr = _Problem()
    pr.num_q_heads, pr.num_kv_heads = w.num_q_heads, w.num_kv_heads
    pr.head_dim, pr.page_size = w.head_dim, w.page_size
    pr.scale = float(getattr(w, "scale_override", None) or w.scale)
    pr.page_ids = arr(w.page_ids, np.int32)
    pr.num_page_ids = len(w.page_ids)
    pr.segs = arr(w.segs, np.int32)
    pr.num_segs = len(w.segs)
    pr.branch_seg_off = arr(w.branch_seg_off, np.int32)
    pr.branch_segs = arr(w.branch_segs, np.int32)
    pr.num_branches = w.num_branches
    pr.branch_q_off = arr(w.branch_q_off, np.int32)
    if w.vis_bits is not None:
        pr.vis_bits = arr(w.vis_bits, np.uint32)
        pr.vis_word_off = arr(w.vis_word_off, np.int64)
    pr.num_pages_pool = w.num_pages_pool
    pr.q, pr.k, pr.v = q.ctypes.data, k.ctypes.data, v.ctypes.data
    return pr


def threads_default() -> int:
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()


def fork_attn(w, rows=None, threads=None):
    """fp64 (out [n, D], lse [n]) for the requested rows (query_token * Hq + head), or all."""
    keep = []
    pr = _problem(w, keep)
    if rows is None:
        n = w.total_q * w.num_q_heads
        rows_ptr = None
    else:
        r = np.ascontiguousarray(rows, dtype=np.int64)
        keep.append(r)
        n = len(r)
        rows_ptr = r.ctypes.data
    out = np.zeros((n, w.head_dim), dtype=np.float64)
    lse = np.zeros(n, dtype=np.float64)
    rc = _lib().oracle_fork_attn(ctypes.byref(pr), rows_ptr, n, out.ctypes.data,
                                 lse.ctypes.data, int(threads or threads_default()))
    if rc != 0:
        raise RuntimeError("oracle_fork_attn failed (bad arguments or out of memory)")
    return out, lse


def unique_slots(w):
    """(distinct visible physical slots, distinct pages holding one) over all branches."""
    keep = []
    import copy
    ww = copy.copy(w)
    if ww.q is None:  # structure-only workloads: no values needed for counting
        ww.q = torch.zeros((ww.total_q, ww.num_q_heads, ww.head_dim), dtype=torch.bfloat16)
        ww.k_pages = torch.zeros((1,), dtype=torch.bfloat16)
        ww.v_pages = ww.k_pages
    pr = _problem(ww, keep)
    s, p = ctypes.c_int64(), ctypes.c_int64()
    if _lib().oracle_unique_slots(ctypes.byref(pr), ctypes.byref(s), ctypes.byref(p)) != 0:
        raise RuntimeError("oracle_unique_slots failed")
    return s.value, p.value
