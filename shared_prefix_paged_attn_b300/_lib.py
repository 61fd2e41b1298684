"""ctypes declarations of the C ABI in ``include/fork_attn.h`` (argument marshalling only)."""
import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
# FORK_ATTN_CHECKED=1 in the environment (read at the first load) selects the build with
# device bounds checks on every index taken from a plan buffer
LIB_PATH = os.path.join(HERE, "libforkattn_checked.so" if os.environ.get("FORK_ATTN_CHECKED") == "1"
                        else "libforkattn.so")

c_int32, c_int64, c_float, c_void_p = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p

FA_OK = 0
FA_STATIC_SCRATCH_BYTES = 32 << 20
FA_BF16, FA_F32 = 0, 1


class FaDims(ctypes.Structure):
    _fields_ = [("num_q_heads", c_int32), ("num_kv_heads", c_int32), ("head_dim", c_int32),
                ("page_size", c_int32), ("scale", c_float), ("out_dtype", c_int32)]


class FaSegment(ctypes.Structure):
    _fields_ = [("page_off", c_int32), ("tok_begin", c_int32), ("len", c_int32)]


class FaDesc(ctypes.Structure):
    _fields_ = [("page_ids", c_void_p), ("num_page_ids", c_int64),
                ("segs", c_void_p), ("num_segs", c_int32),
                ("branch_seg_off", c_void_p), ("branch_segs", c_void_p),
                ("num_branches", c_int32),
                ("branch_q_off", c_void_p),
                ("vis_bits", c_void_p), ("vis_word_off", c_void_p),
                ("num_vis_words", c_int64), ("num_pages_pool", c_int64)]


class FaPlanOpts(ctypes.Structure):
    _fields_ = [("chunk_pages", c_int32), ("num_sms", c_int32), ("tensor_min_rows", c_int32),
                ("tensor_ctas", c_int32), ("tensor_chunk_pages", c_int32),
                ("representatives", c_int32), ("reserved", c_int32 * 2)]


class FaPlanStats(ctypes.Structure):
    _fields_ = [("unique_visible_slots", c_int64), ("touched_pages", c_int64),
                ("listed_visible_slots", c_int64), ("num_chunks", c_int64),
                ("num_items_rows", c_int64), ("num_items_tensor", c_int64),
                ("kv_bytes_rows", c_int64), ("kv_bytes_tensor", c_int64),
                ("partial_rows", c_int64), ("merge_rows", c_int64), ("total_q", c_int64),
                ("unique_slots_rows", c_int64), ("unique_slots_tensor", c_int64),
                ("flops_rows", c_int64), ("flops_tensor", c_int64),
                ("num_items_row8", c_int64), ("unique_slots_row8", c_int64),
                ("unique_slots_row32", c_int64), ("tensor_ctas", c_int64),
                ("items_skipped", c_int64)]


class FaCompactDims(ctypes.Structure):
    _fields_ = [("num_kv_heads", c_int32), ("head_dim", c_int32), ("page_size", c_int32),
                ("reposition", c_int32), ("rope_base", ctypes.c_double),
                ("share_prefix", c_int32), ("reserved", c_int32)]


# name -> (restype, argtypes); every symbol declared in include/fork_attn.h
SIGNATURES = {
    "fork_attn_plan_create": (c_int32, [ctypes.POINTER(FaDims), ctypes.POINTER(FaDesc),
                                        ctypes.POINTER(FaPlanOpts), ctypes.POINTER(c_void_p)]),
    "fork_attn_plan_sizes": (c_int32, [c_void_p, ctypes.POINTER(ctypes.c_size_t),
                                       ctypes.POINTER(ctypes.c_size_t)]),
    "fork_attn_plan_stats": (c_int32, [c_void_p, ctypes.POINTER(FaPlanStats)]),
    "fork_attn_plan_upload": (c_int32, [c_void_p, c_void_p, ctypes.c_size_t, c_void_p,
                                        ctypes.c_size_t, c_void_p]),
    "fork_attn_decode": (c_int32, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                   c_void_p]),
    "fork_attn_decode_timed": (c_int32, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                         c_void_p, c_void_p, ctypes.POINTER(c_void_p), c_int32]),
    "fork_attn_check": (c_int32, [c_void_p, ctypes.POINTER(c_int32), c_void_p]),
    "fork_attn_decode_static_scratch": (c_int32, [c_void_p, c_void_p, c_void_p, c_void_p,
                                                  c_void_p, c_void_p, c_void_p]),
    "fork_attn_plan_destroy": (c_int32, [c_void_p]),
    "fork_attn_compact_create": (c_int32, [ctypes.POINTER(FaCompactDims), ctypes.POINTER(FaDesc),
                                           c_void_p, c_int32, c_void_p, ctypes.c_int64,
                                           ctypes.POINTER(c_void_p)]),
    "fork_attn_compact_sizes": (c_int32, [c_void_p, c_void_p, ctypes.POINTER(ctypes.c_size_t)]),
    "fork_attn_compact_shared": (c_int32, [c_void_p, ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int64)]),
    "fork_attn_merge_parts": (c_int32, [c_void_p, c_void_p, c_int32, ctypes.c_int64, c_void_p, c_int32, c_void_p,
                                         c_void_p]),
    "fork_attn_score_lse": (c_int32, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]),
    "fork_attn_score": (c_int32, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]),
    "fork_attn_topk": (c_int32, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]),
    "fork_attn_score_sizes": (c_int32, [c_void_p, ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int64)]),
    "fork_attn_compact_upload": (c_int32, [c_void_p, c_void_p, ctypes.c_size_t, c_void_p]),
    "fork_attn_compact_run": (c_int32, [c_void_p, c_void_p, c_void_p, c_void_p]),
    "fork_attn_compact_destroy": (c_int32, [c_void_p]),
    "fork_attn_strerror": (ctypes.c_char_p, [c_int32]),
}

_LIB = None


def load():
    """Loads the in-tree library.  There is no fallback: a missing build is an error."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                f"{LIB_PATH} is missing: build it with `python -m shared_prefix_paged_attn_b300.build`"
                " (nvcc, sm_103a); this package has no CPU or PyTorch fallback")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = lib
    return _LIB
