"""Fork decode attention over a branching, paged KV cache, for one NVIDIA B300 (sm_103a).

Thin Python binding over the C ABI of ``libforkattn.so`` (``include/fork_attn.h``): the
functions below keep the C names and only marshal arguments.  Every step of the decode runs
in the library's CUDA kernels; PyTorch supplies device memory and streams.  There is no CPU
or PyTorch fallback: if the library is missing, the calls raise.
"""
import ctypes
from typing import Optional

import numpy as np

from . import _lib
from ._lib import FA_BF16, FA_F32, FaCompactDims, FaDesc, FaDims, FaPlanOpts, FaPlanStats

__all__ = ["ForkAttnError", "Plan", "fork_attn_plan_create", "fork_attn_decode",
           "fork_attn_decode_timed", "fork_attn_decode_static_scratch", "fork_attn_merge_parts", "fork_attn_score_lse", "fork_attn_score",
           "fork_attn_topk", "fork_attn_score_sizes", "KeyScorer", "fork_attn_check",
           "fork_attn_strerror", "FA_BF16", "FA_F32", "plan_for", "ForkAttention", "CompactPlan", "fork_attn_compact_create", "fork_attn_compact_upload", "fork_attn_compact_run"]


class ForkAttnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {fork_attn_strerror(status)} (status {status})")


def fork_attn_strerror(status: int) -> str:
    return _lib.load().fork_attn_strerror(int(status)).decode()


def _check(status: int, what: str):
    if status != _lib.FA_OK:
        raise ForkAttnError(status, what)


def _stream_ptr(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)


def _ptr(t) -> Optional[int]:
    return None if t is None else int(t.data_ptr())


class Plan:
    """A host plan (opaque handle owned by the library) and the arrays it was built from."""

    def __init__(self, handle: int, keep):
        self.handle = handle
        self._keep = keep
        self._bufs = None

    def sizes(self):
        pb, sb = ctypes.c_size_t(), ctypes.c_size_t()
        _check(_lib.load().fork_attn_plan_sizes(self.handle, ctypes.byref(pb), ctypes.byref(sb)),
               "fork_attn_plan_sizes")
        return pb.value, sb.value

    def stats(self) -> dict:
        st = FaPlanStats()
        _check(_lib.load().fork_attn_plan_stats(self.handle, ctypes.byref(st)), "fork_attn_plan_stats")
        return {name: getattr(st, name) for name, _ in FaPlanStats._fields_ if name != "reserved"}

    def upload(self, plan_buf, scratch_buf=None, stream=None):
        """fork_attn_plan_upload: plan_buf / scratch_buf are device tensors (uint8) the caller keeps."""
        sb = 0 if scratch_buf is None else scratch_buf.numel() * scratch_buf.element_size()
        _check(_lib.load().fork_attn_plan_upload(
            self.handle, _ptr(plan_buf), plan_buf.numel() * plan_buf.element_size(),
            _ptr(scratch_buf), sb, _stream_ptr(stream)), "fork_attn_plan_upload")
        self._bufs = (plan_buf, scratch_buf)

    def destroy(self):
        if self.handle:
            _lib.load().fork_attn_plan_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass


def _desc(arr, page_ids, segs, branch_seg_off, branch_segs, num_pages_pool, branch_q_off,
          vis_bits, vis_word_off) -> FaDesc:
    segs = np.ascontiguousarray(segs, dtype=np.int32).reshape(-1, 3)
    desc = FaDesc()
    desc.page_ids = arr(page_ids, np.int32)
    desc.num_page_ids = len(page_ids)
    desc.segs = arr(segs, np.int32)
    desc.num_segs = len(segs)
    desc.branch_seg_off = arr(branch_seg_off, np.int32)
    desc.branch_segs = arr(branch_segs, np.int32)
    desc.num_branches = len(branch_seg_off) - 1
    desc.branch_q_off = arr(branch_q_off, np.int32)
    desc.vis_bits = arr(vis_bits, np.uint32)
    desc.vis_word_off = arr(vis_word_off, np.int64)
    desc.num_vis_words = 0 if vis_bits is None else len(vis_bits)
    desc.num_pages_pool = int(num_pages_pool)
    return desc


def fork_attn_plan_create(num_q_heads, num_kv_heads, page_ids, segs, branch_seg_off,
                          branch_segs, num_pages_pool, branch_q_off=None, vis_bits=None,
                          vis_word_off=None, scale=None, out_dtype=FA_BF16, head_dim=128,
                          page_size=16, chunk_pages=0, num_sms=0, tensor_min_rows=0,
                          tensor_ctas=0, tensor_chunk_pages=0, representatives=0) -> Plan:
    """fork_attn_plan_create over host (numpy) descriptor arrays."""
    keep = []

    def arr(x, dt):
        if x is None:
            return None
        a = np.ascontiguousarray(x, dtype=dt)
        keep.append(a)
        return a.ctypes.data

    dims = FaDims(int(num_q_heads), int(num_kv_heads), int(head_dim), int(page_size),
                  float(scale if scale is not None else 1.0 / np.sqrt(head_dim)), int(out_dtype))
    desc = _desc(arr, page_ids, segs, branch_seg_off, branch_segs, num_pages_pool, branch_q_off,
                 vis_bits, vis_word_off)
    opts = FaPlanOpts()
    opts.chunk_pages, opts.num_sms, opts.tensor_min_rows = int(chunk_pages), int(num_sms), int(tensor_min_rows)
    opts.tensor_ctas, opts.tensor_chunk_pages = int(tensor_ctas), int(tensor_chunk_pages)
    opts.representatives = int(representatives)
    handle = ctypes.c_void_p()
    _check(_lib.load().fork_attn_plan_create(ctypes.byref(dims), ctypes.byref(desc),
                                             ctypes.byref(opts), ctypes.byref(handle)),
           "fork_attn_plan_create")
    return Plan(handle.value, keep)


def fork_attn_decode(q, k_pages, v_pages, plan: Plan, out, lse, stream=None):
    _check(_lib.load().fork_attn_decode(_ptr(q), _ptr(k_pages), _ptr(v_pages), plan.handle,
                                        _ptr(out), _ptr(lse), _stream_ptr(stream)),
           "fork_attn_decode")


def fork_attn_decode_timed(q, k_pages, v_pages, plan: Plan, out, lse, events, stream=None):
    """The decode with its kernels one after another on `stream`; events: 8
    torch.cuda.Event(enable_timing=True), [start, stop] around the row kernel of <= 8 rows, the
    row kernel, the tcgen05 kernel and the merge."""
    if len(events) != 8:
        raise ValueError("fork_attn_decode_timed needs 8 events")
    for e in events:  # torch creates an event's handle on its first record
        if not e.cuda_event:
            e.record()
    handles = (ctypes.c_void_p * 8)(*[ctypes.c_void_p(e.cuda_event) for e in events])
    _check(_lib.load().fork_attn_decode_timed(_ptr(q), _ptr(k_pages), _ptr(v_pages), plan.handle,
                                              _ptr(out), _ptr(lse), _stream_ptr(stream),
                                              handles, 4), "fork_attn_decode_timed")


def fork_attn_decode_static_scratch(q, k_pages, v_pages, plan: Plan, out, lse, stream=None):
    """Decode with the library's built-in device array for plan arrays and partials (for
    callers that cannot allocate device memory); the plan needs no upload."""
    _check(_lib.load().fork_attn_decode_static_scratch(_ptr(q), _ptr(k_pages), _ptr(v_pages),
                                                       plan.handle, _ptr(out), _ptr(lse),
                                                       _stream_ptr(stream)),
           "fork_attn_decode_static_scratch")


def fork_attn_merge_parts(part_out, part_lse, out, lse, stream=None):
    """fork_attn_merge_parts: part_out [n_parts, rows, 128] fp32 and part_lse [n_parts, rows]
    (device tensors, or [n_parts, total_q, Hq, ...]) into out (bf16 or fp32) and lse."""
    import torch
    n_parts = int(part_lse.shape[0])
    rows = int(part_lse.numel() // n_parts)
    odt = FA_F32 if out.dtype == torch.float32 else FA_BF16
    _check(_lib.load().fork_attn_merge_parts(_ptr(part_out), _ptr(part_lse), n_parts, rows, _ptr(out), odt,
                                             _ptr(lse), _stream_ptr(stream)), "fork_attn_merge_parts")


def fork_attn_score_lse(q, k_pages, plan: Plan, lse, stream=None):
    """fork_attn_score_lse: the representatives' lse [device fp32, total_q x Hq]."""
    _check(_lib.load().fork_attn_score_lse(_ptr(q), _ptr(k_pages), plan.handle, _ptr(lse), _stream_ptr(stream)),
           "fork_attn_score_lse")


def fork_attn_score(q, k_pages, plan: Plan, lse, scores, stream=None):
    """fork_attn_score: scores [device fp32, total_entries] of every branch's entries."""
    _check(_lib.load().fork_attn_score(_ptr(q), _ptr(k_pages), plan.handle, _ptr(lse), _ptr(scores),
                                       _stream_ptr(stream)), "fork_attn_score")


def fork_attn_topk(plan: Plan, scores, keep_k, keep_bits, stream=None):
    """fork_attn_topk: keep_k [device int32, B]; keep_bits [device int32/uint32, total_words]."""
    _check(_lib.load().fork_attn_topk(plan.handle, _ptr(scores), _ptr(keep_k), _ptr(keep_bits),
                                      _stream_ptr(stream)), "fork_attn_topk")


def fork_attn_score_sizes(plan: Plan):
    """(total_entries, total_words) of a representatives plan."""
    e, wds = ctypes.c_int64(), ctypes.c_int64()
    _check(_lib.load().fork_attn_score_sizes(plan.handle, ctypes.byref(e), ctypes.byref(wds)),
           "fork_attn_score_sizes")
    return e.value, wds.value


class KeyScorer:
    """Representative-query scoring of a workload whose query tokens are the representatives
    (plan, buffers, and the three calls: decode for lse, score, top-k)."""

    def __init__(self, w, device="cuda", stream=None, **opts):
        import torch
        self.plan = plan_for(w, out_dtype=FA_F32, representatives=1, **opts)
        pb, sb = self.plan.sizes()
        self.plan_buf = torch.empty(pb, dtype=torch.uint8, device=device)
        self.scratch = torch.empty(max(sb, 1), dtype=torch.uint8, device=device)
        self.plan.upload(self.plan_buf, self.scratch, stream)
        E, nw = fork_attn_score_sizes(self.plan)
        self.out = torch.empty((w.total_q, w.num_q_heads, w.head_dim), dtype=torch.float32, device=device)
        self.lse = torch.empty((w.total_q, w.num_q_heads), dtype=torch.float32, device=device)
        self.scores = torch.empty(max(E, 1), dtype=torch.float32, device=device)
        self.keep_bits = torch.empty(max(nw, 1), dtype=torch.int32, device=device)

    def score(self, q, k_pages, v_pages=None, stream=None):
        fork_attn_score_lse(q, k_pages, self.plan, self.lse, stream)
        fork_attn_score(q, k_pages, self.plan, self.lse, self.scores, stream)
        return self.scores

    def topk(self, keep_k, stream=None):
        fork_attn_topk(self.plan, self.scores, keep_k, self.keep_bits, stream)
        return self.keep_bits


def fork_attn_check(plan: Plan, stream=None) -> int:
    """Returns the device error word (0 = fine) and clears it; syncs the stream."""
    word = ctypes.c_int32()
    rc = _lib.load().fork_attn_check(plan.handle, ctypes.byref(word), _stream_ptr(stream))
    if rc not in (_lib.FA_OK, -10):
        _check(rc, "fork_attn_check")
    return word.value


def plan_for(w, out_dtype=FA_BF16, **opts) -> Plan:
    """A plan for a ``workloads.Workload``."""
    return fork_attn_plan_create(w.num_q_heads, w.num_kv_heads, w.page_ids, w.segs,
                                 w.branch_seg_off, w.branch_segs, w.num_pages_pool,
                                 branch_q_off=w.branch_q_off, vis_bits=w.vis_bits,
                                 vis_word_off=w.vis_word_off, scale=w.scale,
                                 out_dtype=out_dtype, **opts)


class ForkAttention:
    """Plan + device buffers for one workload; ``__call__`` runs fork_attn_decode."""

    def __init__(self, w, out_dtype=FA_BF16, device="cuda", stream=None, **opts):
        import torch
        self.plan = plan_for(w, out_dtype=out_dtype, **opts)
        pb, sb = self.plan.sizes()
        self.plan_buf = torch.empty(pb, dtype=torch.uint8, device=device)
        self.scratch = torch.empty(max(sb, 1), dtype=torch.uint8, device=device) if sb else None
        self.plan.upload(self.plan_buf, self.scratch, stream)
        odt = torch.float32 if out_dtype == FA_F32 else torch.bfloat16
        self.out = torch.empty((w.total_q, w.num_q_heads, w.head_dim), dtype=odt, device=device)
        self.lse = torch.empty((w.total_q, w.num_q_heads), dtype=torch.float32, device=device)

    def __call__(self, q, k_pages, v_pages, stream=None):
        fork_attn_decode(q, k_pages, v_pages, self.plan, self.out, self.lse, stream)
        return self.out, self.lse


class CompactPlan:
    """Host handle of a compaction plan (fork_attn_compact_*); freed on destroy() or GC."""

    def __init__(self, handle: int, keep, n_branches: int):
        self.handle = handle
        self._keep = keep
        self.n_branches = n_branches

    def sizes(self):
        kept = np.zeros(self.n_branches, dtype=np.int64)
        wb = ctypes.c_size_t()
        _check(_lib.load().fork_attn_compact_sizes(self.handle, kept.ctypes.data, ctypes.byref(wb)),
               "fork_attn_compact_sizes")
        return kept, wb.value

    def shared(self):
        """(r_s, P): kept entries of the shared run and the common prefix's length (0, 0
        without share_prefix)."""
        rs, pl = ctypes.c_int64(), ctypes.c_int64()
        _check(_lib.load().fork_attn_compact_shared(self.handle, ctypes.byref(rs), ctypes.byref(pl)),
               "fork_attn_compact_shared")
        return rs.value, pl.value

    def destroy(self):
        if self.handle:
            _lib.load().fork_attn_compact_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass


def fork_attn_compact_create(w, branches, dst_page_ids, reposition=False, rope_base=10000.0,
                             head_dim=128, page_size=16, share_prefix=False) -> CompactPlan:
    """fork_attn_compact_create for a ``workloads.Workload``-like descriptor (host arrays)."""
    keep = []

    def arr(x, dt):
        if x is None:
            return None
        a = np.ascontiguousarray(x, dtype=dt)
        keep.append(a)
        return a.ctypes.data

    desc = _desc(arr, w.page_ids, w.segs, w.branch_seg_off, w.branch_segs, w.num_pages_pool,
                 w.branch_q_off, w.vis_bits, w.vis_word_off)
    dims = FaCompactDims(int(w.num_kv_heads), int(head_dim), int(page_size), int(bool(reposition)),
                         float(rope_base), int(bool(share_prefix)), 0)
    br = np.ascontiguousarray(branches, dtype=np.int32)
    dst = np.ascontiguousarray(dst_page_ids, dtype=np.int32)
    keep += [br, dst, desc, dims]
    handle = ctypes.c_void_p()
    _check(_lib.load().fork_attn_compact_create(ctypes.byref(dims), ctypes.byref(desc), br.ctypes.data,
                                                len(br), dst.ctypes.data, len(dst), ctypes.byref(handle)),
           "fork_attn_compact_create")
    return CompactPlan(handle.value, keep, len(br))


def fork_attn_compact_upload(plan: CompactPlan, work, stream=None):
    _check(_lib.load().fork_attn_compact_upload(plan.handle, _ptr(work), work.numel() * work.element_size(),
                                                _stream_ptr(stream)), "fork_attn_compact_upload")
    plan._work = work  # the device buffer must outlive the plan's runs


def fork_attn_compact_run(plan: CompactPlan, k_pages, v_pages, stream=None):
    _check(_lib.load().fork_attn_compact_run(plan.handle, _ptr(k_pages), _ptr(v_pages), _stream_ptr(stream)),
           "fork_attn_compact_run")
