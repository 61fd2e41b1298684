"""fork_attn_decode_static_scratch: the decode for callers that cannot allocate device memory.

Such a caller (an engine plugin handed only its input and output tensors, or code that must
not touch the allocator while it runs) gets the plan arrays and the partial results in the
library's built-in device array instead of buffers of its own.  These tests call the entry
point through the C ABI and compare it with fork_attn_decode on the same inputs, on two calls
in a row (the array keeps the previous call's contents), and check that a plan too large for
the array is refused before anything runs.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import shared_prefix_paged_attn_b300 as fa
from shared_prefix_paged_attn_b300 import _lib
from shared_prefix_paged_attn_b300 import workloads as W

pytestmark = pytest.mark.gpu

MAX_ABS, REL_L2, LSE_ABS = 1e-2, 5e-3, 1e-3


def _close(a_out, a_lse, b_out, b_lse):
    a_out, b_out = a_out.float().cpu().numpy(), b_out.float().cpu().numpy()
    a_lse, b_lse = a_lse.cpu().numpy(), b_lse.cpu().numpy()
    assert np.array_equal(np.isneginf(a_lse), np.isneginf(b_lse))
    fin = ~np.isneginf(b_lse)
    assert np.abs(a_out - b_out).max() <= MAX_ABS
    assert np.linalg.norm(a_out - b_out) <= REL_L2 * max(np.linalg.norm(b_out), 1e-30)
    assert np.abs(a_lse[fin] - b_lse[fin]).max(initial=0.0) <= LSE_ABS


def _static_call(q, k, v, plan, out, lse):
    rc = _lib.load().fork_attn_decode_static_scratch(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), plan.handle, out.data_ptr(), lse.data_ptr(),
        torch.cuda.current_stream().cuda_stream)
    assert rc == 0, fa.fork_attn_strerror(rc)


@pytest.mark.parametrize("case", ["flat_fork_drops", "kv_dag_small", "random_multi_token"])
def test_static_scratch_matches_the_allocating_decode_twice(case):
    if case == "flat_fork_drops":
        w = W.make(2, device="cuda")
    elif case == "kv_dag_small":
        w = W.make(3, small=True, device="cuda")
    else:
        w = W.random_dag(77, num_q_heads=16, num_kv_heads=4, n_segs=6, n_branches=6,
                         max_seg_len=400, pool_pages=60, max_nq=8, device="cuda")
    q, k, v = w.q.cuda(), w.k_pages.cuda(), w.v_pages.cuda()
    ref = fa.ForkAttention(w, out_dtype=fa.FA_F32)
    ref_out, ref_lse = ref(q, k, v)
    torch.cuda.synchronize()
    plan = fa.plan_for(w, out_dtype=fa.FA_F32)
    pb, sb = plan.sizes()
    assert pb + sb <= _lib.FA_STATIC_SCRATCH_BYTES
    for _ in range(2):
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        _static_call(q, k, v, plan, out, lse)
        torch.cuda.synchronize()
        _close(out, lse, ref_out, ref_lse)


def test_static_scratch_after_another_plan():
    # a different plan ran in between: the array's old contents must not leak into the result
    a = W.make(1, device="cuda")
    b = W.make(2, small=True, device="cuda")
    pa = fa.plan_for(a, out_dtype=fa.FA_F32)
    pb = fa.plan_for(b, out_dtype=fa.FA_F32)
    outs = []
    for w, p in ((a, pa), (b, pb), (a, pa)):
        out = torch.empty((w.total_q, w.num_q_heads, 128), dtype=torch.float32, device="cuda")
        lse = torch.empty((w.total_q, w.num_q_heads), dtype=torch.float32, device="cuda")
        _static_call(w.q.cuda(), w.k_pages.cuda(), w.v_pages.cuda(), p, out, lse)
        torch.cuda.synchronize()
        outs.append((out.clone(), lse.clone()))
    ref = fa.ForkAttention(a, out_dtype=fa.FA_F32)
    r_out, r_lse = ref(a.q.cuda(), a.k_pages.cuda(), a.v_pages.cuda())
    torch.cuda.synchronize()
    _close(*outs[0], r_out, r_lse)
    _close(*outs[2], r_out, r_lse)


def test_plan_too_large_for_the_static_array_is_refused():
    w = W.make(4, values=False)  # ~70 MB of partials: more than the built-in array
    plan = fa.plan_for(w)
    pb, sb = plan.sizes()
    assert pb + sb > _lib.FA_STATIC_SCRATCH_BYTES
    fake = ctypes.c_void_p(1 << 20)
    rc = _lib.load().fork_attn_decode_static_scratch(fake, fake, fake, plan.handle, fake, fake, None)
    assert rc == -11
