"""fork_attn_decode_static_scratch: the decode for callers that cannot allocate device memory.

Such a caller (an engine plugin handed only its input and output tensors, or code that must
not touch the allocator while it runs) gets the plan arrays and the partial results in the
library's built-in device array instead of buffers of its own.  These tests call the entry
point through the C ABI and compare it with fork_attn_decode on the same inputs, on two calls
in a row (the array keeps the previous call's contents): the same plan runs the same kernels
on the same data, so every output bit must agree.  One case is also checked against the fp64
oracle, and fork_attn_check must read a clear error word after each call.  A plan too large
for the array is refused before anything runs.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import shared_prefix_paged_attn_b300 as fa
from shared_prefix_paged_attn_b300 import _lib
from shared_prefix_paged_attn_b300 import workloads as W

pytestmark = pytest.mark.gpu

MAX_ABS, REL_L2, LSE_ABS = 1e-2, 5e-3, 1e-3


def _static_call(q, k, v, plan, out, lse):
    rc = _lib.load().fork_attn_decode_static_scratch(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), plan.handle, out.data_ptr(), lse.data_ptr(),
        torch.cuda.current_stream().cuda_stream)
    assert rc == 0, fa.fork_attn_strerror(rc)


def _bitwise(a_out, a_lse, b_out, b_lse):
    assert torch.equal(a_out, b_out) and torch.equal(a_lse, b_lse)


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
    ref_out, ref_lse = (x.clone() for x in ref(q, k, v))
    torch.cuda.synchronize()
    assert fa.fork_attn_check(ref.plan) == 0
    plan = fa.plan_for(w, out_dtype=fa.FA_F32)
    pb, sb = plan.sizes()
    assert pb + sb <= _lib.FA_STATIC_SCRATCH_BYTES
    for _ in range(2):
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        _static_call(q, k, v, plan, out, lse)
        assert fa.fork_attn_check(plan) == 0  # the word the static call wrote is clear
        _bitwise(out, lse, ref_out, ref_lse)


def test_static_scratch_against_the_oracle():
    w = W.make(5, small=True)
    q, k, v = w.q.cuda(), w.k_pages.cuda(), w.v_pages.cuda()
    plan = fa.plan_for(w, out_dtype=fa.FA_F32)
    out = torch.empty((w.total_q, w.num_q_heads, 128), dtype=torch.float32, device="cuda")
    lse = torch.empty((w.total_q, w.num_q_heads), dtype=torch.float32, device="cuda")
    _static_call(q, k, v, plan, out, lse)
    assert fa.fork_attn_check(plan) == 0
    got = out.cpu().numpy().reshape(-1, 128)
    got_lse = lse.cpu().numpy().reshape(-1)
    ref_out, ref_lse = oracle.fork_attn(w)
    assert np.array_equal(np.isneginf(got_lse), np.isneginf(ref_lse))
    fin = ~np.isneginf(ref_lse)
    assert np.abs(got[fin] - ref_out[fin]).max() <= MAX_ABS
    assert np.linalg.norm(got[fin] - ref_out[fin]) <= REL_L2 * np.linalg.norm(ref_out[fin])
    assert np.abs(got_lse[fin] - ref_lse[fin]).max() <= LSE_ABS


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
        assert fa.fork_attn_check(p) == 0
        outs.append((out.clone(), lse.clone()))
    ref = fa.ForkAttention(a, out_dtype=fa.FA_F32)
    r_out, r_lse = ref(a.q.cuda(), a.k_pages.cuda(), a.v_pages.cuda())
    torch.cuda.synchronize()
    _bitwise(*outs[0], r_out, r_lse)
    _bitwise(*outs[2], r_out, r_lse)


def test_plan_too_large_for_the_static_array_is_refused():
    w = W.make(4, values=False)  # ~70 MB of partials: more than the built-in array
    plan = fa.plan_for(w)
    pb, sb = plan.sizes()
    assert pb + sb > _lib.FA_STATIC_SCRATCH_BYTES
    fake = ctypes.c_void_p(1 << 20)
    rc = _lib.load().fork_attn_decode_static_scratch(fake, fake, fake, plan.handle, fake, fake, None)
    assert rc == -11
    # nothing ran: the plan has no error word to read yet
    word = ctypes.c_int32()
    assert _lib.load().fork_attn_check(plan.handle, ctypes.byref(word), None) == -6
