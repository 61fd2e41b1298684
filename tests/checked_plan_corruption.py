"""Run in a child process with FORK_ATTN_CHECKED=1 (the library built with device bounds
checks): corrupts one page id in an uploaded plan buffer and checks that the decode reports
it through the error word, writes nowhere outside its buffers, and decodes correctly again
once the page id is restored.  Prints one line: "ok <error word>" per case."""
import ctypes
import os
import sys

import torch

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import shared_prefix_paged_attn_b300 as fa  # noqa: E402
from shared_prefix_paged_attn_b300 import _lib  # noqa: E402
from shared_prefix_paged_attn_b300 import workloads as W  # noqa: E402

assert _lib.LIB_PATH.endswith("libforkattn_checked.so"), _lib.LIB_PATH
KERR_BOUNDS = 2


def case(cfg, small, kernel_bits, **opts):
    w = W.make(cfg, small=small, device="cuda")
    run = fa.ForkAttention(w, out_dtype=fa.FA_F32, **opts)
    out0, lse0 = (x.clone() for x in run(w.q, w.k_pages, w.v_pages))
    torch.cuda.synchronize()
    assert fa.fork_attn_check(run.plan) == 0
    # the plan buffer: a 256-byte header, then the chunks' page ids (chunk 0 first)
    words = run.plan_buf.view(torch.int32)
    orig = int(words[64].item())
    words[64] = w.num_pages_pool + 7  # one past the pool and more: caught by the check
    run(w.q, w.k_pages, w.v_pages)
    torch.cuda.synchronize()
    word = ctypes.c_int32()
    rc = _lib.load().fork_attn_check(run.plan.handle, ctypes.byref(word), None)
    assert rc == -10, rc
    assert word.value & KERR_BOUNDS and word.value & kernel_bits, word.value
    words[64] = orig
    out, lse = run(w.q, w.k_pages, w.v_pages)
    torch.cuda.synchronize()
    assert fa.fork_attn_check(run.plan) == 0
    assert torch.equal(out, out0) and torch.equal(lse, lse0)
    print("ok", word.value, flush=True)


case(1, False, 8 | 16)                    # row kernels (tiny fork: no tcgen05 items)
case(4, True, 4, tensor_min_rows=1)       # every item on the tcgen05 kernel
