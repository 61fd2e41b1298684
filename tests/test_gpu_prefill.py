"""GPU parity of prefill-shaped plans: every token of a branch is a query.

Octopus (zicq.com), "Packed DAG-GRPO": the branches of an episode are packed into one
block-sparse attention (causal inside a thread, plus the allowed cross-thread reads).  The
same fork_attn_decode call computes it from a descriptor whose branches list the segments
each thread may read and whose queries are the thread's own tokens.  The planner leaves out
(row group, chunk) pairs that no row of the group can see and stops every item at the last
page one of its rows can see; the merge gives zero weight to the partials of chunks that
start after a token.  Checked against the fp64 oracle with the decode tolerances.
"""
import numpy as np
import pytest
import torch

import oracle
import shared_prefix_paged_attn_b300 as fa
from shared_prefix_paged_attn_b300 import workloads as W

from test_gpu_parity import assert_parity

pytestmark = pytest.mark.gpu


def run_prefill(w, out_dtype=fa.FA_BF16, poison=True, **opts):
    dev = torch.device("cuda")
    run = fa.ForkAttention(w, out_dtype=out_dtype, **opts)
    if poison and run.scratch is not None:
        # NaN in every partial: a partial the merge reads without an item having written it
        # shows up in the output
        run.scratch.fill_(255)
    out, lse = run(w.q.to(dev), w.k_pages.to(dev), w.v_pages.to(dev))
    torch.cuda.synchronize()
    assert fa.fork_attn_check(run.plan) == 0
    return (out.float().cpu().numpy().reshape(-1, w.head_dim), lse.cpu().numpy().reshape(-1),
            run.plan.stats())


def as_prefill(w):
    """The same cache with every token of every branch a query (values redrawn)."""
    lens = [w.branch_len(b) for b in range(w.num_branches)]
    w.branch_q_off = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    W.fill_values(w)
    return w


@pytest.mark.parametrize("out_dtype", [fa.FA_BF16, fa.FA_F32])
@pytest.mark.parametrize("chunk_pages", [0, 3])
def test_packed_dag_prefill_small_every_row(out_dtype, chunk_pages):
    w = W.packed_dag_prefill(**W.PREFILL_SMALL)
    out, lse, st = run_prefill(w, out_dtype, chunk_pages=chunk_pages)
    if chunk_pages:
        assert st["items_skipped"] > 0  # short chunks: whole (row group, chunk) pairs left out
    ref_out, ref_lse = oracle.fork_attn(w)
    assert_parity(out, lse, ref_out, ref_lse, f"packed DAG prefill, chunks of {chunk_pages}")


@pytest.mark.parametrize("seed", range(12))
def test_random_prefill_shaped_caches(seed):
    # mid-page starts, shared and duplicated segments, drops (a token may see nothing at
    # all), short chunks so that skipped pairs and per-item page limits both occur; row
    # kernels and the tcgen05 kernel
    w = as_prefill(W.random_dag(3000 + seed, num_q_heads=8 if seed % 2 else 16, num_kv_heads=2,
                                n_segs=5, n_branches=4, max_list=4, max_seg_len=200,
                                pool_pages=40, drop_p=(0.0, 0.3, 0.9)[seed % 3], values=False))
    tmin = (0, 1, -1)[seed % 3]
    out, lse, _ = run_prefill(w, fa.FA_F32, chunk_pages=(0, 2, 5, 1)[seed % 4], tensor_min_rows=tmin)
    ref_out, ref_lse = oracle.fork_attn(w)
    assert_parity(out, lse, ref_out, ref_lse, f"seed {seed}")


def test_packed_dag_prefill_full_size_sampled_rows():
    # the workload the benchmark times, in its launch configuration: sampled rows against
    # the oracle, including each branch's first and last token (the causal edges)
    w = W.packed_dag_prefill(device="cuda")
    out, lse, st = run_prefill(w, poison=False)
    assert st["num_items_tensor"] > 0
    Hq = w.num_q_heads
    rng = np.random.default_rng(6)
    picks = set(rng.choice(w.total_q * Hq, size=1500, replace=False).tolist())
    for b in range(w.num_branches):
        for t in (int(w.branch_q_off[b]), int(w.branch_q_off[b + 1]) - 1):
            picks.update(range(t * Hq, t * Hq + Hq))
    rows = np.array(sorted(picks), dtype=np.int64)
    w.q, w.k_pages, w.v_pages = w.q.cpu(), w.k_pages.cpu(), w.v_pages.cpu()
    ref_out, ref_lse = oracle.fork_attn(w, rows=rows)
    assert_parity(out[rows], lse[rows], ref_out, ref_lse, "packed DAG prefill full")


def test_prefill_is_deterministic_and_a_decode_of_its_last_tokens_agrees():
    # run to run bitwise; and the last token of every branch, decoded on its own (n_q = 1),
    # equals the prefill's row for it within the tolerances
    w = W.packed_dag_prefill(**W.PREFILL_SMALL)
    a = run_prefill(w, fa.FA_F32)
    b = run_prefill(w, fa.FA_F32)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    last = w.branch_q_off[1:] - 1
    d = W.Workload(w.name, w.num_q_heads, w.num_kv_heads, w.page_ids, w.segs, w.branch_seg_off,
                   w.branch_segs, np.arange(w.num_branches + 1, dtype=np.int32), None, None,
                   w.num_pages_pool, meta=dict(w.meta))
    d.q, d.k_pages, d.v_pages = w.q[torch.as_tensor(last)], w.k_pages, w.v_pages
    out, lse, _ = run_prefill(d, fa.FA_F32)
    Hq = w.num_q_heads
    rows = np.concatenate([np.arange(t * Hq, t * Hq + Hq) for t in last])
    assert_parity(out, lse, a[0][rows].astype(np.float64), a[1][rows].astype(np.float64), "last tokens")
