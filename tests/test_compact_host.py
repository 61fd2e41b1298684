"""Compaction planner (host, C ABI) on the CPU: kept counts against the oracle, refusals."""
import numpy as np
import pytest

import shared_prefix_paged_attn_b300 as fa
from oracle import compact as C
from shared_prefix_paged_attn_b300 import build
from shared_prefix_paged_attn_b300 import workloads as W


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()


def _source_pages(w, branches):
    pages = set()
    for b in branches:
        pages |= set((C.branch_slots(w, b) // 16).tolist())
    return pages


def _grow(w, extra):
    # a larger pool: `extra` fresh destination pages after the original ones
    fresh = np.arange(w.num_pages_pool, w.num_pages_pool + extra, dtype=np.int32)
    w.num_pages_pool += extra
    return fresh


@pytest.mark.parametrize("seed", range(8))
def test_kept_counts_match_the_oracle(seed):
    w = W.random_dag(400 + seed, n_branches=5, drop_p=(0.0, 0.3, 0.9)[seed % 3], values=False)
    branches = list(range(w.num_branches))[:: 1 + seed % 2]
    want = [len(C.kept_indices(w, b)) for b in branches]
    need = sum((r + 15) // 16 for r in want)
    plan = fa.fork_attn_compact_create(w, branches, _grow(w, need + 3))
    kept, work = plan.sizes()
    assert kept.tolist() == want
    assert work >= 12 * max(sum(want), 1)


def test_refusals():
    w = W.random_dag(5, n_branches=3, drop_p=0.2, values=False)
    need = sum((len(C.kept_indices(w, b)) + 15) // 16 for b in range(3))
    fresh = _grow(w, need + 4)

    def rc(branches=(0, 1, 2), dst=None, **kw):
        try:
            fa.fork_attn_compact_create(w, list(branches), fresh if dst is None else dst, **kw)
            return 0
        except fa.ForkAttnError as e:
            return e.status
    assert rc() == 0
    assert rc(branches=(3,)) == -2                      # no such branch
    assert rc(dst=fresh[: need - 1]) == -2              # too few destination pages
    src = sorted(_source_pages(w, [0]))
    assert rc(dst=np.concatenate([[src[0]], fresh]).astype(np.int32)) == -2  # overwrites a source
    dup = fresh.copy(); dup[1] = dup[0]
    assert rc(dst=dup) == -2                            # a page listed twice
    bad = fresh.copy(); bad[0] = w.num_pages_pool
    assert rc(dst=bad) == -4                            # out of the pool
    assert rc(reposition=True, rope_base=1.0) == -2     # no valid RoPE base
    assert rc(head_dim=64) == -3
    assert rc(branches=()) == 0                         # nothing to do is fine
