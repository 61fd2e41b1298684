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


@pytest.mark.parametrize("cfg", [1, 2, 4, 5])
def test_shared_prefix_mode_packs_the_common_prefix_once(cfg):
    # a fork's shared prefix (with the same drops for every reader) is the common prefix; it
    # takes ceil(r_s / 16) destination pages once, each branch the rest of its entries
    w = W.make(cfg, small=True, values=False)
    branches = list(range(min(w.num_branches, 6)))
    want = [len(C.kept_indices(w, b)) for b in branches]
    P, rs = C.common_prefix(w, branches)
    assert rs > 0
    need = (rs + 15) // 16 + sum((r - rs + 15) // 16 for r in want)
    fresh = _grow(w, need)
    plan = fa.fork_attn_compact_create(w, branches, fresh, share_prefix=True)
    kept, _ = plan.sizes()
    assert kept.tolist() == want
    assert plan.shared() == (rs, P)
    # exactly that many pages: one fewer is refused
    with pytest.raises(fa.ForkAttnError):
        fa.fork_attn_compact_create(w, branches, fresh[:-1], share_prefix=True)
    # without the mode nothing is shared
    assert fa.fork_attn_compact_create(w, branches, _grow(w, sum((r + 15) // 16 for r in want))).shared() == (0, 0)


def test_common_prefix_stops_at_the_first_difference():
    w = W.random_dag(9, n_branches=3, drop_p=0.0, values=False)
    w.branch_seg_off = np.array([0, 2, 4, 6], np.int32)
    w.branch_segs = np.array([0, 1, 0, 2, 0, 1], np.int32)
    n0 = int(w.segs[0][2])
    if int(w.segs[1][2]) == 0 or np.array_equal(C.branch_slots(w, 0)[n0:n0 + 1], C.branch_slots(w, 1)[n0:n0 + 1]):
        pytest.skip("segments 1 and 2 start on the same slot")
    assert C.common_prefix(w, [0, 1, 2])[0] == n0
    assert C.common_prefix(w, [0, 2])[0] == sum(int(w.segs[s][2]) for s in (0, 1))
    # a bit that differs at index 3 ends the prefix there
    bits = [np.ones(w.branch_len(b), bool) for b in range(3)]
    bits[1][3] = False
    w.vis_bits, w.vis_word_off = W._pack_branch_bits(bits)
    assert C.common_prefix(w, [0, 1])[0] == min(3, n0) and C.common_prefix(w, [0, 1])[1] == min(3, n0)
    need = 64
    plan = fa.fork_attn_compact_create(w, [0, 1], _grow(w, need), share_prefix=True)
    assert plan.shared() == (min(3, n0), min(3, n0))


def test_shared_prefix_refusals():
    w = W.random_dag(5, n_branches=3, drop_p=0.2, values=False)
    fresh = _grow(w, 64)
    import ctypes
    from shared_prefix_paged_attn_b300 import _lib
    for share, res in ((2, 0), (0, 1)):
        dims = _lib.FaCompactDims(w.num_kv_heads, 128, 16, 0, 10000.0, share, res)
        keep = [np.ascontiguousarray(x) for x in (w.page_ids, w.segs, w.branch_seg_off, w.branch_segs,
                                                 w.branch_q_off, w.vis_bits, w.vis_word_off)]
        desc = fa._desc(lambda x, dt: np.ascontiguousarray(x, dtype=dt).ctypes.data if x is not None else None,
                        *keep[:4], w.num_pages_pool, *keep[4:])
        br = np.array([0, 1], np.int32)
        h = ctypes.c_void_p()
        rc = _lib.load().fork_attn_compact_create(ctypes.byref(dims), ctypes.byref(desc), br.ctypes.data, 2,
                                                  fresh.ctypes.data, len(fresh), ctypes.byref(h))
        assert rc == -2
