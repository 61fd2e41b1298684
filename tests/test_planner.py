"""Host planner (C++) through the C ABI, on the CPU: validation, counters, structure."""
import ctypes

import numpy as np
import pytest

import oracle
import shared_prefix_paged_attn_b300 as fa
from shared_prefix_paged_attn_b300 import _lib, build
from shared_prefix_paged_attn_b300 import workloads as W


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()


def _plan_rc(w, **kw):
    try:
        fa.plan_for(w, **kw)
        return 0
    except fa.ForkAttnError as e:
        return e.status


def test_unique_counters_match_the_oracle_on_all_five_configs():
    for c in range(1, 6):
        w = W.make(c, values=False)
        st = fa.plan_for(w).stats()
        slots, pages = oracle.unique_slots(w)
        assert st["unique_visible_slots"] == slots
        assert st["touched_pages"] == pages
        assert st["total_q"] == w.total_q


def test_unique_counters_on_random_caches():
    for seed in range(20):
        w = W.random_dag(seed, n_branches=5, n_segs=5, pool_pages=6, values=False)
        st = fa.plan_for(w).stats()
        assert (st["unique_visible_slots"], st["touched_pages"]) == oracle.unique_slots(w)


def test_shared_prefix_pages_are_listed_once():
    w = W.config1(values=False)
    st = fa.plan_for(w).stats()
    # 64 prefix pages + 4 x 16 private pages, each read once per KV head and row group
    assert st["touched_pages"] == 64 + 4 * 16
    assert st["kv_bytes_rows"] == (64 + 64) * 16 * 128 * 2 * 2 * w.num_kv_heads


def test_fully_dropped_pages_are_skipped():
    w = W.config4(shrink=16, values=False)
    st = fa.plan_for(w).stats()
    listed = sum(w.branch_len(b) for b in range(w.num_branches))
    assert st["touched_pages"] * 16 < listed  # dropped tool segments are never read
    assert st["kv_bytes_rows"] / (w.num_kv_heads * 512) < (w.num_pages_pool * 16) * 8


def test_validation_errors():
    good = W.random_dag(3, values=False)
    assert _plan_rc(good) == 0

    def variant(**kw):
        import copy
        v = copy.copy(good)
        for k, val in kw.items():
            setattr(v, k, val)
        return v

    bad_page = good.page_ids.copy(); bad_page[0] = good.num_pages_pool
    assert _plan_rc(variant(page_ids=bad_page)) == -4
    bad_seg = good.segs.copy(); bad_seg[0, 1] = 16
    assert _plan_rc(variant(segs=bad_seg)) == -4
    bad_len = good.segs.copy(); bad_len[0, 2] = 0
    assert _plan_rc(variant(segs=bad_len)) == -2
    past_end = good.segs.copy(); past_end[0, 0] = len(good.page_ids)
    assert _plan_rc(variant(segs=past_end)) == -4
    bad_list = good.branch_segs.copy(); bad_list[0] = len(good.segs)
    assert _plan_rc(variant(branch_segs=bad_list)) == -4
    big_q = good.branch_q_off.copy(); big_q[1:] += 10 ** 6
    assert _plan_rc(variant(branch_q_off=big_q)) == -2
    if good.vis_bits is not None:
        assert _plan_rc(variant(vis_bits=good.vis_bits[:1])) == -4
    for hq, hkv, rc in ((6, 4, -3), (64, 1, -3)):
        assert _plan_rc(variant(num_q_heads=hq, num_kv_heads=hkv)) == rc
    # a page-head index (page x Hkv + head, one page past the pool too) must fit in int32
    assert _plan_rc(variant(num_q_heads=1 << 16, num_kv_heads=1 << 16, num_pages_pool=(1 << 15) - 2)) == 0
    assert _plan_rc(variant(num_q_heads=1 << 16, num_kv_heads=1 << 16, num_pages_pool=(1 << 15) - 1)) == -4
    for knob in ("chunk_pages", "num_sms", "tensor_ctas", "tensor_chunk_pages"):
        assert _plan_rc(good, **{knob: -1}) == -2


def test_reserved_planner_fields_must_be_zero():
    w = W.config1(values=False)
    lib = _lib.load()
    dims = _lib.FaDims(8, 2, 128, 16, 1.0 / np.sqrt(128), fa.FA_BF16)
    keep = [np.ascontiguousarray(x) for x in (w.page_ids, w.segs, w.branch_seg_off, w.branch_segs)]
    desc = _lib.FaDesc()
    desc.page_ids, desc.num_page_ids = keep[0].ctypes.data, len(w.page_ids)
    desc.segs, desc.num_segs = keep[1].ctypes.data, len(w.segs)
    desc.branch_seg_off, desc.branch_segs = keep[2].ctypes.data, keep[3].ctypes.data
    desc.num_branches = len(w.branch_seg_off) - 1
    desc.num_pages_pool = w.num_pages_pool
    handle = ctypes.c_void_p()
    for i in range(4):
        opts = _lib.FaPlanOpts()
        if i < 2:
            opts.reserved[i] = 1
        elif i == 2:
            opts.representatives = 2  # only 0 or 1
        rc = lib.fork_attn_plan_create(ctypes.byref(dims), ctypes.byref(desc), ctypes.byref(opts),
                                       ctypes.byref(handle))
        assert rc == (-2 if i < 3 else 0)
    assert lib.fork_attn_plan_destroy(handle) == 0


def test_unsupported_dims_and_nulls():
    w = W.config1(values=False)
    with pytest.raises(fa.ForkAttnError) as e:
        fa.fork_attn_plan_create(8, 2, w.page_ids, w.segs, w.branch_seg_off, w.branch_segs,
                                 w.num_pages_pool, head_dim=64)
    assert e.value.status == -3
    with pytest.raises(fa.ForkAttnError) as e:
        fa.fork_attn_plan_create(8, 2, w.page_ids, w.segs, w.branch_seg_off, w.branch_segs,
                                 w.num_pages_pool, page_size=32)
    assert e.value.status == -3
    lib = _lib.load()
    assert lib.fork_attn_plan_create(None, None, None, None) == -1
    assert lib.fork_attn_decode(None, None, None, None, None, None, None) == -1


def test_decode_before_upload_is_rejected():
    w = W.config1(values=False)
    p = fa.plan_for(w)
    fake = ctypes.c_void_p(256)
    rc = _lib.load().fork_attn_decode(fake, fake, fake, p.handle, fake, fake, None)
    assert rc == -6


def test_upload_rejects_small_or_misaligned_buffers():
    w = W.config1(values=False)
    p = fa.plan_for(w)
    pb, sb = p.sizes()
    lib = _lib.load()
    assert lib.fork_attn_plan_upload(p.handle, ctypes.c_void_p(256), pb - 1, ctypes.c_void_p(512), sb, None) == -9
    assert lib.fork_attn_plan_upload(p.handle, ctypes.c_void_p(260), pb, ctypes.c_void_p(512), sb, None) == -5
    assert lib.fork_attn_plan_upload(p.handle, ctypes.c_void_p(256), pb, None, sb, None) == -1


def test_plan_is_deterministic():
    w = W.config3(shrink=16, values=False)
    a, b = fa.plan_for(w), fa.plan_for(w)
    assert a.sizes() == b.sizes() and a.stats() == b.stats()


def _visible_pairs(w, b):
    """Sum over branch b's query tokens i of |V_{b,i}|: its visible entries at positions up to
    the token's own, n_b - n_q + i (the definition's visible set, counted by brute force)."""
    n = w.branch_len(b)
    nq = int(w.branch_q_off[b + 1] - w.branch_q_off[b])
    j = np.arange(n)
    if w.vis_bits is None:
        vis = np.ones(n, bool)
    else:
        words = w.vis_bits[w.vis_word_off[b]:w.vis_word_off[b + 1]]
        vis = ((words[j // 32] >> (j % 32)) & 1).astype(bool)
    return sum(int(vis[:n - nq + i + 1].sum()) for i in range(nq))


@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5])
def test_flop_counters_match_the_definition(cfg):
    # QK^T and P V: 2 x 128 multiply-adds for every (query row, KV head, visible entry at or
    # before the query token's position)
    w = W.make(cfg, small=True, values=False)
    st = fa.plan_for(w).stats()
    G = w.num_q_heads // w.num_kv_heads
    want = sum(_visible_pairs(w, b) for b in range(w.num_branches)) * G * w.num_kv_heads * 4 * 128
    assert st["flops_rows"] + st["flops_tensor"] == want
    assert st["flops_tensor"] > 0 or cfg == 1


@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5])
def test_per_kernel_slot_counters(cfg):
    # each row kernel's count covers the chunks it reads; together they cover every row chunk,
    # a chunk split between both kernels counting in both
    w = W.make(cfg, small=True, values=False)
    for tmin in (0, -1):
        st = fa.plan_for(w, tensor_min_rows=tmin).stats()
        r8, r32, rows = st["unique_slots_row8"], st["unique_slots_row32"], st["unique_slots_rows"]
        assert max(r8, r32) <= rows <= r8 + r32
        assert (r8 > 0) == (st["num_items_row8"] > 0)
        assert (r32 > 0) == (st["num_items_rows"] > st["num_items_row8"])
        assert rows + st["unique_slots_tensor"] == st["unique_visible_slots"]
        if st["num_items_tensor"]:
            assert 1 <= st["tensor_ctas"] <= min(148, st["num_items_tensor"])
        else:
            assert st["tensor_ctas"] == 0
    st = fa.plan_for(w, tensor_min_rows=1, tensor_ctas=3).stats()
    assert st["tensor_ctas"] == min(3, st["num_items_tensor"])


def test_row_chunk_length_follows_the_item_count():
    # long private runs with many row items get chunks of up to 128 pages; the flat-fork
    # workload, whose 64-page chunks give only 256 row items, keeps them
    def mean_pages(st):
        return st["kv_bytes_rows"] / st["num_items_rows"] / (16 * 128 * 2 * 2)
    long_ctx = fa.plan_for(W.make(4, values=False)).stats()
    flat = fa.plan_for(W.make(2, values=False)).stats()
    assert long_ctx["num_items_rows"] >= 3 * 148 and mean_pages(long_ctx) > 64
    assert flat["num_items_rows"] == 256 and mean_pages(flat) <= 64
    # an explicit chunk size overrides the choice
    pinned = fa.plan_for(W.make(4, values=False), chunk_pages=64).stats()
    assert mean_pages(pinned) <= 64 and pinned["num_items_rows"] > long_ctx["num_items_rows"]


def test_tensor_cta_split_matches_the_measured_optima():
    # the planner's replay of the work counter picks the counts measured best on B300: one
    # item per CTA for the flat fork's 128 equal items, two per CTA for the 240 items of the
    # long-context workload (112 CTAs would leave 16 of them a third item)
    assert fa.plan_for(W.make(2, values=False)).stats()["tensor_ctas"] == 128
    assert fa.plan_for(W.make(4, values=False)).stats()["tensor_ctas"] == 120


@pytest.mark.parametrize("seed", range(4))
def test_prefill_shaped_descriptors_plan_like_decodes(seed):
    # every token a query (n_q = n_b): the packed-prefill case of the same definition; the
    # planner accepts it and its counters keep their meaning
    w = W.random_dag(900 + seed, n_branches=3, n_segs=3, max_seg_len=60, pool_pages=30,
                     drop_p=0.2, values=False)
    lens = [w.branch_len(b) for b in range(w.num_branches)]
    w.branch_q_off = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    st = fa.plan_for(w).stats()
    assert st["total_q"] == sum(lens)
    assert (st["unique_visible_slots"], st["touched_pages"]) == oracle.unique_slots(w)
    G = w.num_q_heads // w.num_kv_heads
    # only the causally visible (query, key) pairs count: about half of the full rectangle
    want = sum(_visible_pairs(w, b) for b in range(w.num_branches)) * G * w.num_kv_heads * 4 * 128
    assert st["flops_rows"] + st["flops_tensor"] == want
    # one token too many is refused
    w.branch_q_off = w.branch_q_off.copy()
    w.branch_q_off[1:] += 1
    with pytest.raises(fa.ForkAttnError):
        fa.plan_for(w)


def test_packed_dag_prefill_workload_structure():
    # one branch per thread: the root's tokens query the root; thread j's tokens query the
    # root, one mounted terminal block of an earlier thread (j >= 1), and its own segment
    w = W.packed_dag_prefill(shrink=16, values=False)
    assert w.num_branches == 9
    root = int(w.branch_segs[w.branch_seg_off[0]])
    assert w.branch_len(0) == int(w.branch_q_off[1]) == 256
    for b in range(1, w.num_branches):
        lst = w.branch_segs[w.branch_seg_off[b]:w.branch_seg_off[b + 1]]
        assert int(lst[0]) == root and len(lst) == (2 if b == 1 else 3)
        own = int(lst[-1])
        assert int(w.branch_q_off[b + 1] - w.branch_q_off[b]) == int(w.segs[own][2])
        if b >= 2:  # the mount reads the last 32 tokens of an earlier thread's pages in place
            m = w.segs[int(lst[1])]
            assert int(m[2]) == 32
            slots = set(W.logical_slots(w, b)[256:256 + 32].tolist())
            assert any(slots <= set(W.logical_slots(w, a)[-32:].tolist()) for a in range(1, b))


@pytest.mark.parametrize("chunk_pages", [0, 3])
def test_packed_dag_prefill_plan(chunk_pages):
    # causally visible pairs only; with short chunks whole (row group, chunk) pairs are left
    # out (every row of the group lies before the chunk), with one chunk per run none are
    w = W.packed_dag_prefill(shrink=16, values=False)
    st = fa.plan_for(w, chunk_pages=chunk_pages).stats()
    G = w.num_q_heads // w.num_kv_heads
    want = sum(_visible_pairs(w, b) for b in range(w.num_branches)) * G * w.num_kv_heads * 4 * 128
    assert st["flops_rows"] + st["flops_tensor"] == want
    assert st["total_q"] == w.total_q
    assert (st["unique_visible_slots"], st["touched_pages"]) == oracle.unique_slots(w)
    if chunk_pages:
        assert st["items_skipped"] > 0
    full = fa.plan_for(W.packed_dag_prefill(values=False)).stats()
    assert full["num_items_tensor"] > 0 and full["num_items_rows"] == 0


def test_representatives_plans():
    # representative queries see the whole list: n_q may exceed n_b, every (row, visible
    # entry) pair counts, a branch's rows (n_q x G) must fit one 256-row group
    w = W.make(2, small=True)
    ws = W.with_representatives(w, list(range(3)), reps=32)
    st = fa.plan_for(ws, representatives=1).stats()
    G = ws.num_q_heads // ws.num_kv_heads
    vis = sum(len(__import__("oracle.compact", fromlist=["x"]).kept_indices(ws, b)) for b in range(3))
    assert st["flops_rows"] + st["flops_tensor"] == vis * 32 * G * ws.num_kv_heads * 4 * 128
    assert st["num_items_rows"] == 0 and st["num_items_tensor"] > 0
    E, nw = fa.fork_attn_score_sizes(fa.plan_for(ws, representatives=1))
    assert E == sum(ws.branch_len(b) for b in range(3))
    assert nw == sum((ws.branch_len(b) + 31) // 32 for b in range(3))
    with pytest.raises(fa.ForkAttnError):
        fa.fork_attn_score_sizes(fa.plan_for(w))  # a decode plan has no scores
    tiny = W.random_dag(5, n_branches=2, max_seg_len=10, values=True)
    t = W.with_representatives(tiny, reps=40)  # more representatives than entries
    assert _plan_rc(t, representatives=1) == 0
    assert _plan_rc(t) == -2
    big = W.with_representatives(W.make(4, small=True), [0], reps=33)  # 33 x 8 rows > 256
    assert _plan_rc(big, representatives=1) == -3
