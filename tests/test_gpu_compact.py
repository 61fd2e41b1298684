"""GPU parity of physical compaction with optional repositioning (through the C ABI) against
the fp64 oracle: V and un-repositioned K bit-exact; repositioned K within half a bf16 ulp of
the fp64 rotation (fp32 arithmetic on the device); nothing outside the destination slots
written; a decode over the compacted cache equals the oracle on the original one."""
import copy

import numpy as np
import pytest
import torch

import oracle
import shared_prefix_paged_attn_b300 as fa
from oracle import compact as C
from shared_prefix_paged_attn_b300 import workloads as W

pytestmark = pytest.mark.gpu


def compact_on_gpu(w, branches, reposition, base=10000.0):
    dev = torch.device("cuda")
    kept_want = [len(C.kept_indices(w, b)) for b in branches]
    need = sum((r + 15) // 16 for r in kept_want)
    pool = w.num_pages_pool
    shape = (pool + need + 1,) + tuple(w.k_pages.shape[1:])
    filler = torch.Generator().manual_seed(9)
    k = torch.randn(shape, generator=filler).to(torch.bfloat16)
    v = torch.randn(shape, generator=filler).to(torch.bfloat16)
    k[:pool], v[:pool] = w.k_pages, w.v_pages
    k0, v0 = k.clone(), v.clone()
    w2 = copy.copy(w)
    w2.num_pages_pool = shape[0]
    fresh = np.arange(pool, pool + need, dtype=np.int32)
    plan = fa.fork_attn_compact_create(w2, branches, fresh, reposition=reposition, rope_base=base)
    kept, wb = plan.sizes()
    assert kept.tolist() == kept_want
    kd, vd = k.to(dev), v.to(dev)
    work = torch.empty(wb // 4 + 64, dtype=torch.int32, device=dev)
    fa.fork_attn_compact_upload(plan, work)
    fa.fork_attn_compact_run(plan, kd, vd)
    torch.cuda.synchronize()
    return kd.cpu(), vd.cpu(), k0, v0, fresh, kept_want


def _check(w, branches, reposition, base=10000.0):
    kd, vd, k0, v0, fresh, kept = compact_on_gpu(w, branches, reposition, base)
    written = torch.zeros(kd.shape[0], kd.shape[2], dtype=torch.bool)  # (page, slot)
    at = 0
    for b, r in zip(branches, kept):
        K, V, _ = C.compact(w, b, reposition=reposition, base=base)
        pages = torch.as_tensor(fresh[at:at + (r + 15) // 16].astype(np.int64))
        at += (r + 15) // 16
        n = torch.arange(r)
        pg, sl = pages[n // 16], n % 16
        written[pg, sl] = True
        got_v = vd[pg, :, sl, :].double().numpy()
        got_k = kd[pg, :, sl, :].double().numpy()
        assert np.array_equal(got_v, V)
        if not reposition:
            assert np.array_equal(got_k, K)
        else:
            # bf16 rounding of an fp32 rotation: half a bf16 ulp of the exact value, plus the
            # fp32 error, which scales with the pair's operands (not with the possibly
            # cancelling result)
            ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(K), 1e-30))) - 7)
            src = C.compact(w, b)[0]
            pair = np.abs(src[..., :64]) + np.abs(src[..., 64:])
            opnd = np.concatenate([pair, pair], axis=-1)
            err = np.abs(got_k - K)
            assert np.all(err <= 0.5 * ulp + 1e-6 * opnd + 1e-9), err.max()
    # every slot outside the destinations keeps its bits (sources included)
    keep = ~written
    assert torch.equal(kd.transpose(1, 2)[keep], k0.transpose(1, 2)[keep])
    assert torch.equal(vd.transpose(1, 2)[keep], v0.transpose(1, 2)[keep])


@pytest.mark.parametrize("seed", range(8))
@pytest.mark.parametrize("reposition", [False, True])
def test_random_caches(seed, reposition):
    w = W.random_dag(500 + seed, n_branches=5, n_segs=5, max_seg_len=300, pool_pages=60,
                     drop_p=(0.0, 0.3, 0.9)[seed % 3])
    _check(w, list(range(w.num_branches)), reposition)


@pytest.mark.parametrize("cfg", [1, 2, 4])
def test_small_workloads_with_reposition(cfg):
    w = W.make(cfg, small=True)
    _check(w, list(range(min(w.num_branches, 4))), True, base=500000.0)


def test_long_position_changes_keep_full_precision():
    # the rolling-drop prefix drops tens of thousands of positions: the exact angle reduction
    # must keep the rotation to bf16 rounding for changes of that size
    w = W.make(4, small=True)
    kept = C.kept_indices(w, 0)
    assert (kept - np.arange(len(kept))).max() > 1000
    _check(w, [0], True)


def test_decode_over_the_compacted_cache_matches_the_original():
    # compaction without repositioning changes storage only: a branch's packed copy, read as
    # one segment with nothing dropped, gives the original decode
    # one query token per branch: its causal limit is the whole kept sequence in both layouts
    w = W.random_dag(77, n_branches=4, n_segs=4, max_seg_len=200, pool_pages=40, drop_p=0.3, max_nq=1)
    branches = list(range(w.num_branches))
    kd, vd, _, _, fresh, kept = compact_on_gpu(w, branches, False)
    c = copy.copy(w)
    c.k_pages, c.v_pages = kd, vd
    c.num_pages_pool = kd.shape[0]
    page_ids, segs, at = [], [], 0
    for r in kept:
        npg = (r + 15) // 16
        segs.append((len(page_ids), 0, r))
        page_ids.extend(fresh[at:at + npg].tolist())
        at += npg
    c.page_ids = np.asarray(page_ids, np.int32)
    c.segs = np.asarray(segs, np.int32).reshape(-1, 3)
    c.branch_seg_off = np.arange(len(kept) + 1, dtype=np.int32)
    c.branch_segs = np.arange(len(kept), dtype=np.int32)
    c.vis_bits, c.vis_word_off = None, None
    dev = torch.device("cuda")
    run = fa.ForkAttention(c, out_dtype=fa.FA_F32)
    out, lse = run(c.q.to(dev), c.k_pages.to(dev), c.v_pages.to(dev))
    torch.cuda.synchronize()
    ref_out, ref_lse = oracle.fork_attn(w)  # the original cache, with its drops
    out = out.cpu().numpy().reshape(-1, 128)
    lse = lse.cpu().numpy().reshape(-1)
    fin = ~np.isneginf(ref_lse)
    assert np.array_equal(np.isneginf(lse), ~fin)
    assert np.abs(out[fin] - ref_out[fin]).max() <= 1e-2
    assert np.abs(lse[fin] - ref_lse[fin]).max() <= 1e-3


def _check_shared(w, branches, reposition, base=10000.0):
    # share_prefix: the common prefix's kept entries packed once, then each branch's own;
    # every branch, read through [shared pages][its own pages], holds exactly what the
    # per-branch definition gives (so the rotation of a shared entry is the same for every
    # reader: the common prefix starts at logical index 0)
    dev = torch.device("cuda")
    P, rs = C.common_prefix(w, branches)
    want = [len(C.kept_indices(w, b)) for b in branches]
    need = (rs + 15) // 16 + sum((r - rs + 15) // 16 for r in want)
    pool = w.num_pages_pool
    shape = (pool + need,) + tuple(w.k_pages.shape[1:])
    filler = torch.Generator().manual_seed(10)
    k = torch.randn(shape, generator=filler).to(torch.bfloat16)
    v = torch.randn(shape, generator=filler).to(torch.bfloat16)
    k[:pool], v[:pool] = w.k_pages, w.v_pages
    k0, v0 = k.clone(), v.clone()
    w2 = copy.copy(w)
    w2.num_pages_pool = shape[0]
    fresh = np.arange(pool, pool + need, dtype=np.int32)
    plan = fa.fork_attn_compact_create(w2, branches, fresh, reposition=reposition, rope_base=base,
                                       share_prefix=True)
    assert plan.shared() == (rs, P)
    kept, wb = plan.sizes()
    assert kept.tolist() == want
    kd, vd = k.to(dev), v.to(dev)
    work = torch.empty(wb // 4 + 64, dtype=torch.int32, device=dev)
    fa.fork_attn_compact_upload(plan, work)
    fa.fork_attn_compact_run(plan, kd, vd)
    torch.cuda.synchronize()
    kd, vd = kd.cpu(), vd.cpu()
    written = torch.zeros(kd.shape[0], kd.shape[2], dtype=torch.bool)
    shared_pages = fresh[:(rs + 15) // 16].astype(np.int64)
    at = len(shared_pages)
    for b, r in zip(branches, want):
        own = fresh[at:at + (r - rs + 15) // 16].astype(np.int64)
        at += len(own)
        n = np.arange(r)
        pg = np.where(n < rs, shared_pages[np.minimum(n, max(rs - 1, 0)) // 16] if rs else 0,
                      own[np.maximum(n - rs, 0) // 16] if len(own) else 0)
        sl = np.where(n < rs, n % 16, (n - rs) % 16)
        pg, sl = torch.as_tensor(pg), torch.as_tensor(sl)
        written[pg, sl] = True
        K, V, _ = C.compact(w, b, reposition=reposition, base=base)
        assert np.array_equal(vd[pg, :, sl, :].double().numpy(), V)
        got_k = kd[pg, :, sl, :].double().numpy()
        if not reposition:
            assert np.array_equal(got_k, K)
        else:
            ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(K), 1e-30))) - 7)
            src = C.compact(w, b)[0]
            pair = np.abs(src[..., :64]) + np.abs(src[..., 64:])
            opnd = np.concatenate([pair, pair], axis=-1)
            assert np.all(np.abs(got_k - K) <= 0.5 * ulp + 1e-6 * opnd + 1e-9)
    assert at == need
    keep = ~written
    assert torch.equal(kd.transpose(1, 2)[keep], k0.transpose(1, 2)[keep])
    assert torch.equal(vd.transpose(1, 2)[keep], v0.transpose(1, 2)[keep])


@pytest.mark.parametrize("cfg", [1, 2, 4])
@pytest.mark.parametrize("reposition", [False, True])
def test_shared_prefix_mode(cfg, reposition):
    w = W.make(cfg, small=True)
    _check_shared(w, list(range(min(w.num_branches, 6))), reposition)


@pytest.mark.parametrize("seed", range(4))
def test_shared_prefix_mode_random_caches(seed):
    # random caches: the common prefix is often empty or a single segment
    w = W.random_dag(700 + seed, n_branches=4, n_segs=4, max_seg_len=200, pool_pages=50,
                     drop_p=(0.0, 0.3)[seed % 2])
    _check_shared(w, list(range(w.num_branches)), seed >= 2)
