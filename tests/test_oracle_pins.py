"""Pins for the fp64 oracle: checks against things other than the oracle itself.

* closed forms (one visible entry, identical keys, constant values);
* a special case that is a library routine (one branch, one segment: torch's fp64
  scaled-dot-product attention and logsumexp);
* an independent Python brute force over explicit membership sets on tiny random caches;
* the invariants the pages state: a fork reads what a copied context holds (Octopus,
  "Zero-Copy Radix Forking"), dropped entries have no effect (AKV, "AKV 如何工作？"), the
  log-sum-exp merge of split partials equals the unsplit result (Agentrix, "CUDA ForkAttention":
  shared and private parts computed apart, then merged per branch), physical page placement
  does not matter, and the causal rule for several new tokens per branch;
* the page-sharing arithmetic printed by Agentrix ("实验结果", 工具页面共享) for the
  unique-page counter.
"""
import copy
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from shared_prefix_paged_attn_b300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bits(w, b):
    n = w.branch_len(b)
    if w.vis_bits is None:
        return np.ones(n, dtype=bool)
    words = w.vis_bits[w.vis_word_off[b]:w.vis_word_off[b + 1]]
    return np.array([(int(words[j // 32]) >> (j % 32)) & 1 for j in range(n)], dtype=bool)


def _single_branch(length, n_q=1, tok_begin=0, hq=4, hkv=2, seed=0, values=True):
    """One branch over one segment stored in consecutive pages 0.. (no drops)."""
    n_pages = (tok_begin + length + 15) // 16
    w = W.Workload("single", hq, hkv, np.arange(n_pages, dtype=np.int32),
                   np.array([[0, tok_begin, length]], np.int32), np.array([0, 1], np.int32),
                   np.array([0], np.int32), np.array([0, n_q], np.int32), None, None, n_pages,
                   meta={"seed": seed})
    if values:
        W.fill_values(w)
    return w


# ------------------------------------------------------------------------------ closed forms

def test_single_visible_entry_gives_its_value_and_score():
    w = _single_branch(10, hq=2, hkv=1)
    w.q.zero_()
    w.q[0, :, 0] = 1.5
    w.k_pages[0, 0, 3].zero_()
    w.k_pages[0, 0, 3, 0] = -2.0
    vis = np.zeros(10, bool)
    vis[3] = True
    w.vis_bits, w.vis_word_off = W._pack_branch_bits([vis])
    out, lse = oracle.fork_attn(w)
    expect_s = 1.5 * -2.0 / math.sqrt(128)
    for h in range(2):
        assert lse[h] == pytest.approx(expect_s, abs=1e-15)
        np.testing.assert_array_equal(out[h], w.v_pages[0, 0, 3].double().numpy())


def test_identical_keys_give_mean_value_and_log_count():
    w = _single_branch(37, tok_begin=5, hq=4, hkv=2)
    w.k_pages[:] = w.k_pages[0, 0, 5]  # every slot holds the same key
    vis = np.ones(37, bool)
    vis[[0, 7, 20, 21]] = False
    w.vis_bits, w.vis_word_off = W._pack_branch_bits([vis])
    out, lse = oracle.fork_attn(w)
    slots = W.logical_slots(w, 0)[vis]
    for h in range(4):
        g = h // 2
        s = float((w.q[0, h].double() * w.k_pages[0, 0, 5].double()).sum()) / math.sqrt(128)
        vrows = w.v_pages.double().numpy()[slots // 16, g, slots % 16]
        assert lse[h] == pytest.approx(s + math.log(vis.sum()), abs=1e-12)
        np.testing.assert_allclose(out[h], vrows.mean(axis=0), atol=1e-12)


def test_constant_values_give_that_constant():
    w = _single_branch(50, n_q=3, hq=4, hkv=1)
    w.v_pages[:] = torch.linspace(-3, 3, 128).to(torch.bfloat16)
    out, _ = oracle.fork_attn(w)
    c = torch.linspace(-3, 3, 128).to(torch.bfloat16).double().numpy()
    for r in range(out.shape[0]):
        np.testing.assert_allclose(out[r], c, atol=1e-12)


def test_fully_masked_row_gives_zero_and_minus_infinity():
    w = _single_branch(20, hq=2, hkv=1)
    w.vis_bits, w.vis_word_off = W._pack_branch_bits([np.zeros(20, bool)])
    out, lse = oracle.fork_attn(w)
    assert np.all(out == 0) and np.all(np.isneginf(lse))


# ------------------------------------------------------------- library special case (SDPA)

@pytest.mark.parametrize("length,n_q,tok_begin", [(1, 1, 0), (77, 1, 3), (200, 4, 9),
                                                  (64, 8, 0)])
def test_single_branch_is_textbook_attention(length, n_q, tok_begin):
    hq, hkv = 8, 2
    w = _single_branch(length, n_q=n_q, tok_begin=tok_begin, hq=hq, hkv=hkv, seed=length)
    out, lse = oracle.fork_attn(w)
    slots = np.arange(length) + tok_begin
    K = w.k_pages.double()[torch.as_tensor(slots // 16), :, torch.as_tensor(slots % 16)]
    V = w.v_pages.double()[torch.as_tensor(slots // 16), :, torch.as_tensor(slots % 16)]
    K = K.repeat_interleave(hq // hkv, dim=1).transpose(0, 1)  # [Hq, n, D]
    V = V.repeat_interleave(hq // hkv, dim=1).transpose(0, 1)
    q = w.q.double().transpose(0, 1)  # [Hq, n_q, D]
    pos_q = torch.arange(length - n_q, length)[:, None]
    allowed = torch.arange(length)[None, :] <= pos_q
    ref = torch.nn.functional.scaled_dot_product_attention(q, K, V, attn_mask=allowed)
    logits = (q @ K.transpose(1, 2)) / math.sqrt(128)
    ref_lse = torch.logsumexp(logits.masked_fill(~allowed, -math.inf), dim=-1)
    got = torch.from_numpy(out).view(n_q, hq, 128).transpose(0, 1)
    got_lse = torch.from_numpy(lse).view(n_q, hq).transpose(0, 1)
    torch.testing.assert_close(got, ref, atol=1e-12, rtol=1e-12)
    torch.testing.assert_close(got_lse, ref_lse, atol=1e-12, rtol=1e-12)


# --------------------------------------------------------------- brute force (tiny caches)

def brute_force(w):
    """Explicit membership sets per (branch, query token); scipy's softmax / logsumexp."""
    D, G = w.head_dim, w.num_q_heads // w.num_kv_heads
    K = w.k_pages.double().numpy()
    V = w.v_pages.double().numpy()
    Q = w.q.double().numpy()
    rows_out, rows_lse = [], []
    for b in range(w.num_branches):
        entries = []  # logical index -> (physical page, slot)
        for s in w.branch_segs[w.branch_seg_off[b]:w.branch_seg_off[b + 1]]:
            po, tb, ln = (int(x) for x in w.segs[s])
            entries += [(int(w.page_ids[po + (tb + t) // 16]), (tb + t) % 16) for t in range(ln)]
        vis = _bits(w, b)
        n_q = int(w.branch_q_off[b + 1] - w.branch_q_off[b])
        for i in range(n_q):
            p = len(entries) - n_q + i
            members = sorted(j for j in range(len(entries)) if vis[j] and j <= p)
            for h in range(w.num_q_heads):
                g = h // G
                if not members:
                    rows_out.append(np.zeros(D))
                    rows_lse.append(-np.inf)
                    continue
                kk = np.stack([K[entries[j][0], g, entries[j][1]] for j in members])
                vv = np.stack([V[entries[j][0], g, entries[j][1]] for j in members])
                logits = kk @ Q[int(w.branch_q_off[b]) + i, h] * w.scale
                rows_lse.append(scipy.special.logsumexp(logits))
                rows_out.append(scipy.special.softmax(logits) @ vv)
    return np.array(rows_out), np.array(rows_lse)


@pytest.mark.parametrize("seed", range(12))
def test_matches_brute_force_on_tiny_random_caches(seed):
    w = W.random_dag(seed, n_branches=3, n_segs=3, max_seg_len=30, pool_pages=3,
                     drop_p=0.25 if seed % 3 else 0.0)
    out, lse = oracle.fork_attn(w)
    ref_out, ref_lse = brute_force(w)
    np.testing.assert_allclose(out, ref_out, atol=1e-12, rtol=1e-12)
    fin = np.isfinite(ref_lse)
    assert np.array_equal(fin, np.isfinite(lse))
    np.testing.assert_allclose(lse[fin], ref_lse[fin], atol=1e-12, rtol=1e-12)


def test_selected_rows_equal_full_rows():
    w = W.random_dag(99, n_branches=4, n_segs=5, pool_pages=5, max_nq=3)
    out, lse = oracle.fork_attn(w)
    rows = np.array([5, 0, w.total_q * w.num_q_heads - 1, 3, 5])
    o2, l2 = oracle.fork_attn(w, rows=rows, threads=3)
    np.testing.assert_array_equal(o2, out[rows])
    np.testing.assert_array_equal(l2, lse[rows])


# ------------------------------------------------------------------------------ invariants

def copied_context(w):
    """Every branch's logical sequence copied into fresh contiguous pages of its own."""
    pages, segs, k_rows, v_rows = [], [], [], []
    K, V = w.k_pages, w.v_pages
    next_page = 0
    bit_lists = []
    for b in range(w.num_branches):
        slots = W.logical_slots(w, b)
        n = len(slots)
        n_pages = (n + 15) // 16
        segs.append((len(pages), 0, n))
        pages.extend(range(next_page, next_page + n_pages))
        next_page += n_pages
        idx_p = torch.as_tensor(slots // 16)
        idx_s = torch.as_tensor(slots % 16)
        kb = torch.zeros((n_pages * 16, w.num_kv_heads, 128), dtype=K.dtype)
        vb = torch.zeros_like(kb)
        kb[:n] = K[idx_p, :, idx_s]
        vb[:n] = V[idx_p, :, idx_s]
        k_rows.append(kb.view(n_pages, 16, w.num_kv_heads, 128).transpose(1, 2))
        v_rows.append(vb.view(n_pages, 16, w.num_kv_heads, 128).transpose(1, 2))
        bit_lists.append(_bits(w, b))
    c = W.Workload("copied", w.num_q_heads, w.num_kv_heads, np.array(pages, np.int32),
                   np.array(segs, np.int32), np.arange(w.num_branches + 1, dtype=np.int32),
                   np.arange(w.num_branches, dtype=np.int32), w.branch_q_off.copy(), None,
                   None, next_page, meta=dict(w.meta))
    if w.vis_bits is not None:
        c.vis_bits, c.vis_word_off = W._pack_branch_bits(bit_lists)
    c.q = w.q
    c.k_pages = torch.cat(k_rows).contiguous()
    c.v_pages = torch.cat(v_rows).contiguous()
    return c


@pytest.mark.parametrize("cfg", [1, 3])
def test_fork_equals_copied_context(cfg):
    w = W.make(cfg, small=True) if cfg == 1 else W.config3(shrink=64)
    rows = np.arange(0, w.total_q * w.num_q_heads, 3)
    out, lse = oracle.fork_attn(w, rows=rows)
    c = copied_context(w)
    out2, lse2 = oracle.fork_attn(c, rows=rows)
    np.testing.assert_array_equal(out, out2)
    np.testing.assert_array_equal(lse, lse2)


def test_fork_equals_copied_context_random():
    for seed in range(5):
        w = W.random_dag(100 + seed, n_branches=4, n_segs=4, pool_pages=4)
        out, lse = oracle.fork_attn(w)
        out2, lse2 = oracle.fork_attn(copied_context(w))
        np.testing.assert_array_equal(out, out2)
        np.testing.assert_array_equal(lse, lse2)


def test_masked_entries_have_no_effect():
    w = W.config2(shrink=64)
    out, lse = oracle.fork_attn(w)
    G = w.num_q_heads
    for b in (0, 7):
        visible = W.logical_slots(w, b)[_bits(w, b)]
        g2 = copy.copy(w)
        g2.k_pages = w.k_pages.clone()
        g2.v_pages = w.v_pages.clone()
        mask = torch.ones(w.num_pages_pool * 16, dtype=torch.bool)
        mask[torch.as_tensor(visible)] = False
        kf = g2.k_pages.transpose(1, 2).reshape(-1, w.num_kv_heads, 128)
        vf = g2.v_pages.transpose(1, 2).reshape(-1, w.num_kv_heads, 128)
        kf[mask] = 3.0e4
        vf[mask] = -3.0e4
        g2.k_pages = kf.view(w.num_pages_pool, 16, w.num_kv_heads, 128).transpose(1, 2).contiguous()
        g2.v_pages = vf.view(w.num_pages_pool, 16, w.num_kv_heads, 128).transpose(1, 2).contiguous()
        rows = np.arange(b * G, (b + 1) * G)
        o2, l2 = oracle.fork_attn(g2, rows=rows)
        np.testing.assert_array_equal(o2, out[rows])
        np.testing.assert_array_equal(l2, lse[rows])


def test_all_ones_mask_equals_no_mask():
    w = W.config1(shrink=4)
    out, lse = oracle.fork_attn(w)
    w2 = copy.copy(w)
    w2.vis_bits, w2.vis_word_off = W._pack_branch_bits(
        [np.ones(w.branch_len(b), bool) for b in range(w.num_branches)])
    o2, l2 = oracle.fork_attn(w2)
    np.testing.assert_array_equal(o2, out)
    np.testing.assert_array_equal(l2, lse)


def lse_merge(parts):
    """Combine (out, lse) partials over disjoint entry sets."""
    lses = np.stack([p[1] for p in parts])
    L = np.logaddexp.reduce(lses, axis=0)
    out = sum(np.exp(p[1] - L)[:, None] * p[0] for p in parts)
    return out, L


@pytest.mark.parametrize("seed", range(4))
def test_lse_merge_of_split_partials_equals_unsplit(seed):
    w = W.config2(shrink=64) if seed == 0 else W.random_dag(200 + seed, n_branches=3,
                                                           drop_p=0.0, max_seg_len=60)
    out, lse = oracle.fork_attn(w)
    rng = np.random.default_rng(seed)
    a_bits, b_bits = [], []
    for b in range(w.num_branches):
        vis = _bits(w, b)
        n_q = int(w.branch_q_off[b + 1] - w.branch_q_off[b])
        pick = rng.random(len(vis)) < 0.5
        pick[-n_q:] = True  # every query row keeps at least its own entry in part A
        a_bits.append(vis & pick)
        b_bits.append(vis & ~pick)
    wa, wb = copy.copy(w), copy.copy(w)
    wa.vis_bits, wa.vis_word_off = W._pack_branch_bits(a_bits)
    wb.vis_bits, wb.vis_word_off = W._pack_branch_bits(b_bits)
    merged_out, merged_lse = lse_merge([oracle.fork_attn(wa), oracle.fork_attn(wb)])
    np.testing.assert_allclose(merged_out, out, atol=1e-12, rtol=1e-10)
    np.testing.assert_allclose(merged_lse, lse, atol=1e-12, rtol=1e-12)


def test_physical_page_permutation_changes_nothing():
    w = W.config3(shrink=64)
    rows = np.arange(0, w.total_q * w.num_q_heads, 5)
    out, lse = oracle.fork_attn(w, rows=rows)
    perm = torch.randperm(w.num_pages_pool, generator=torch.Generator().manual_seed(5))
    w2 = copy.copy(w)
    w2.page_ids = perm.numpy()[w.page_ids].astype(np.int32)
    w2.k_pages = torch.empty_like(w.k_pages)
    w2.v_pages = torch.empty_like(w.v_pages)
    w2.k_pages[perm] = w.k_pages
    w2.v_pages[perm] = w.v_pages
    o2, l2 = oracle.fork_attn(w2, rows=rows)
    np.testing.assert_array_equal(o2, out)
    np.testing.assert_array_equal(l2, lse)


def test_multi_token_query_equals_truncated_single_token_decode():
    w = W.config5(shrink=64, requests=2)
    out, lse = oracle.fork_attn(w)
    Hq = w.num_q_heads
    for b in (0, 9, 15):
        n_q = int(w.branch_q_off[b + 1] - w.branch_q_off[b])
        assert n_q == 8
        for i in range(n_q):
            t = copy.copy(w)
            cut = n_q - 1 - i  # drop the later new tokens from the last segment
            segs = w.segs.copy()
            last = int(w.branch_segs[w.branch_seg_off[b + 1] - 1])
            segs[last, 2] -= cut
            t.segs = segs
            t.branch_q_off = w.branch_q_off.copy()
            t.branch_q_off[b + 1:] -= (n_q - 1)
            t.q = torch.cat([w.q[:int(w.branch_q_off[b])],
                             w.q[int(w.branch_q_off[b]) + i:int(w.branch_q_off[b]) + i + 1],
                             w.q[int(w.branch_q_off[b + 1]):]])
            # the other branches keep their own lists; only branch b's last segment is cut,
            # so restrict the comparison to branch b (its segment is private)
            row_t = (int(w.branch_q_off[b])) * Hq
            rows = np.arange(row_t, row_t + Hq)
            o1, l1 = oracle.fork_attn(t, rows=rows)
            ref_rows = np.arange((int(w.branch_q_off[b]) + i) * Hq,
                                 (int(w.branch_q_off[b]) + i + 1) * Hq)
            np.testing.assert_allclose(o1, out[ref_rows], atol=1e-13)
            np.testing.assert_allclose(l1, lse[ref_rows], atol=1e-13)


# ------------------------------------------------------------------- page-sharing golden

def test_unique_page_counter_matches_the_page_sharing_example():
    g = json.load(open(os.path.join(GOLDEN, "agentrix_page_sharing.json")))
    n_pages = g["object_mib"] * 1024 // g["page_kib"]  # 2048 pages of 4 KiB
    branches = g["branches"]
    # one 4 KiB page = 16 slots x 1 KV head x 128 dims x 2 bytes (K only)
    edited = [7 + 250 * b for b in range(branches)]
    page_ids = list(range(n_pages)) + [n_pages + b for b in range(branches)]
    segs, lists = [], []
    for b, k in enumerate(edited):
        before = (0, 0, 16 * k)
        mine = (n_pages + b, 0, 16)
        after = (k + 1, 0, 16 * (n_pages - k - 1))
        base = len(segs)
        segs += [before, mine, after]
        lists.append([base, base + 1, base + 2])
    w = W.Workload("cow", 1, 1, np.array(page_ids, np.int32), np.array(segs, np.int32),
                   np.arange(0, 3 * branches + 1, 3, dtype=np.int32),
                   np.array(sum(lists, []), np.int32), np.arange(branches + 1, dtype=np.int32),
                   None, None, n_pages + branches, meta={"seed": 0})
    slots, pages = oracle.unique_slots(w)
    page_kib = g["page_kib"]
    assert pages * page_kib / 1024 == g["unique_payload_after_mib"]
    assert slots == pages * 16
    full_copies = (1 + branches) * n_pages * page_kib / 1024
    assert full_copies == g["unique_payload_before_mib"]
    assert round(100 * (1 - pages * page_kib / 1024 / full_copies), 2) == g["reduction_percent"]
