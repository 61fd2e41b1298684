"""Seeded synthetic inputs for fork decode attention over a branching, paged KV cache.

This module only builds inputs: the page table, the segment descriptors, the per-branch
visibility bits and random Q / K / V. It holds none of the attention arithmetic, so both the
CUDA path and the fp64 oracle can take their inputs from it.

Structure follows the pages:

* Octopus (zicq.com), "Zero-Copy Radix Forking": branches reference the same physical KV pages
  of a shared radix prefix; new tokens of a branch go to pages of its own.
* Octopus, "Attention-Only KV Mounting": a thread mounts the terminal KV block of a sibling;
  here that is a segment whose page list points into the sibling's pages (no new pages).
* AKV (news.farwalk.ai), "AKV 如何工作？": Drop hides entries from attention but keeps their
  positions; here that is a cleared bit in a branch's visibility bits.  "AKV 在智能体基准上
  表现如何？": the rolling policy keeps the latest 12 tool responses (config 4).

Draw order for every workload: structure -> masks (both on a CPU ``torch.Generator``) -> Q -> K
-> V (on a generator of the requested device, seeded with the same seed). All values are
fp32 ``randn`` cast to bf16 with round-to-nearest-even. Physical pages are handed out from a
random permutation of a pool with 5% spare pages.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional

import numpy as np
import torch

HEAD_DIM = 128
PAGE_SIZE = 16
SEED_BASE = 20260000


@dataclass
class Workload:
    """One fork-decode problem: descriptors (host numpy) plus Q/K/V tensors."""

    name: str
    num_q_heads: int
    num_kv_heads: int
    page_ids: np.ndarray  # int32 [num_page_ids] physical page per listed page
    segs: np.ndarray  # int32 [num_segs, 3] = (page_off, tok_begin, len)
    branch_seg_off: np.ndarray  # int32 [B+1]
    branch_segs: np.ndarray  # int32 [sum of list lengths]
    branch_q_off: np.ndarray  # int32 [B+1]
    vis_bits: Optional[np.ndarray]  # uint32 words, or None = all visible
    vis_word_off: Optional[np.ndarray]  # int64 [B+1], or None
    num_pages_pool: int
    q: Optional[torch.Tensor] = None  # bf16 [total_q, Hq, 128]
    k_pages: Optional[torch.Tensor] = None  # bf16 [pool, Hkv, 16, 128]
    v_pages: Optional[torch.Tensor] = None
    head_dim: int = HEAD_DIM
    page_size: int = PAGE_SIZE
    meta: dict = field(default_factory=dict)

    @property
    def num_branches(self) -> int:
        return len(self.branch_seg_off) - 1

    @property
    def total_q(self) -> int:
        return int(self.branch_q_off[-1])

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    def branch_len(self, b: int) -> int:
        ids = self.branch_segs[self.branch_seg_off[b]:self.branch_seg_off[b + 1]]
        return int(self.segs[ids, 2].sum())


class _Builder:
    """Collects segments and branch lists; pages are assigned once the pool size is known."""

    def __init__(self, seed: int):
        self.gen = torch.Generator().manual_seed(seed)
        self.seed = seed
        self.seg_pages: List[int] = []  # pages owned by each "owned" segment (or -1 for views)
        self.segs: List[list] = []  # [page_off or None, tok_begin, len, owner_seg]
        self.branches: List[List[int]] = []
        self.n_q: List[int] = []

    # -- structure -------------------------------------------------------------------
    def new_segment(self, length: int) -> int:
        """A segment stored in pages of its own, starting at slot 0."""
        assert length >= 1
        self.segs.append([None, 0, int(length), -1])
        return len(self.segs) - 1

    def tail_view(self, seg: int, m: int) -> int:
        """A segment that reads the last ``m`` tokens of ``seg`` in place (a mount)."""
        owner = seg if self.segs[seg][3] < 0 else self.segs[seg][3]
        assert self.segs[seg][3] < 0, "views of views are not needed here"
        length = self.segs[seg][2]
        m = min(m, length)
        t0 = length - m
        self.segs.append([("view", owner, t0), t0 % PAGE_SIZE, int(m), owner])
        return len(self.segs) - 1

    def add_branch(self, seg_list: List[int], n_q: int = 1) -> int:
        self.branches.append(list(seg_list))
        self.n_q.append(int(n_q))
        return len(self.branches) - 1

    # -- random helpers (CPU generator: structure and masks) -----------------------------
    def randint(self, lo: int, hi_incl: int) -> int:
        return int(torch.randint(lo, hi_incl + 1, (1,), generator=self.gen).item())

    def rand(self, n: int = 1) -> torch.Tensor:
        return torch.rand(n, generator=self.gen, dtype=torch.float64)

    def randn1(self) -> float:
        return float(torch.randn(1, generator=self.gen, dtype=torch.float64).item())

    # -- layout ----------------------------------------------------------------------------
    def layout(self, spare: float = 0.05):
        owned = [i for i, s in enumerate(self.segs) if s[3] < 0]
        need = sum((self.segs[i][2] + PAGE_SIZE - 1) // PAGE_SIZE for i in owned)
        pool = int(math.ceil(need * (1.0 + spare))) + 1
        perm = torch.randperm(pool, generator=self.gen).numpy().astype(np.int32)
        page_ids: List[np.ndarray] = []
        seg_rows = np.zeros((len(self.segs), 3), dtype=np.int32)
        off = 0
        nxt = 0
        for i in owned:
            n = (self.segs[i][2] + PAGE_SIZE - 1) // PAGE_SIZE
            page_ids.append(perm[nxt:nxt + n])
            seg_rows[i] = (off, 0, self.segs[i][2])
            off += n
            nxt += n
        for i, s in enumerate(self.segs):
            if s[3] >= 0:
                _, owner, t0 = s[0]
                seg_rows[i] = (seg_rows[owner, 0] + t0 // PAGE_SIZE, t0 % PAGE_SIZE, s[2])
        page_ids_arr = np.concatenate(page_ids) if page_ids else np.zeros(0, np.int32)
        bso = np.zeros(len(self.branches) + 1, dtype=np.int32)
        bso[1:] = np.cumsum([len(b) for b in self.branches])
        bsegs = np.array([s for b in self.branches for s in b], dtype=np.int32)
        bqo = np.zeros(len(self.branches) + 1, dtype=np.int32)
        bqo[1:] = np.cumsum(self.n_q)
        return page_ids_arr, seg_rows, bso, bsegs, bqo, pool


def logical_slots(w: Workload, b: int) -> np.ndarray:
    """Physical slot ids (page * 16 + slot) of branch ``b``'s logical sequence, in order.

    Pure index bookkeeping (used to place drops by physical token and by tests)."""
    out = []
    for s in w.branch_segs[w.branch_seg_off[b]:w.branch_seg_off[b + 1]]:
        po, tb, ln = (int(x) for x in w.segs[s])
        t = np.arange(ln, dtype=np.int64) + tb
        pages = w.page_ids[po + t // PAGE_SIZE].astype(np.int64)
        out.append(pages * PAGE_SIZE + t % PAGE_SIZE)
    return np.concatenate(out) if out else np.zeros(0, np.int64)


def pack_bits(vis: np.ndarray) -> np.ndarray:
    """Pack a bool vector into little-endian uint32 words (bit j of word j//32)."""
    n = len(vis)
    nw = (n + 31) // 32
    padded = np.zeros(nw * 32, dtype=np.uint8)
    padded[:n] = vis
    by = np.packbits(padded, bitorder="little")
    return by.view("<u4").astype(np.uint32) if nw else np.zeros(0, np.uint32)


def _pack_branch_bits(per_branch: List[np.ndarray]):
    words = [pack_bits(v) for v in per_branch]
    off = np.zeros(len(words) + 1, dtype=np.int64)
    off[1:] = np.cumsum([len(x) for x in words])
    return (np.concatenate(words) if words else np.zeros(0, np.uint32)).astype(np.uint32), off


def _finish(name, hq, hkv, bld: _Builder, drop_phys_p: float = 0.0, vis_fn=None,
            device: str = "cpu", values: bool = True, meta=None) -> Workload:
    page_ids, segs, bso, bsegs, bqo, pool = bld.layout()
    w = Workload(name, hq, hkv, page_ids, segs, bso, bsegs, bqo, None, None, pool,
                 meta=dict(meta or {}, seed=bld.seed))
    # masks: one Bernoulli per physical token (all readers of a shared run agree) and/or a
    # structural visibility function; the query tokens themselves are never dropped.
    if drop_phys_p > 0.0 or vis_fn is not None:
        dropped = None
        if drop_phys_p > 0.0:
            dropped = (torch.rand(pool * PAGE_SIZE, generator=bld.gen) < drop_phys_p).numpy()
        per_branch = []
        for b in range(w.num_branches):
            slots = logical_slots(w, b)
            vis = np.ones(len(slots), dtype=bool)
            if dropped is not None:
                vis &= ~dropped[slots]
            if vis_fn is not None:
                vis &= vis_fn(b, len(slots))
            nq = int(bqo[b + 1] - bqo[b])
            vis[len(slots) - nq:] = True
            per_branch.append(vis)
        w.vis_bits, w.vis_word_off = _pack_branch_bits(per_branch)
    if values:
        fill_values(w, device=device)
    return w


def fill_values(w: Workload, device: str = "cpu") -> None:
    """Draw Q, then K, then V: N(0, 1) fp32 cast to bf16 (RNE), on ``device``'s generator."""
    seed = int(w.meta["seed"])
    gen = torch.Generator(device=device).manual_seed(seed)
    hq, hkv, d, p = w.num_q_heads, w.num_kv_heads, w.head_dim, w.page_size

    def draw(shape):
        out = torch.empty(shape, dtype=torch.bfloat16, device=device)
        flat = out.view(-1)
        chunk = 1 << 24
        for i in range(0, flat.numel(), chunk):
            n = min(chunk, flat.numel() - i)
            flat[i:i + n] = torch.randn(n, generator=gen, device=device,
                                        dtype=torch.float32).to(torch.bfloat16)
        return out

    w.q = draw((w.total_q, hq, d))
    w.k_pages = draw((w.num_pages_pool, hkv, p, d))
    w.v_pages = draw((w.num_pages_pool, hkv, p, d))


# ----------------------------------------------------------------------------------------
# The five workloads. ``shrink`` divides token counts (and, where stated, request counts) so
# that the fp64 oracle can check every output in seconds; shrink=1 is the full size.
# ----------------------------------------------------------------------------------------

def config1(shrink: int = 1, device="cpu", values=True) -> Workload:
    """Tiny fork decode: Hq 8 / Hkv 2, prefix 1024 + 4 branches x 256 private, n_q 1."""
    bld = _Builder(SEED_BASE + 1)
    pre = bld.new_segment(max(1024 // shrink, 1))
    for _ in range(4):
        bld.add_branch([pre, bld.new_segment(max(256 // shrink, 1))], 1)
    return _finish("tiny_fork", 8, 2, bld, device=device, values=values)


def config2(shrink: int = 1, device="cpu", values=True) -> Workload:
    """Flat fork with drops: Hq 32 / Hkv 8, prefix 32K + 16 x 2K, Bernoulli(0.1) drops."""
    bld = _Builder(SEED_BASE + 2)
    pre = bld.new_segment(32768 // shrink)
    for _ in range(16):
        bld.add_branch([pre, bld.new_segment(2048 // shrink)], 1)
    return _finish("flat_fork_drops", 32, 8, bld, drop_phys_p=0.1, device=device, values=values)


def config3(shrink: int = 1, device="cpu", values=True) -> Workload:
    """KV DAG with mounting: Hq 16 / Hkv 4, root 64K, depth 3 fan-out 4, nodes U{1K..4K},
    each leaf mounts the last 512 tokens of 2 distinct random sibling leaves."""
    bld = _Builder(SEED_BASE + 3)
    root = bld.new_segment(65536 // shrink)
    lo, hi = 1024 // shrink, 4096 // shrink
    l1 = [bld.new_segment(bld.randint(lo, hi)) for _ in range(4)]
    l2 = [[bld.new_segment(bld.randint(lo, hi)) for _ in range(4)] for _ in range(4)]
    leaves = [[[bld.new_segment(bld.randint(lo, hi)) for _ in range(4)] for _ in range(4)]
              for _ in range(4)]
    mount = max(512 // shrink, 1)
    for a in range(4):
        for c in range(4):
            for e in range(4):
                sibs = [x for x in range(4) if x != e]
                pick = torch.randperm(3, generator=bld.gen)[:2].tolist()
                mounts = [bld.tail_view(leaves[a][c][sibs[k]], mount) for k in pick]
                bld.add_branch([root, l1[a], l2[a][c], leaves[a][c][e]] + mounts, 1)
    return _finish("kv_dag_mounts", 16, 4, bld, device=device, values=values)


def config4(shrink: int = 1, device="cpu", values=True) -> Workload:
    """Long-context rolling drop: Hq 64 / Hkv 8, prefix 128K of alternating 256-token reasoning
    and U{2K..8K} tool segments (reasoning first, last one truncated); the latest 12 tool
    segments and every reasoning segment stay visible; 64 branches with lognormal private
    lengths, median 2K, sigma = ln(4)/2, clipped to [512, 8K]."""
    bld = _Builder(SEED_BASE + 4)
    total = 131072 // shrink
    reason = max(256 // shrink, 1)
    tlo, thi = 2048 // shrink, 8192 // shrink
    pieces = []  # (start, len, is_tool)
    pos, tool = 0, False
    while pos < total:
        ln = bld.randint(tlo, thi) if tool else reason
        ln = min(ln, total - pos)
        pieces.append((pos, ln, tool))
        pos += ln
        tool = not tool
    tools = [p for p in pieces if p[2]]
    keep = np.ones(total, dtype=bool)
    for (s, ln, _) in tools[:-12] if len(tools) > 12 else []:
        keep[s:s + ln] = False
    pre = bld.new_segment(total)
    sigma = math.log(4.0) / 2.0
    plo, phi = max(512 // shrink, 1), 8192 // shrink
    for _ in range(64):
        ln = int(round(math.exp(math.log(2048.0 / shrink) + sigma * bld.randn1())))
        ln = min(max(ln, plo), phi)
        bld.add_branch([pre, bld.new_segment(ln)], 1)

    def vis_fn(b, n):
        v = np.ones(n, dtype=bool)
        v[:total] = keep
        return v

    meta = {"prefix_pieces": len(pieces), "tool_segments": len(tools)}
    return _finish("long_ctx_rolling_drop", 64, 8, bld, vis_fn=vis_fn, device=device,
                   values=values, meta=meta)


def config5(shrink: int = 1, requests: int = 32, device="cpu", values=True) -> Workload:
    """Batched multi-tree multi-token: 32 requests, prefix round(exp(U(ln 8K, ln 64K))),
    8 branches each with U{256..4K} private tokens, n_q 8 causal, Bernoulli(0.05) drops."""
    bld = _Builder(SEED_BASE + 5)
    for _ in range(requests):
        u = float(bld.rand(1).item())
        ln = int(round(math.exp(math.log(8192.0) + u * (math.log(65536.0) - math.log(8192.0)))))
        pre = bld.new_segment(max(ln // shrink, 8))
        for _ in range(8):
            priv = max(bld.randint(256, 4096) // shrink, 8)
            bld.add_branch([pre, bld.new_segment(priv)], 8)
    return _finish("multi_tree_multi_token", 32, 8, bld, drop_phys_p=0.05, device=device,
                   values=values)


def packed_dag_prefill(shrink: int = 1, threads: int = 8, device="cpu", values=True) -> Workload:
    """Packed DAG prefill of one episode: Hq 32 / Hkv 8, a root of 4K tokens, ``threads``
    threads of U{1K..3K} tokens each; thread j >= 1 mounts the last 512 tokens of one random
    earlier thread.  Every token is a query: the root's tokens see the root causally, a
    thread's tokens see the root, its mount, and its own tokens causally (no drops).

    Octopus (zicq.com), "Packed DAG-GRPO": all branches of an episode go through one
    block-sparse attention whose mask holds intra-thread causality and the allowed
    cross-thread reads; as a descriptor that is one branch per thread, listing the segments
    it may read, with its own tokens as its queries."""
    bld = _Builder(SEED_BASE + 6)
    root = bld.new_segment(max(4096 // shrink, 1))
    bld.add_branch([root], max(4096 // shrink, 1))
    own = []
    mount = max(512 // shrink, 1)
    for j in range(threads):
        ln = max(bld.randint(1024, 3072) // shrink, 1)
        seg = bld.new_segment(ln)
        lst = [root]
        if j >= 1:
            lst.append(bld.tail_view(own[bld.randint(0, j - 1)], mount))
        own.append(seg)
        bld.add_branch(lst + [seg], ln)
    return _finish("packed_dag_prefill", 32, 8, bld, device=device, values=values)


CONFIGS = {1: config1, 2: config2, 3: config3, 4: config4, 5: config5}
PREFILL_SMALL = dict(shrink=16)

# Shrink factors for the parity cases the oracle checks in full (seconds on a few cores).
SMALL = {1: dict(shrink=1), 2: dict(shrink=8), 3: dict(shrink=16), 4: dict(shrink=16),
         5: dict(shrink=8, requests=4)}


def with_representatives(w: Workload, branches: Optional[List[int]] = None, reps: int = 32,
                         device: str = "cpu") -> Workload:
    """The cache of ``w`` restricted to ``branches`` (all by default), each with ``reps``
    representative queries of its own: N(0, 1) fp32 cast to bf16, drawn after the workload's
    own values from seed + 7.

    AgentKV blog (rit.work), "Как AgentKV выбирает и освобождает записи кэша": the queries kept
    per phase are merged into one set of representatives (32 in the main experiments) that
    scores every key before a compression."""
    sub = subset(w, list(range(w.num_branches)) if branches is None else list(branches))
    B = sub.num_branches
    sub.branch_q_off = (np.arange(B + 1, dtype=np.int64) * reps).astype(np.int32)
    sub.name = w.name + f"_reps{reps}"
    sub.meta = dict(sub.meta, reps=reps)
    gen = torch.Generator(device=device).manual_seed(int(w.meta["seed"]) + 7)
    sub.q = torch.randn((B * reps, w.num_q_heads, w.head_dim), generator=gen, device=device,
                        dtype=torch.float32).to(torch.bfloat16)
    sub.k_pages, sub.v_pages = sub.k_pages.to(device), sub.v_pages.to(device)
    return sub


# Workload 6: the prefill-shaped one (every token a query), beside the five decodes.
PREFILL = 6


def make(config: int, small: bool = False, device: str = "cpu", values: bool = True) -> Workload:
    if config == PREFILL:
        kw = dict(PREFILL_SMALL) if small else {}
        return packed_dag_prefill(device=device, values=values, **kw)
    kw = dict(SMALL[config]) if small else {}
    return CONFIGS[config](device=device, values=values, **kw)


def subset(w: Workload, branches: List[int]) -> Workload:
    """A workload holding only ``branches`` of ``w``, with its pages compacted into a new pool.

    Index bookkeeping only: the values are gathered, not recomputed."""
    seg_ids = sorted({int(s) for b in branches
                      for s in w.branch_segs[w.branch_seg_off[b]:w.branch_seg_off[b + 1]]})
    seg_map = {s: i for i, s in enumerate(seg_ids)}
    used_pages = []
    new_segs = np.zeros((len(seg_ids), 3), dtype=np.int32)
    pid_list = []
    for i, s in enumerate(seg_ids):
        po, tb, ln = (int(x) for x in w.segs[s])
        n = (tb + ln + PAGE_SIZE - 1) // PAGE_SIZE
        new_segs[i] = (len(pid_list), tb, ln)
        pid_list.extend(int(p) for p in w.page_ids[po:po + n])
    uniq = sorted(set(pid_list))
    pmap = {p: i for i, p in enumerate(uniq)}
    page_ids = np.array([pmap[p] for p in pid_list], dtype=np.int32)
    bso = [0]
    bsegs = []
    bqo = [0]
    words = []
    for b in branches:
        lst = w.branch_segs[w.branch_seg_off[b]:w.branch_seg_off[b + 1]]
        bsegs.extend(seg_map[int(s)] for s in lst)
        bso.append(len(bsegs))
        bqo.append(bqo[-1] + int(w.branch_q_off[b + 1] - w.branch_q_off[b]))
        if w.vis_bits is not None:
            words.append(w.vis_bits[w.vis_word_off[b]:w.vis_word_off[b + 1]])
    if w.vis_bits is not None:
        vis_bits = np.concatenate(words).astype(np.uint32)
        vwo = np.zeros(len(branches) + 1, dtype=np.int64)
        vwo[1:] = np.cumsum([len(x) for x in words])
    else:
        vis_bits, vwo = None, None
    sub = Workload(w.name + "_subset", w.num_q_heads, w.num_kv_heads, page_ids, new_segs,
                   np.array(bso, np.int32), np.array(bsegs, np.int32), np.array(bqo, np.int32),
                   vis_bits, vwo, len(uniq), meta=dict(w.meta))
    if w.k_pages is not None:
        idx = torch.tensor(uniq, dtype=torch.long, device=w.k_pages.device)
        sub.k_pages = w.k_pages.index_select(0, idx)
        sub.v_pages = w.v_pages.index_select(0, idx)
        qrows = torch.cat([torch.arange(int(w.branch_q_off[b]), int(w.branch_q_off[b + 1]))
                           for b in branches]).to(w.q.device)
        sub.q = w.q.index_select(0, qrows)
    return sub


def to_device(w: Workload, device) -> Workload:
    w.q = w.q.to(device)
    w.k_pages = w.k_pages.to(device)
    w.v_pages = w.v_pages.to(device)
    return w


def random_dag(seed: int, num_q_heads: int = 4, num_kv_heads: int = 2, n_segs: int = 4,
               n_branches: int = 3, max_list: int = 4, max_seg_len: int = 40,
               pool_pages: int = 6, drop_p: float = 0.2, max_nq: int = 3,
               mid_page: bool = True, allow_dup: bool = True, device: str = "cpu",
               values: bool = True) -> Workload:
    """A small random branching cache for edge cases: segments may start mid-page, share or
    overlap physical pages, be listed by several branches or twice by one; visibility bits
    are random (a query row may see nothing at all)."""
    gen = torch.Generator().manual_seed(seed)

    def ri(lo, hi):  # inclusive
        return int(torch.randint(lo, hi + 1, (1,), generator=gen).item())

    page_ids: List[int] = []
    segs = []
    for _ in range(n_segs):
        ln = ri(1, max_seg_len)
        tb = ri(0, PAGE_SIZE - 1) if mid_page else 0
        n_pages = (tb + ln + PAGE_SIZE - 1) // PAGE_SIZE
        segs.append((len(page_ids), tb, ln))
        page_ids.extend(torch.randint(0, pool_pages, (n_pages,), generator=gen).tolist())
    lists = []
    for _ in range(n_branches):
        k = ri(1, max_list)
        if allow_dup:
            lst = torch.randint(0, n_segs, (k,), generator=gen).tolist()
        else:
            lst = torch.randperm(n_segs, generator=gen)[:min(k, n_segs)].tolist()
        lists.append(lst)
    seg_arr = np.array(segs, dtype=np.int32).reshape(-1, 3)
    bso = np.zeros(n_branches + 1, np.int32)
    bso[1:] = np.cumsum([len(x) for x in lists])
    bsegs = np.array([s for x in lists for s in x], np.int32)
    nqs = []
    for lst in lists:
        n_b = int(seg_arr[lst, 2].sum())
        nqs.append(ri(1, min(max_nq, n_b)))
    bqo = np.zeros(n_branches + 1, np.int32)
    bqo[1:] = np.cumsum(nqs)
    w = Workload("random_dag", num_q_heads, num_kv_heads, np.array(page_ids, np.int32),
                 seg_arr, bso, bsegs, bqo, None, None, pool_pages, meta={"seed": seed})
    if drop_p > 0:
        per_branch = []
        for b in range(n_branches):
            n_b = w.branch_len(b)
            per_branch.append((torch.rand(n_b, generator=gen) >= drop_p).numpy())
        w.vis_bits, w.vis_word_off = _pack_branch_bits(per_branch)
    if values:
        fill_values(w, device=device)
    return w
