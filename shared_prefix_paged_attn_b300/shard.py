"""Splitting one fork-decode problem over several GPUs (host-side index bookkeeping only).

Every output row of the decode depends on one query head of one query token and the K/V of
its KV head over its branch's visible entries, so the problem splits without any exchange on
the data path two ways, and a third way with one all-gather:

* by KV head: rank r takes KV heads [r Hkv / N, (r + 1) Hkv / N) and the query heads of their
  groups; every rank reads every page, but only its heads' slices of it.
* by request: branches that share a physical page (a prefix, a mount) stay on one rank;
  these groups are dealt to the ranks by listed tokens, largest first, each to the rank with
  the fewest so far.  Shared pages are then read by one rank only.
* by sequence: rank r takes the logical positions [r L / N, (r + 1) L / N) of every branch
  (L the longest branch), i.e. the same problem with every other entry's visibility bit
  cleared; positions, and so causal limits, are unchanged, and a shared prefix (the same
  positions in every branch) falls to one rank per range.  Each rank's result is a partial
  (out, lse) of every query row; the ranks all-gather them and merge them with the
  log-sum-exp merge (``fork_attn_merge_parts``): the one split with an exchange.

The outputs concatenate back: by head along the head axis, by request along the query-token
axis in the ranks' branch order (``gather_rows`` puts them back in the problem's order).
"""
from __future__ import annotations

from typing import List, Tuple

import numpy as np
import torch

from . import workloads as W


def head_range(num_kv_heads: int, rank: int, world: int) -> Tuple[int, int]:
    """KV heads [lo, hi) of `rank` (contiguous, sizes differing by at most one)."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("rank out of range")
    if num_kv_heads < world:
        raise ValueError("fewer KV heads than ranks")
    base, extra = divmod(num_kv_heads, world)
    lo = rank * base + min(rank, extra)
    return lo, lo + base + (1 if rank < extra else 0)


def split_by_kv_head(w: W.Workload, rank: int, world: int) -> W.Workload:
    """Rank `rank`'s share of `w`: the same descriptors, its KV heads and their query heads."""
    lo, hi = head_range(w.num_kv_heads, rank, world)
    G = w.num_q_heads // w.num_kv_heads
    sub = W.Workload(f"{w.name}_kvheads{lo}-{hi}", G * (hi - lo), hi - lo, w.page_ids, w.segs,
                     w.branch_seg_off, w.branch_segs, w.branch_q_off, w.vis_bits,
                     w.vis_word_off, w.num_pages_pool, meta=dict(w.meta, kv_heads=(lo, hi)))
    if w.q is not None:
        sub.q = w.q[:, G * lo:G * hi].contiguous()
        sub.k_pages = w.k_pages[:, lo:hi].contiguous()
        sub.v_pages = w.v_pages[:, lo:hi].contiguous()
    return sub


def request_groups(w: W.Workload) -> List[List[int]]:
    """Branches grouped by shared physical pages (connected components), each group in
    branch order, groups ordered by their first branch."""
    B = w.num_branches
    parent = list(range(B))

    def find(x):
        while parent[x] != x:
            parent[x] = parent[parent[x]]
            x = parent[x]
        return x

    owner = {}
    for b in range(B):
        for s in w.branch_segs[w.branch_seg_off[b]:w.branch_seg_off[b + 1]]:
            po, tb, ln = (int(x) for x in w.segs[s])
            for p in w.page_ids[po:po + (tb + ln + W.PAGE_SIZE - 1) // W.PAGE_SIZE]:
                p = int(p)
                if p in owner:
                    ra, rb = find(owner[p]), find(b)
                    if ra != rb:
                        parent[max(ra, rb)] = min(ra, rb)
                else:
                    owner[p] = b
    groups = {}
    for b in range(B):
        groups.setdefault(find(b), []).append(b)
    return [groups[k] for k in sorted(groups)]


def request_assignment(w: W.Workload, world: int) -> List[List[int]]:
    """Branches of each rank (ascending): request groups dealt largest first (listed tokens)
    to the rank with the fewest listed tokens so far (ties to the lower rank)."""
    if world < 1:
        raise ValueError("world must be >= 1")
    groups = request_groups(w)
    if len(groups) < world:
        raise ValueError("fewer independent requests than ranks")
    size = [sum(w.branch_len(b) for b in g) for g in groups]
    load = [0] * world
    ranks: List[List[int]] = [[] for _ in range(world)]
    for gi in sorted(range(len(groups)), key=lambda i: (-size[i], i)):
        r = min(range(world), key=lambda x: (load[x], x))
        load[r] += size[gi]
        ranks[r].extend(groups[gi])
    return [sorted(x) for x in ranks]


def split_by_request(w: W.Workload, rank: int, world: int) -> Tuple[W.Workload, List[int]]:
    """Rank `rank`'s share of `w` (its branches, pages compacted into a pool of their own)
    and the branches it holds, in the order of its output rows."""
    mine = request_assignment(w, world)[rank]
    sub = W.subset(w, mine)
    sub.name = f"{w.name}_requests_r{rank}of{world}"
    return sub, mine


def gather_heads(parts: List[torch.Tensor], w: W.Workload) -> torch.Tensor:
    """Per-rank outputs [total_q, Hq_r, ...] of a split by KV head back into [total_q, Hq, ...]."""
    out = torch.cat(parts, dim=1)
    if out.shape[1] != w.num_q_heads:
        raise ValueError("the parts do not cover every query head")
    return out


def gather_rows(parts: List[torch.Tensor], branches: List[List[int]], w: W.Workload) -> torch.Tensor:
    """Per-rank outputs [total_q_r, ...] of a split by request back into the problem's
    query-token order."""
    shape = (w.total_q,) + tuple(parts[0].shape[1:])
    out = torch.empty(shape, dtype=parts[0].dtype, device=parts[0].device)
    seen = np.zeros(w.total_q, dtype=bool)
    for part, bl in zip(parts, branches):
        at = 0
        for b in bl:
            q0, q1 = int(w.branch_q_off[b]), int(w.branch_q_off[b + 1])
            out[q0:q1] = part[at:at + q1 - q0]
            seen[q0:q1] = True
            at += q1 - q0
        if at != part.shape[0]:
            raise ValueError("a part has more rows than its branches")
    if not seen.all():
        raise ValueError("the parts do not cover every query token")
    return out


def sequence_cuts(w: W.Workload, world: int) -> List[int]:
    """Logical-position cuts [c_0 = 0, ..., c_N = L] of the split by sequence."""
    if world < 1:
        raise ValueError("world must be >= 1")
    L = max(w.branch_len(b) for b in range(w.num_branches))
    return [r * L // world for r in range(world + 1)]


def split_by_sequence(w: W.Workload, rank: int, world: int) -> W.Workload:
    """Rank `rank`'s share of `w` by sequence: the same descriptors and values with the
    visibility bits of every entry outside [c_r, c_{r+1}) cleared."""
    if not 0 <= rank < world:
        raise ValueError("rank out of range")
    lo, hi = sequence_cuts(w, world)[rank:rank + 2]
    per_branch = []
    for b in range(w.num_branches):
        n = w.branch_len(b)
        j = np.arange(n)
        if w.vis_bits is None:
            vis = np.ones(n, dtype=bool)
        else:
            words = w.vis_bits[w.vis_word_off[b]:w.vis_word_off[b + 1]].astype(np.uint64)
            vis = ((words[j // 32] >> (j % 32).astype(np.uint64)) & 1).astype(bool)
        per_branch.append(vis & (j >= lo) & (j < hi))
    bits, off = W._pack_branch_bits(per_branch)
    sub = W.Workload(f"{w.name}_seq{rank}of{world}", w.num_q_heads, w.num_kv_heads, w.page_ids, w.segs,
                     w.branch_seg_off, w.branch_segs, w.branch_q_off, bits, off, w.num_pages_pool,
                     meta=dict(w.meta, positions=(lo, hi)))
    sub.q, sub.k_pages, sub.v_pages = w.q, w.k_pages, w.v_pages
    return sub
