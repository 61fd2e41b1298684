"""fp64 CPU oracle for physical compaction with optional repositioning (test infrastructure
only: ``tests/`` and the benchmark's CPU legs use it, the library never does).

AgentKV blog (rit.work), "Как AgentKV выбирает и освобождает записи кэша": the kept cache
entries are physically packed into fresh pages and the freed pages go back to the allocator,
so that a smaller cache is also fewer bytes read.  AKV (news.farwalk.ai), "AKV 如何工作？":
Drop hides entries from later attention and keeps positions; Repos rewrites the kept keys
to positions 0..r-1 by a RoPE rotation and leaves the values unchanged.

Definition computed here, for branch b of a paged cache with visibility bits (the same
descriptors as the decode):
  kept_b = [j in 0 .. n_b - 1 with vis_b[j] = 1], in logical order; r_b = |kept_b|
  the n-th kept entry j_n, stored at physical slot s(j_n), becomes entry n of the packed
  copy (n // page_size-th destination page, slot n % page_size):
     V'[n, g] = V[s(j_n), g]
     K'[n, g] = K[s(j_n), g]                    without repositioning
     K'[n, g] = rot(K[s(j_n), g], n - j_n)      with repositioning (position j_n -> n)
  rot(x, d), rotate-half pairing, theta_i = base ** (-2 i / D) for i in 0 .. D/2 - 1:
     x_i       -> x_i cos(d theta_i) - x_{i+D/2} sin(d theta_i)
     x_{i+D/2} -> x_{i+D/2} cos(d theta_i) + x_i sin(d theta_i)
Positions are logical indices in the branch's sequence (the decode's reading too).  Values
are the exact bf16 inputs in fp64; the result is fp64 (the device rounds K' to bf16).
"""
import numpy as np


def branch_slots(w, b):
    """Physical slot (page id * page_size + offset) of every logical index of branch b,
    walked from the segment list (own walk: shares nothing with the library's planner)."""
    P = 16
    out = []
    for sid in w.branch_segs[w.branch_seg_off[b]:w.branch_seg_off[b + 1]]:
        page_off, tok_begin, length = (int(x) for x in w.segs[int(sid)])
        for t in range(length):
            pos = tok_begin + t
            out.append(int(w.page_ids[page_off + pos // P]) * P + pos % P)
    return np.asarray(out, dtype=np.int64)


def kept_indices(w, b):
    """Logical indices of branch b whose visibility bit is set (all of them without bits)."""
    n = int(sum(int(w.segs[int(s)][2]) for s in w.branch_segs[w.branch_seg_off[b]:w.branch_seg_off[b + 1]]))
    if w.vis_bits is None:
        return np.arange(n, dtype=np.int64)
    words = np.asarray(w.vis_bits[w.vis_word_off[b]:w.vis_word_off[b + 1]], dtype=np.uint64)
    j = np.arange(n, dtype=np.int64)
    bits = (words[j // 32] >> (j % 32).astype(np.uint64)) & np.uint64(1)
    return j[bits.astype(bool)]


def rope_rotate(x, d, base=10000.0):
    """rot(x, d) over the last axis (length D) in fp64; d broadcasts against x[..., 0]."""
    x = np.asarray(x, dtype=np.float64)
    D = x.shape[-1]
    h = D // 2
    theta = base ** (-2.0 * np.arange(h, dtype=np.float64) / D)
    ang = np.asarray(d, dtype=np.float64)[..., None] * theta
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., :h], x[..., h:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def compact(w, b, reposition=False, base=10000.0):
    """(K', V', kept): K', V' fp64 [r_b, Hkv, D] of branch b; kept the logical indices."""
    slots = branch_slots(w, b)
    kept = kept_indices(w, b)
    src = slots[kept]
    P = 16
    import torch
    pg, off = torch.as_tensor(src // P), torch.as_tensor(src % P)
    K = w.k_pages[pg, :, off, :].double().numpy()      # [r, Hkv, D], exact bf16 values
    V = w.v_pages[pg, :, off, :].double().numpy()
    if reposition:
        delta = np.arange(len(kept), dtype=np.int64) - kept
        K = rope_rotate(K, delta[:, None], base)
    return K, V, kept


def common_prefix(w, branches):
    """(P, r_s): the listed branches' common prefix -- the first P logical indices at which
    all of them have the same physical slot and the same visibility bit -- and the number of
    kept entries in it.  A plain walk, one index at a time."""
    if len(branches) == 0:
        return 0, 0
    slots = [branch_slots(w, b) for b in branches]
    vis = []
    for b, s in zip(branches, slots):
        v = np.zeros(len(s), dtype=bool)
        v[kept_indices(w, b)] = True
        vis.append(v)
    P = 0
    while all(P < len(s) for s in slots) and \
            all(slots[k][P] == slots[0][P] and vis[k][P] == vis[0][P] for k in range(len(slots))):
        P += 1
    return P, int(vis[0][:P].sum())
