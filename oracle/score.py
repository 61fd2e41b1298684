"""fp64 CPU oracle for phase-aware key scoring and top-k keep (test infrastructure only).

AgentKV blog (rit.work), "Как AgentKV выбирает и освобождает записи кэша": recent attention
queries are queued per phase (reasoning, action, tool response, other); before a compression
the queues are merged into one set of representatives (32 queries in the main experiments),
every key is scored by its mean attention from them, and the entries with the largest mean
attention are kept.  The cache is not split per phase.

Definition computed here, for branch b with visible logical entries V_b (its visibility
bits) and representative queries q_r, r < R, each with Hq heads:
  p_{r,h}(j) = exp(s_{r,h,j}) / sum_{j' in V_b} exp(s_{r,h,j'}),  s_{r,h,j} = scale <q_{r,h}, K[slot(j), h // G]>
  score(j)   = mean over r < R and h < Hq of p_{r,h}(j)                 for j in V_b
  keep(k)    = the k entries of V_b with the largest score; equal scores keep the smaller
               logical index (all of V_b when k >= |V_b|)
Readings (the page leaves them open): the mean runs over every query head too, because a
page holds all heads of a token and a token is kept or evicted whole; the softmax runs over
the branch's visible entries only, without a causal limit (the representatives are earlier
queries scoring the whole cache).
"""
import numpy as np

from . import compact as _compact


def scores(w, b, q_rep, scale=None):
    """score(j) for the visible entries of branch b, in logical order: (kept_j, score)."""
    kept = _compact.kept_indices(w, b)
    if len(kept) == 0:
        return kept, np.zeros(0)
    K, _, _ = _compact.compact(w, b)                      # [r, Hkv, D] fp64, visible only
    q = np.asarray(q_rep, dtype=np.float64)              # [R, Hq, D]
    R, Hq, D = q.shape
    G = Hq // K.shape[1]
    sc = (1.0 / np.sqrt(D)) if scale is None else scale
    total = np.zeros(len(kept))
    for h in range(Hq):
        s = sc * (q[:, h, :] @ K[:, h // G, :].T)         # [R, r]
        s -= s.max(axis=1, keepdims=True)
        p = np.exp(s)
        p /= p.sum(axis=1, keepdims=True)
        total += p.sum(axis=0)
    return kept, total / (R * Hq)


def keep(w, b, q_rep, k, scale=None):
    """Logical indices of the k kept entries of branch b, ascending."""
    kept, sc = scores(w, b, q_rep, scale)
    if k >= len(kept):
        return kept
    order = sorted(range(len(kept)), key=lambda t: (-sc[t], kept[t]))
    return np.sort(kept[order[:k]])
