"""GPU parity of key scoring by representative queries and of the top-k keep (C ABI) against
the fp64 oracle (oracle/score.py).

AgentKV blog (rit.work), "Как AgentKV выбирает и освобождает записи кэша": every key is scored
by the mean attention of the representative queries; the highest-scoring entries are kept.

Tolerance of a score (derived from the arithmetic): bf16 inputs are exact on both sides; the
device's QK^T accumulates in fp32 (relative ~1e-6 of the dot product's magnitude, i.e. an
absolute error of s around 1e-5 for |s| ~ 10), its lse is within ~1e-6 of the fp64 one, and
exp2 is the hardware approximation (~2e-7 relative); each term exp(s - lse) then carries a
relative error of about 1e-5 at most, and so does their mean (about 4e-7 is seen).  Tested:
|got - ref| <= 2e-5 * ref + 1e-9.  The kept set is compared exactly with a selection
made on the device's own scores (ties to the smaller index), and with the oracle's set where
the oracle's k-th and (k+1)-th scores are further apart than the tolerance; where they are not,
every entry clearly above (below) the threshold must be kept (dropped).
"""
import numpy as np
import pytest
import torch

from oracle import compact as C
from oracle import score as S
import shared_prefix_paged_attn_b300 as fa
from shared_prefix_paged_attn_b300 import workloads as W

pytestmark = pytest.mark.gpu

REL, ABS = 2e-5, 1e-9


def run_scores(w, keep_k=None):
    dev = torch.device("cuda")
    sc = fa.KeyScorer(w)
    scores = sc.score(w.q.to(dev), w.k_pages.to(dev), w.v_pages.to(dev))
    bits = None
    if keep_k is not None:
        bits = sc.topk(torch.as_tensor(np.asarray(keep_k, np.int32), device=dev))
    torch.cuda.synchronize()
    assert fa.fork_attn_check(sc.plan) == 0
    E, nw = fa.fork_attn_score_sizes(sc.plan)
    out = scores[:E].cpu().numpy()
    return out, (bits[:nw].cpu().numpy().view(np.uint32) if bits is not None else None)


def branch_views(w, scores, bits=None):
    """Per branch: (its scores over logical indices, its keep bits as bools)."""
    off = np.concatenate([[0], np.cumsum([w.branch_len(b) for b in range(w.num_branches)])])
    woff = np.concatenate([[0], np.cumsum([(w.branch_len(b) + 31) // 32 for b in range(w.num_branches)])])
    res = []
    for b in range(w.num_branches):
        n = w.branch_len(b)
        kb = None
        if bits is not None:
            words = bits[woff[b]:woff[b + 1]].astype(np.uint64)
            j = np.arange(n)
            kb = ((words[j // 32] >> (j % 32).astype(np.uint64)) & 1).astype(bool)
        res.append((scores[off[b]:off[b + 1]], kb))
    return res


def q_rep(w, b):
    return w.q[int(w.branch_q_off[b]):int(w.branch_q_off[b + 1])].double().numpy()


def check_scores(w, scores, branches=None):
    for b, (got, _) in enumerate(branch_views(w, scores)):
        if branches is not None and b not in branches:
            continue
        kept, ref = S.scores(w, b, q_rep(w, b))
        vis = np.zeros(len(got), bool)
        vis[kept] = True
        assert np.all(np.isnan(got[~vis])), f"branch {b}: an unseen entry has a score"
        g = got[kept].astype(np.float64)
        assert np.all(np.isfinite(g))
        err = np.abs(g - ref)
        assert np.all(err <= REL * ref + ABS), f"branch {b}: worst rel {np.max(err / np.maximum(ref, 1e-30))}"
        assert abs(g.sum() - 1.0) < 1e-3  # every representative's distribution sums to one


def expected_keep(got, k):
    """The kept set a selection on these exact scores must give (ties to the smaller index)."""
    vis = np.flatnonzero(~np.isnan(got))
    if k <= 0:
        return np.zeros(len(got), bool)
    order = sorted(vis.tolist(), key=lambda j: (-float(got[j]), j))
    keep = np.zeros(len(got), bool)
    keep[order[:k]] = True
    return keep


@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5])
def test_scores_small_workloads(cfg):
    w = W.make(cfg, small=True)
    branches = list(range(min(w.num_branches, 6)))
    reps = 32 if w.num_q_heads // w.num_kv_heads <= 8 else 16
    ws = W.with_representatives(w, branches, reps=reps)
    scores, _ = run_scores(ws)
    check_scores(ws, scores)


@pytest.mark.parametrize("seed", range(6))
def test_scores_random_caches(seed):
    # mid-page starts, duplicated segments, drops (a branch may see few entries), fewer
    # representatives than entries or more
    w = W.random_dag(800 + seed, num_q_heads=8, num_kv_heads=2, n_segs=5, n_branches=5,
                     max_seg_len=300, pool_pages=50, drop_p=(0.0, 0.3, 0.9)[seed % 3])
    ws = W.with_representatives(w, reps=(32, 7, 1)[seed % 3])
    scores, _ = run_scores(ws)
    check_scores(ws, scores)


@pytest.mark.parametrize("cfg", [2, 4])
def test_topk_matches_a_selection_on_the_scores_and_the_oracle(cfg):
    w = W.make(cfg, small=True)
    ws = W.with_representatives(w, list(range(4)), reps=16)
    n_vis = [len(C.kept_indices(ws, b)) for b in range(ws.num_branches)]
    ks = [n_vis[0] // 2, 0, n_vis[2] + 5, max(1, n_vis[3] // 5)]
    scores, bits = run_scores(ws, ks)
    for b, (got, kb) in enumerate(branch_views(ws, scores, bits)):
        want = expected_keep(got, ks[b])
        assert np.array_equal(kb, want), f"branch {b}: kept set differs from the selection on its scores"
        assert kb.sum() == min(max(ks[b], 0), n_vis[b])
        # against the oracle's fp64 scores
        kept, ref = S.scores(ws, b, q_rep(ws, b))
        k = min(max(ks[b], 0), len(kept))
        if k == 0 or k == len(kept):
            assert kb.sum() == k and kb[kept].all() == (k == len(kept))
            continue
        srt = np.sort(ref)[::-1]
        T, tol = srt[k - 1], REL * srt[k - 1] + ABS
        clear_in = kept[ref > T + 2 * tol]
        clear_out = kept[ref < T - 2 * tol]
        assert kb[clear_in].all() and not kb[clear_out].any()
        if srt[k - 1] - srt[k] > 2 * tol:
            assert np.array_equal(np.flatnonzero(kb), np.sort(S.keep(ws, b, q_rep(ws, b), k)))


def test_topk_equal_scores_keep_the_smaller_index():
    # a cache whose keys are all equal: every visible entry of a branch has the same score,
    # so the first k visible entries (logical order) are kept
    w = W.random_dag(31, num_q_heads=4, num_kv_heads=2, n_segs=3, n_branches=3, max_seg_len=100,
                     pool_pages=20, drop_p=0.3)
    w.k_pages = torch.ones_like(w.k_pages)
    ws = W.with_representatives(w, reps=8)
    n_vis = [len(C.kept_indices(ws, b)) for b in range(ws.num_branches)]
    ks = [max(1, n // 3) for n in n_vis]
    scores, bits = run_scores(ws, ks)
    for b, (got, kb) in enumerate(branch_views(ws, scores, bits)):
        kept = C.kept_indices(ws, b)
        assert len(set(got[kept].tolist())) == 1
        assert np.array_equal(np.flatnonzero(kb), kept[:ks[b]])


def test_full_size_long_context_scoring():
    # the benchmark's workload (8 branches of the 128K-token rolling-drop cache, 32
    # representatives each): every branch's scores sum to one; branch 0 against the oracle
    w = W.make(4, device="cuda")
    ws = W.with_representatives(w, list(range(8)), reps=32, device="cuda")
    ks = [int(0.25 * len(C.kept_indices(ws, b))) for b in range(8)]
    scores, bits = run_scores(ws, ks)
    views = branch_views(ws, scores, bits)
    for b, (got, kb) in enumerate(views):
        vis = ~np.isnan(got)
        assert abs(got[vis].astype(np.float64).sum() - 1.0) < 1e-3
        assert np.array_equal(kb, expected_keep(got, ks[b]))
    ws.q, ws.k_pages, ws.v_pages = ws.q.cpu(), ws.k_pages.cpu(), ws.v_pages.cpu()
    check_scores(ws, scores, branches=[0])


@pytest.mark.parametrize("cfg", [2, 4, 5])
def test_lse_pass_equals_the_decode_lse_bitwise(cfg):
    # the lse-only pass runs the decode's kernels without V, P V or output rows: every
    # representative row's lse carries the same bits as the full decode's
    dev = torch.device("cuda")
    ws = W.with_representatives(W.make(cfg, small=True), [0, 1, 2], reps=16)
    sc = fa.KeyScorer(ws)
    q, k, v = ws.q.to(dev), ws.k_pages.to(dev), ws.v_pages.to(dev)
    fa.fork_attn_decode(q, k, v, sc.plan, sc.out, sc.lse)
    ref = sc.lse.clone()
    sc.lse.fill_(float("nan"))
    fa.fork_attn_score_lse(q, k, sc.plan, sc.lse)
    torch.cuda.synchronize()
    assert fa.fork_attn_check(sc.plan) == 0
    assert torch.equal(sc.lse, ref)
