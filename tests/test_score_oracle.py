"""Pins of the phase-aware scoring oracle (CPU): a library softmax special case, closed forms,
invariants and brute-force top-k; planted mistakes fail them."""
import numpy as np
import pytest
import torch

from oracle import compact as C
from oracle import score as S
from shared_prefix_paged_attn_b300 import workloads as W


def _case(seed, drop_p=0.3, R=32):
    w = W.random_dag(seed, num_q_heads=8, num_kv_heads=2, n_branches=3, max_seg_len=120,
                     pool_pages=30, drop_p=drop_p)
    q = np.random.default_rng(seed).standard_normal((R, w.num_q_heads, 128))
    return w, q


@pytest.mark.parametrize("seed", range(4))
def test_scores_are_a_mean_of_library_softmaxes(seed):
    w, q = _case(600 + seed)
    for b in range(w.num_branches):
        kept, sc = S.scores(w, b, q)
        if len(kept) == 0:
            continue
        K = torch.from_numpy(C.compact(w, b)[0])             # [r, Hkv, D]
        qt = torch.from_numpy(q)                             # [R, Hq, D]
        G = w.num_q_heads // w.num_kv_heads
        Kh = K[:, torch.arange(w.num_q_heads) // G, :]       # [r, Hq, D]
        logits = torch.einsum("rhd,jhd->rhj", qt, Kh) / np.sqrt(128)
        want = torch.softmax(logits, dim=-1).mean(dim=(0, 1)).numpy()
        assert np.allclose(sc, want, atol=1e-12)
        assert np.isclose(sc.sum(), 1.0)


def test_identical_keys_score_uniformly_and_ties_keep_the_earliest():
    w, q = _case(700, drop_p=0.2)
    w.k_pages = torch.ones_like(w.k_pages)
    kept, sc = S.scores(w, 0, q)
    assert np.allclose(sc, 1.0 / len(kept))
    assert np.array_equal(S.keep(w, 0, q, 5), kept[:5])


def test_a_key_aligned_with_every_query_wins():
    for seed in range(701, 801):  # a branch that lists no physical slot twice
        w = W.random_dag(seed, num_q_heads=8, num_kv_heads=2, n_branches=1, max_seg_len=120,
                         pool_pages=4000, drop_p=0.0, allow_dup=False)
        slots = C.branch_slots(w, 0)
        if len(set(slots.tolist())) == len(slots):
            break
    q = np.random.default_rng(seed).standard_normal((32, w.num_q_heads, 128))
    q[:] = np.abs(q[0, 0])        # every representative and head points the same way
    kept = C.kept_indices(w, 0)
    j = int(kept[len(kept) // 2])
    kp = w.k_pages.clone()
    kp[slots[j] // 16, :, slots[j] % 16, :] = torch.from_numpy(4.0 * np.abs(q[0, 0])).to(torch.bfloat16)
    w.k_pages = kp
    assert np.array_equal(S.keep(w, 0, q, 1), [j])


def test_dropped_entries_never_count():
    w, q = _case(702, drop_p=0.5)
    kept, sc = S.scores(w, 1, q)
    slots = C.branch_slots(w, 1)
    hidden = np.setdiff1d(np.arange(len(slots)), kept)
    kp = w.k_pages.clone()
    for j in hidden:  # garbage in dropped slots that no visible entry shares
        if slots[j] not in set(slots[kept].tolist()):
            kp[slots[j] // 16, :, slots[j] % 16, :] = 30.0
    w.k_pages = kp
    kept2, sc2 = S.scores(w, 1, q)
    assert np.array_equal(kept, kept2) and np.allclose(sc, sc2, atol=1e-15)


@pytest.mark.parametrize("k", [1, 3, 10, 10_000])
def test_keep_is_the_brute_force_top_k(k):
    w, q = _case(703)
    kept, sc = S.scores(w, 2, q)
    got = set(S.keep(w, 2, q, k).tolist())
    assert len(got) == min(k, len(kept))
    for t, j in enumerate(kept):
        better = sum(1 for u, i in enumerate(kept) if sc[u] > sc[t] or (sc[u] == sc[t] and i < j))
        assert (j in got) == (better < k)


def test_planted_mistakes_fail_the_pins(monkeypatch):
    w, q = _case(704)
    good_kept, good = S.scores(w, 0, q)
    # mistake 1: GQA head mapping h % Hkv instead of h // G
    real = C.compact

    def swapped(w_, b_, reposition=False, base=10000.0):
        K, V, kept = real(w_, b_, reposition, base)
        return K[:, ::-1, :], V, kept
    monkeypatch.setattr(C, "compact", swapped)
    assert not np.allclose(S.scores(w, 0, q)[1], good, atol=1e-6)
    monkeypatch.setattr(C, "compact", real)
    # mistake 2: dropped entries scored too
    n_listed = len(C.branch_slots(w, 0))
    assert len(good_kept) < n_listed
    monkeypatch.setattr(C, "kept_indices", lambda w_, b_: np.arange(len(C.branch_slots(w_, b_))))
    bad_kept, bad = S.scores(w, 0, q)
    assert len(bad_kept) == n_listed and not np.isclose(bad[np.isin(bad_kept, good_kept)].sum(), 1.0)
