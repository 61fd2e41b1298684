"""Pins of the compaction / repositioning oracle (CPU), each against something other than
the oracle itself: a complex-number formulation of RoPE, keys built at their positions by
that formulation, brute-force slot membership, and closed forms."""
import numpy as np
import pytest
import torch

from oracle import compact as C
from shared_prefix_paged_attn_b300 import workloads as W


def rope_complex(x, pos, base=10000.0):
    # RoPE as complex multiplication: z_i = x_i + i x_{i+D/2}, z_i * exp(i pos theta_i)
    x = np.asarray(x, dtype=np.float64)
    D = x.shape[-1]
    h = D // 2
    theta = base ** (-2.0 * np.arange(h) / D)
    z = (x[..., :h] + 1j * x[..., h:]) * np.exp(1j * np.asarray(pos, np.float64)[..., None] * theta)
    return np.concatenate([z.real, z.imag], axis=-1)


def test_rotation_matches_the_complex_form_and_composes():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((5, 128))
    d = np.array([0, 1, -7, 1000, 131071])
    assert np.allclose(C.rope_rotate(x, d), rope_complex(x, d), atol=1e-9)
    assert np.array_equal(C.rope_rotate(x, np.zeros(5)), x)
    a, b = 123, -4567
    assert np.allclose(C.rope_rotate(C.rope_rotate(x, a), b), C.rope_rotate(x, a + b), atol=1e-9)
    # a rotation keeps every (i, i + 64) pair's length
    y = C.rope_rotate(x, 999)
    assert np.allclose(x[:, :64] ** 2 + x[:, 64:] ** 2, y[:, :64] ** 2 + y[:, 64:] ** 2)
    # unit vector e_i goes to (cos, sin) of the angle at components i and i + 64
    e = np.zeros(128); e[3] = 1.0
    th = 10000.0 ** (-6.0 / 128)
    r = C.rope_rotate(e, 50)
    assert np.isclose(r[3], np.cos(50 * th)) and np.isclose(r[67], np.sin(50 * th))
    assert np.count_nonzero(np.abs(r) > 1e-15) == 2


def test_dot_products_depend_on_relative_position_only():
    rng = np.random.default_rng(1)
    q, k = rng.standard_normal(128), rng.standard_normal(128)
    for a, b in ((0, 5), (100, 105), (70000, 70005)):
        assert np.isclose(C.rope_rotate(q, a) @ C.rope_rotate(k, b), q @ C.rope_rotate(k, b - a))


def _workload_with_positions(seed, drop_p):
    # keys stored as they would be after prefill: k0 rotated to its logical position in its
    # branch; a single-branch cache so that every slot has one position
    for s in range(seed, seed + 100):  # the first cache whose branch lists no slot twice
        w = W.random_dag(s, n_segs=3, n_branches=1, max_list=3, max_seg_len=300, pool_pages=4000,
                         drop_p=drop_p, max_nq=1, allow_dup=False)
        slots = C.branch_slots(w, 0)
        if len(set(slots.tolist())) == len(slots):
            break
    assert len(set(slots.tolist())) == len(slots)
    k0 = np.random.default_rng(seed).standard_normal((len(slots), w.num_kv_heads, 128))
    kp = w.k_pages.clone()
    rot = rope_complex(k0, np.arange(len(slots))[:, None])
    kp[torch.as_tensor(slots // 16), :, torch.as_tensor(slots % 16), :] = torch.from_numpy(rot).to(torch.bfloat16)
    w.k_pages = kp
    return w, k0


@pytest.mark.parametrize("seed", range(4))
def test_reposition_equals_keys_rotated_at_their_new_positions(seed):
    # Repos: kept keys end up as if rotated at positions 0..r-1 from the start (up to the
    # bf16 rounding of the stored keys, which the rotation carries along)
    w, k0 = _workload_with_positions(100 + seed, drop_p=0.4)
    K, V, kept = C.compact(w, 0, reposition=True)
    want = rope_complex(k0[kept], np.arange(len(kept))[:, None])
    assert np.abs(K - want).max() < 0.06  # bf16 storage: |k| <= ~4, 2^-8 relative
    stored = C.compact(w, 0, reposition=False)[0]
    assert np.allclose(C.rope_rotate(stored, (np.arange(len(kept)) - kept)[:, None]), K, atol=1e-12)


def test_compaction_gathers_the_visible_slots_in_order():
    for seed in range(6):
        w = W.random_dag(200 + seed, n_branches=4, drop_p=(0.0, 0.5)[seed % 2], values=True)
        for b in range(w.num_branches):
            K, V, kept = C.compact(w, b)
            # brute force: walk the logical sequence token by token through explicit pages
            slots = []
            for sid in w.branch_segs[w.branch_seg_off[b]:w.branch_seg_off[b + 1]]:
                po, tb, ln = (int(x) for x in w.segs[int(sid)])
                pages = w.page_ids[po:po + (tb + ln + 15) // 16]
                for t in range(tb, tb + ln):
                    slots.append((int(pages[t // 16]), t % 16))
            n = len(slots)
            if w.vis_bits is None:
                vis = np.ones(n, bool)
            else:
                words = w.vis_bits[w.vis_word_off[b]:w.vis_word_off[b + 1]]
                vis = np.array([(int(words[j // 32]) >> (j % 32)) & 1 for j in range(n)], bool)
            assert np.array_equal(kept, np.nonzero(vis)[0])
            for idx, j in enumerate(kept[:50]):
                pg, off = slots[j]
                assert np.array_equal(V[idx], w.v_pages[pg, :, off, :].double().numpy())
                assert np.array_equal(K[idx], w.k_pages[pg, :, off, :].double().numpy())


def test_nothing_dropped_and_no_reposition_is_the_identity_on_a_contiguous_branch():
    w = W.random_dag(300, n_segs=1, n_branches=1, max_list=1, max_seg_len=100, drop_p=0.0)
    K, V, kept = C.compact(w, 0, reposition=True)
    assert np.array_equal(kept, np.arange(len(kept)))  # positions unchanged: delta 0
    assert np.array_equal(K, C.compact(w, 0)[0])


def _rot_sign_flipped(x, d, base=10000.0):
    x = np.asarray(x, dtype=np.float64)
    h = x.shape[-1] // 2
    th = base ** (-2.0 * np.arange(h) / x.shape[-1])
    a = np.asarray(d, np.float64)[..., None] * th
    return np.concatenate([x[..., :h] * np.cos(a) + x[..., h:] * np.sin(a),
                           x[..., h:] * np.cos(a) - x[..., :h] * np.sin(a)], axis=-1)


def _rot_interleaved(x, d, base=10000.0):
    x = np.asarray(x, dtype=np.float64)
    D = x.shape[-1]
    th = base ** (-2.0 * np.arange(D // 2) / D)
    a = np.asarray(d, np.float64)[..., None] * th
    e, o = x[..., 0::2], x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = e * np.cos(a) - o * np.sin(a)
    out[..., 1::2] = o * np.cos(a) + e * np.sin(a)
    return out


@pytest.mark.parametrize("mutant", [_rot_sign_flipped, _rot_interleaved])
def test_planted_rotation_mistakes_fail_the_pins(monkeypatch, mutant):
    monkeypatch.setattr(C, "rope_rotate", mutant)
    rng = np.random.default_rng(0)
    x = rng.standard_normal((3, 128))
    assert not np.allclose(C.rope_rotate(x, np.array([1, 50, 1000])), rope_complex(x, np.array([1, 50, 1000])))
    w, k0 = _workload_with_positions(100, drop_p=0.4)
    K, _, kept = C.compact(w, 0, reposition=True)
    assert np.abs(K - rope_complex(k0[kept], np.arange(len(kept))[:, None])).max() > 0.5
