"""Pins for the oracle's router top-k, gates and route map (CPU only).

Each check below is independent of the oracle's own code path: brute force over
all k-subsets, pairwise dominance, hand-worked examples and closed forms.
"""
import itertools

import numpy as np
import pytest

from oracle import layer as ol


def _beats(z, a, b):
    """a precedes b in the total order (logit descending, id ascending)."""
    return z[a] > z[b] or (z[a] == z[b] and a < b)


def _brute_topk_row(z, k):
    E = len(z)
    winners = [S for S in itertools.combinations(range(E), k)
               if all(_beats(z, a, b) for a in S for b in range(E) if b not in S)]
    assert len(winners) == 1, "the total order admits exactly one top-k set"
    S = winners[0]
    # position of a within the selected set = how many selected ids beat it
    pos = {a: sum(_beats(z, b, a) for b in S if b != a) for a in S}
    return [a for a, _ in sorted(pos.items(), key=lambda kv: kv[1])]


@pytest.mark.parametrize("E,k", [(1, 1), (3, 1), (4, 2), (6, 3), (8, 4), (8, 8), (5, 5)])
def test_topk_brute_force_with_ties(E, k):
    rng = np.random.default_rng(E * 10 + k)
    # values from a tiny set force many exact ties; include both signed zeros
    choices = np.array([-1.0, -0.0, 0.0, 0.5, 1.0], np.float32)
    z = rng.choice(choices, size=(64, E)).astype(np.float32)
    idx = ol.topk(z, k)
    for t in range(z.shape[0]):
        assert list(idx[t]) == _brute_topk_row(z[t], k), (t, z[t])


def test_topk_brute_force_continuous():
    rng = np.random.default_rng(1)
    z = rng.standard_normal((64, 7)).astype(np.float32)
    idx = ol.topk(z, 3)
    for t in range(64):
        assert list(idx[t]) == _brute_topk_row(z[t], 3)


def test_topk_signed_zero_is_a_tie():
    z = np.array([[-0.0, 0.0, -1.0]], np.float32)
    assert list(ol.topk(z, 2)[0]) == [0, 1]
    z = np.array([[0.0, -0.0, -1.0]], np.float32)
    assert list(ol.topk(z, 2)[0]) == [0, 1]


def test_topk_rejects_nan_and_bad_k():
    with pytest.raises(ValueError):
        ol.topk(np.array([[np.nan, 1.0]], np.float32), 1)
    with pytest.raises(ValueError):
        ol.topk(np.zeros((1, 3), np.float32), 4)


def test_gates_closed_forms():
    rng = np.random.default_rng(2)
    z = rng.standard_normal((128, 16)).astype(np.float32)
    for k in (1, 2, 4, 16):
        idx = ol.topk(z, k)
        g = ol.topk_gates(z, idx)
        np.testing.assert_allclose(g.sum(axis=1), 1.0, rtol=0, atol=1e-14)
        assert np.all(np.diff(g, axis=1) <= 0), "slot order is descending logit"
        # renormalised full softmax over the selected experts (closed form)
        full = np.exp(z.astype(np.float64))
        full /= full.sum(axis=1, keepdims=True)
        sel = np.take_along_axis(full, idx.astype(np.int64), axis=1)
        np.testing.assert_allclose(g, sel / sel.sum(axis=1, keepdims=True), rtol=1e-12)
    # k = 1 gives gate 1 exactly; equal logits give 1/k
    assert np.all(ol.topk_gates(z, ol.topk(z, 1)) == 1.0)
    eq = np.full((3, 4), 0.7, np.float32)
    np.testing.assert_allclose(ol.topk_gates(eq, ol.topk(eq, 4)), 0.25, rtol=1e-15)


def test_route_map_hand_worked():
    # T=4, k=2, E=3; flattened slots s = t*k + j hold experts 2,0 | 0,1 | 2,1 | 0,2
    idx = np.array([[2, 0], [0, 1], [2, 1], [0, 2]], np.int32)
    counts, offsets, ros, sor = ol.route_map(idx, 3)
    # expert 0 owns slots 1,2,6; expert 1 slots 3,5; expert 2 slots 0,4,7
    assert list(counts) == [3, 2, 3]
    assert list(offsets) == [0, 3, 5, 8]
    assert list(sor) == [1, 2, 6, 3, 5, 0, 4, 7]
    assert list(ros) == [5, 0, 1, 3, 6, 4, 2, 7]


@pytest.mark.parametrize("T,k,E", [(1, 1, 1), (7, 2, 5), (33, 4, 8), (50, 3, 64), (0, 2, 4)])
def test_route_map_brute_force(T, k, E):
    rng = np.random.default_rng(T + 100 * E)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]) if T else np.zeros((0, k), np.int32)
    counts, offsets, ros, sor = ol.route_map(idx, E)
    flat = list(np.asarray(idx).reshape(-1))
    R = len(flat)
    assert counts.sum() == R and offsets[0] == 0 and offsets[-1] == R
    assert np.all(np.diff(offsets) >= 0)
    for e in range(E):
        assert counts[e] == sum(1 for v in flat if v == e)
    for s in range(R):
        e = flat[s]
        rank = sum(1 for s2 in range(s) if flat[s2] == e)
        assert ros[s] == sum(counts[:e]) + rank
    # bijection: slot_of_row is the inverse of row_of_slot
    assert sorted(ros) == list(range(R))
    assert all(sor[ros[s]] == s for s in range(R))
    # each segment lists its slots in ascending order
    for e in range(E):
        seg = sor[offsets[e]:offsets[e + 1]]
        assert np.all(np.diff(seg) > 0)


def test_route_map_rejects_bad_expert_id():
    with pytest.raises(ValueError):
        ol.route_map(np.array([[0, 3]]), 3)
