"""Pins for the oracle's routing steps (router, softmax/top-k, counts, offsets, slots).

Each test checks the oracle against something other than its own formula:
a brute-force selection procedure, a closed form, a library routine or an
invariant.  CPU only.
"""
import numpy as np
import pytest
import scipy.special

from oracle import cpp as O
from synth import make_inputs, f32_from_bf16_bits


def _brute_topk(row, k):
    """Repeatedly take the largest remaining logit, lowest id first on ties."""
    remaining = list(range(len(row)))
    chosen = []
    for _ in range(k):
        best = remaining[0]
        for e in remaining[1:]:
            if row[e] > row[best]:
                best = e
        chosen.append(best)
        remaining.remove(best)
    return chosen


@pytest.mark.parametrize("T,E,k", [(64, 8, 2), (50, 16, 4), (33, 5, 5), (40, 32, 1)])
def test_topk_matches_brute_force(T, E, k):
    rng = np.random.default_rng(T * 1000 + E)
    # coarse values so that ties are frequent
    L = rng.integers(-3, 4, size=(T, E)).astype(np.float64) * 0.5
    idx, gates = O.softmax_topk_gates(L, k)
    for t in range(T):
        assert list(idx[t]) == _brute_topk(L[t], k)


def test_all_equal_logits_pick_lowest_ids_with_uniform_gates():
    T, E, k = 7, 12, 4
    idx, gates = O.softmax_topk_gates(np.full((T, E), 0.37), k)
    assert (idx == np.arange(k)[None, :]).all()
    np.testing.assert_allclose(gates, 1.0 / k, rtol=0, atol=1e-15)


def test_k_equals_E_is_the_full_softmax():
    rng = np.random.default_rng(3)
    L = rng.standard_normal((20, 9))
    idx, gates = O.softmax_topk_gates(L, 9)
    ref = scipy.special.softmax(L, axis=1)
    np.testing.assert_allclose(gates, np.take_along_axis(ref, idx, axis=1), rtol=1e-13)
    # descending logits
    assert (np.diff(np.take_along_axis(L, idx, axis=1), axis=1) <= 0).all()


def test_top2_gate_is_logistic_of_the_logit_gap():
    rng = np.random.default_rng(4)
    L = rng.standard_normal((30, 6)) * 3
    idx, gates = O.softmax_topk_gates(L, 2)
    l1 = np.take_along_axis(L, idx[:, :1], axis=1)[:, 0]
    l2 = np.take_along_axis(L, idx[:, 1:2], axis=1)[:, 0]
    np.testing.assert_allclose(gates[:, 0], scipy.special.expit(l1 - l2), rtol=1e-13)
    np.testing.assert_allclose(gates.sum(1), 1.0, rtol=0, atol=1e-14)


def test_negative_zero_ties_with_zero():
    L = np.array([[0.0, -0.0, -1.0, -0.0]])
    idx, _ = O.softmax_topk_gates(L, 3)
    assert list(idx[0]) == [0, 1, 3]


def test_nonfinite_logits_raise():
    L = np.zeros((2, 4))
    L[1, 2] = np.nan
    with pytest.raises(FloatingPointError):
        O.softmax_topk_gates(L, 2)
    L[1, 2] = np.inf
    with pytest.raises(FloatingPointError):
        O.softmax_topk_gates(L, 2)


def test_router_logits_against_float_sum():
    inp = make_inputs(T=5, d=64, E=4, k=2, f=128, seed=1)
    L = O.router_logits(inp["x"], inp["w_router"], inp["bias"])
    x = f32_from_bf16_bits(inp["x"]).astype(float)
    w = f32_from_bf16_bits(inp["w_router"]).astype(float)
    for t in range(5):
        for e in range(4):
            s = float(inp["bias"][t, e])
            for i in range(64):
                s += x[t, i] * w[e, i]
            assert abs(L[t, e] - s) <= 1e-12 * (1 + abs(s))


@pytest.mark.parametrize("bm", [1, 16, 128])
def test_counts_offsets_slots_invariants(bm):
    rng = np.random.default_rng(bm)
    T, E, k = 300, 10, 3
    L = rng.standard_normal((T, E))
    L[:, 7] -= 50.0                       # expert 7 receives nothing
    idx, _ = O.softmax_topk_gates(L, k)
    counts = O.expert_counts(idx, E)
    assert counts.sum() == T * k and counts[7] == 0
    np.testing.assert_array_equal(counts, np.bincount(idx.ravel(), minlength=E))
    offsets = O.exclusive_scan(counts)
    assert offsets[0] == 0 and offsets[-1] == T * k
    np.testing.assert_array_equal(np.diff(offsets), counts)
    tile_offsets, row_offsets = O.tile_layout(counts, bm)
    np.testing.assert_array_equal(np.diff(tile_offsets), -(-counts // bm))
    slot_of_route, route_of_slot = O.assign_slots(idx, row_offsets)
    # inverse permutations on the real rows; -1 exactly on padding rows
    assert (route_of_slot[slot_of_route] == np.arange(T * k)).all()
    assert (route_of_slot >= 0).sum() == T * k
    expert_of_route = idx.ravel()
    for e in range(E):
        seg = route_of_slot[row_offsets[e]:row_offsets[e + 1]]
        real = seg[: counts[e]]
        assert (seg[counts[e]:] == -1).all()
        assert (expert_of_route[real] == e).all()
        assert (np.diff(real) > 0).all()          # ascending (token, choice) order
    if bm == 1:
        # with no padding the slot order is a stable sort of the routes by expert
        order = np.argsort(expert_of_route, kind="stable")
        np.testing.assert_array_equal(route_of_slot, order)


def test_dispatch_copies_rows_exactly():
    inp = make_inputs(T=40, d=32, E=6, k=2, f=64, seed=5)
    fwd = O.layer_forward(inp["x"], inp["w_router"], inp["bias"], inp["w_gate"], inp["w_up"],
                          inp["w_down"], k=2, bm=8)
    x = f32_from_bf16_bits(inp["x"])
    for r, s in enumerate(fwd["slot_of_route"]):
        assert np.array_equal(fwd["Xd"][s], x[r // 2].astype(np.float64))
    pad = fwd["route_of_slot"] < 0
    assert not fwd["Xd"][pad].any()
