"""The C++ oracle against the independent float64 numpy restatement of the same
definition (CPU only).  Integer results (top-k ids, counts, offsets, slots,
quantised codes and scales) must be identical; floating-point results may
differ only by float64 rounding order (BLAS blocking on the numpy side)."""
import numpy as np
import pytest

from oracle import cpp as C
from oracle import moe_oracle as N
from synth import make_inputs

INT_KEYS = ("topk_idx", "counts", "offsets", "tile_offsets", "row_offsets", "slot_of_route",
            "route_of_slot")


def _rel(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return np.abs(a - b).max() / max(np.abs(b).max(), 1e-300)


SHAPES = [(64, 32, 6, 2, 64, 16), (300, 64, 8, 3, 96, 128), (45, 32, 5, 5, 32, 1)]


@pytest.mark.parametrize("T,d,E,k,f,bm", SHAPES)
@pytest.mark.parametrize("mx", [False, True])
def test_layer_forward_backward(T, d, E, k, f, bm, mx):
    inp = make_inputs(T=T, d=d, E=E, k=k, f=f, seed=T + E)
    inp["bias"][:, 1] -= 50.0                       # an expert without routes
    args = (inp["x"], inp["w_router"], inp["bias"], inp["w_gate"], inp["w_up"], inp["w_down"])
    if mx:
        cf, nf = C.layer_forward_mxfp8(*args, k=k, bm=bm), N.layer_forward_mxfp8(*args, k=k, bm=bm)
    else:
        cf, nf = C.layer_forward(*args, k=k, bm=bm), N.layer_forward(*args, k=k, bm=bm)
    for key in INT_KEYS:
        np.testing.assert_array_equal(cf[key], nf[key], err_msg=key)
    for key in ("logits", "gates", "Xd", "H", "U", "A", "Y", "out") + (("Aq",) if mx else ()):
        assert _rel(cf[key], nf[key]) < 1e-12, key
    bw = (C.layer_backward_mxfp8, N.layer_backward_mxfp8) if mx else (C.layer_backward,
                                                                       N.layer_backward)
    cb = bw[0](cf, inp["d_out"], inp["x"], inp["w_router"], inp["w_gate"], inp["w_up"],
               inp["w_down"], lb_coef=0.05)
    nb = bw[1](nf, inp["d_out"], inp["x"], inp["w_router"], inp["w_gate"], inp["w_up"],
               inp["w_down"], lb_coef=0.05)
    assert set(cb) == set(nb)
    for key in nb:
        assert _rel(cb[key], nb[key]) < 1e-12, key


def test_routing_ties_and_dense_forward():
    rng = np.random.default_rng(3)
    L = rng.integers(-3, 3, (200, 16)).astype(np.float64)   # many equal logits
    ci, cg = C.softmax_topk_gates(L, 5)
    ni, ng = N.softmax_topk_gates(L, 5)
    np.testing.assert_array_equal(ci, ni)
    assert _rel(cg, ng) < 1e-14
    inp = make_inputs(T=20, d=16, E=4, k=2, f=24, seed=4)
    args = (inp["x"], inp["w_router"], inp["bias"], inp["w_gate"], inp["w_up"], inp["w_down"])
    assert _rel(C.dense_forward(*args, 2), N.dense_forward(*args, 2)) < 1e-12
    with pytest.raises(FloatingPointError):
        C.softmax_topk_gates(np.array([[0.0, np.inf]]), 1)


def test_quantiser_and_e4m3_table():
    np.testing.assert_array_equal(C.E4M3_VALUES[:127], N.E4M3_VALUES[:127])
    np.testing.assert_array_equal(C.E4M3_VALUES[128:255], N.E4M3_VALUES[128:255])
    assert np.isnan(C.E4M3_VALUES[127]) and np.isnan(C.E4M3_VALUES[255])
    rng = np.random.default_rng(5)
    v = rng.standard_normal((96, 256)) * np.exp2(rng.integers(-130, 130, (96, 1)))
    v[0] = 0.0
    v[1, :32] = -0.0
    v[2, :32] = N.E4M3_VALUES[rng.integers(0, 126, 32)] * 4.0
    for a, b in zip(C.quantize_mxfp8(v), N.quantize_mxfp8(v)):
        np.testing.assert_array_equal(a, b)
    amax = np.abs(rng.standard_normal(1000)) * np.exp2(rng.integers(-140, 140, 1000))
    np.testing.assert_array_equal(C.mx_scale_exponent(amax), N.mx_scale_exponent(amax))
    w = rng.standard_normal(5000) * 300
    np.testing.assert_array_equal(C.e4m3_encode(w), N.e4m3_encode(w))


def test_load_balance():
    rng = np.random.default_rng(6)
    L = rng.standard_normal((128, 12))
    idx, _ = C.softmax_topk_gates(L, 3)
    c, n = C.load_balance(L, idx, 12), N.load_balance(L, idx, 12)
    assert abs(c[0] - n[0]) < 1e-13
    assert _rel(c[1], n[1]) < 1e-13 and _rel(c[2], n[2]) < 1e-15
    assert _rel(C.load_balance_dlogits(L, idx, 12, 0.3), N.load_balance_dlogits(L, idx, 12, 0.3)) < 1e-12
