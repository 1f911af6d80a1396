"""Pins for the oracle's expert layer: forward and backward.

Forward: a brute-force restatement with no dispatch (every expert on every
token, masked by the gate matrix) and, for E = 1, k = 1, a dense SwiGLU MLP
written with torch ops.  Backward: torch.autograd in float64 on a dense torch
restatement, plus central finite differences on tiny shapes.  CPU only.
"""
import numpy as np
import pytest
import torch

from oracle import cpp as O
from synth import make_inputs, f32_from_bf16_bits


def _f(a):
    return torch.from_numpy(f32_from_bf16_bits(a).astype(np.float64))


def _rel(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return np.abs(a - b).max() / max(np.abs(b).max(), 1e-300)


def _layer(inp, k, bm=16):
    return O.layer_forward(inp["x"], inp["w_router"], inp["bias"], inp["w_gate"], inp["w_up"],
                           inp["w_down"], k=k, bm=bm)


@pytest.mark.parametrize("T,d,E,k,f", [(24, 32, 6, 2, 48), (17, 16, 4, 4, 32), (9, 8, 3, 1, 16)])
def test_forward_matches_dense_restatement(T, d, E, k, f):
    inp = make_inputs(T=T, d=d, E=E, k=k, f=f, seed=T)
    fwd = _layer(inp, k)
    dense = O.dense_forward(inp["x"], inp["w_router"], inp["bias"], inp["w_gate"], inp["w_up"],
                            inp["w_down"], k)
    assert _rel(fwd["out"], dense) < 1e-12


def test_single_expert_top1_is_a_dense_swiglu_mlp():
    inp = make_inputs(T=31, d=24, E=1, k=1, f=40, seed=7)
    fwd = _layer(inp, 1)
    x, wg, wu, wd = _f(inp["x"]), _f(inp["w_gate"])[0], _f(inp["w_up"])[0], _f(inp["w_down"])[0]
    ref = (torch.nn.functional.silu(x @ wg.T) * (x @ wu.T)) @ wd.T
    assert np.allclose(fwd["gates"], 1.0)
    assert _rel(fwd["out"], ref.numpy()) < 1e-13


def test_padding_does_not_change_the_result():
    inp = make_inputs(T=50, d=16, E=5, k=2, f=32, seed=8)
    a = _layer(inp, 2, bm=1)
    b = _layer(inp, 2, bm=128)
    # BLAS may block differently for different row counts: equal up to rounding
    assert _rel(a["out"], b["out"]) < 1e-13
    assert b["row_offsets"][-1] % 128 == 0


def _torch_dense(x, wr, bias, wg, wu, wd, k):
    logits = x @ wr.T + bias
    logits.retain_grad()
    p = torch.softmax(logits, dim=-1)
    idx = torch.topk(logits, k, dim=-1).indices
    psel = torch.gather(p, 1, idx)
    g = psel / psel.sum(-1, keepdim=True)
    G = torch.zeros_like(logits).scatter(1, idx, g)
    out = torch.zeros_like(x)
    for e in range(wg.shape[0]):
        ye = (torch.nn.functional.silu(x @ wg[e].T) * (x @ wu[e].T)) @ wd[e].T
        out = out + G[:, e:e + 1] * ye
    return out, logits


@pytest.mark.parametrize("T,d,E,k,f", [(32, 16, 6, 2, 24), (20, 8, 4, 3, 16), (12, 8, 3, 3, 8)])
def test_backward_matches_torch_autograd(T, d, E, k, f):
    inp = make_inputs(T=T, d=d, E=E, k=k, f=f, seed=100 + T)
    fwd = _layer(inp, k)
    bwd = O.layer_backward(fwd, inp["d_out"], inp["x"], inp["w_router"], inp["w_gate"], inp["w_up"],
                           inp["w_down"])
    x = _f(inp["x"]).requires_grad_()
    wr = _f(inp["w_router"]).requires_grad_()
    wg = _f(inp["w_gate"]).requires_grad_()
    wu = _f(inp["w_up"]).requires_grad_()
    wd = _f(inp["w_down"]).requires_grad_()
    bias = torch.from_numpy(inp["bias"].astype(np.float64))
    out, logits = _torch_dense(x, wr, bias, wg, wu, wd, k)
    assert _rel(fwd["out"], out.detach().numpy()) < 1e-12
    out.backward(_f(inp["d_out"]))
    for name, ref in [("dx", x.grad), ("dW_router", wr.grad), ("dW_gate", wg.grad),
                      ("dW_up", wu.grad), ("dW_down", wd.grad), ("dlogits", logits.grad)]:
        assert _rel(bwd[name], ref.numpy()) < 1e-11, name


def test_backward_central_finite_differences():
    T, d, E, k, f = 6, 8, 4, 2, 8
    inp = make_inputs(T=T, d=d, E=E, k=k, f=f, seed=42)
    dO = O.as_f64(inp["d_out"])
    base = {n: O.as_f64(inp[n]) for n in ("x", "w_router", "w_gate", "w_up", "w_down")}
    bias = O.as_f64(inp["bias"])

    def loss(p):
        fw = O.layer_forward(p["x"], p["w_router"], bias, p["w_gate"], p["w_up"], p["w_down"], k, bm=4)
        return float((fw["out"] * dO).sum()), fw

    _, fw = loss(base)
    g = O.layer_backward(fw, inp["d_out"], base["x"], base["w_router"], base["w_gate"],
                         base["w_up"], base["w_down"])
    grads = {"x": g["dx"], "w_router": g["dW_router"], "w_gate": g["dW_gate"], "w_up": g["dW_up"],
             "w_down": g["dW_down"]}
    rng = np.random.default_rng(0)
    eps = 1e-6
    for name, arr in base.items():
        for _ in range(6):
            pos = tuple(rng.integers(0, s) for s in arr.shape)
            p_plus = dict(base)
            p_minus = dict(base)
            p_plus[name] = arr.copy()
            p_minus[name] = arr.copy()
            p_plus[name][pos] += eps
            p_minus[name][pos] -= eps
            num = (loss(p_plus)[0] - loss(p_minus)[0]) / (2 * eps)
            ana = grads[name][pos]
            assert abs(num - ana) <= 1e-6 * (1 + abs(ana)), (name, pos, num, ana)


def test_empty_experts_get_exact_zero_weight_gradients():
    inp = make_inputs(T=40, d=16, E=6, k=2, f=16, seed=9)
    inp["bias"][:, 4] -= 100.0
    fwd = _layer(inp, 2)
    assert fwd["counts"][4] == 0
    bwd = O.layer_backward(fwd, inp["d_out"], inp["x"], inp["w_router"], inp["w_gate"], inp["w_up"],
                           inp["w_down"])
    for n in ("dW_gate", "dW_up", "dW_down"):
        assert not bwd[n][4].any()
        assert bwd[n][0].any()
    assert not bwd["dlogits"][:, 4].any()


def test_dx_sums_over_routes():
    """sum_t dx[t] (without the router term) equals the column sum of dXd over real rows."""
    inp = make_inputs(T=30, d=16, E=5, k=3, f=16, seed=10)
    fwd = _layer(inp, 3)
    bwd = O.layer_backward(fwd, inp["d_out"], inp["x"], None, inp["w_gate"], inp["w_up"], inp["w_down"])
    real = fwd["route_of_slot"] >= 0
    np.testing.assert_allclose(bwd["dx"].sum(0), bwd["dXd"][real].sum(0), rtol=1e-12, atol=1e-12)
