"""Pins for the oracle's load-balancing scalar and its gradient.

Closed forms (uniform scores give 1; scores concentrated on the k chosen
experts give E / k), torch float64 autograd of the same scalar with the counts
held fixed, central finite differences, and the whole layer's backward with
the scalar added to the loss against torch autograd on a dense restatement.
CPU only.
"""
import numpy as np
import pytest
import torch

from oracle import cpp as O
from synth import make_inputs, f32_from_bf16_bits


def _routing(L, k):
    idx, _ = O.softmax_topk_gates(L, k)
    return idx


@pytest.mark.parametrize("T,E,k", [(64, 8, 2), (33, 5, 1), (100, 16, 4)])
def test_uniform_scores_give_one(T, E, k):
    rng = np.random.default_rng(T)
    L = np.full((T, E), 0.25)
    idx = rng.integers(0, E, size=(T, k))          # any routing: sum_e f_e = 1
    lbl, P, f = O.load_balance(L, idx, E)
    assert abs(lbl - 1.0) < 1e-14
    np.testing.assert_allclose(P, 1.0 / E, rtol=0, atol=1e-15)
    assert abs(f.sum() - 1.0) < 1e-15


@pytest.mark.parametrize("E,k", [(8, 2), (32, 4), (6, 6)])
def test_scores_concentrated_on_the_chosen_experts_give_E_over_k(E, k):
    T = 50
    L = np.zeros((T, E))
    L[:, :k] = 60.0                                  # all tokens choose experts 0..k-1
    idx = _routing(L, k)
    assert (np.sort(idx, axis=1) == np.arange(k)).all()
    lbl, P, f = O.load_balance(L, idx, E)
    assert abs(lbl - E / k) < 1e-12 * E


def _torch_lbl(L, idx, E, coef):
    T, k = idx.shape
    f = torch.from_numpy(np.bincount(idx.ravel(), minlength=E) / (T * k))
    p = torch.softmax(L, dim=-1)
    return coef * E * (f * p.mean(0)).sum()


def test_gradient_matches_torch_autograd():
    rng = np.random.default_rng(7)
    T, E, k, coef = 40, 12, 3, 0.37
    L = rng.standard_normal((T, E)) * 2
    idx = _routing(L, k)
    Lt = torch.from_numpy(L).requires_grad_()
    _torch_lbl(Lt, idx, E, coef).backward()
    ours = O.load_balance_dlogits(L, idx, E, coef)
    np.testing.assert_allclose(ours, Lt.grad.numpy(), rtol=1e-12, atol=1e-16)


def test_gradient_central_finite_differences():
    rng = np.random.default_rng(8)
    T, E, k, coef = 9, 6, 2, 1.3
    L = rng.standard_normal((T, E))
    idx = _routing(L, k)                             # the counts stay fixed
    g = O.load_balance_dlogits(L, idx, E, coef)
    eps = 1e-6
    for _ in range(12):
        t, e = int(rng.integers(T)), int(rng.integers(E))
        Lp, Lm = L.copy(), L.copy()
        Lp[t, e] += eps
        Lm[t, e] -= eps
        num = coef * (O.load_balance(Lp, idx, E)[0] - O.load_balance(Lm, idx, E)[0]) / (2 * eps)
        assert abs(num - g[t, e]) <= 1e-8 * (1 + abs(g[t, e]))


def _f(a):
    return torch.from_numpy(f32_from_bf16_bits(a).astype(np.float64))


def test_layer_backward_with_the_balance_term_matches_autograd():
    """Loss = <out, dOut> + coef * LBL(logits): dlogits, dx and dW_r pick up the
    scalar's gradient through the router; the expert weight gradients do not."""
    T, d, E, k, f, coef = 24, 16, 6, 2, 16, 0.8
    inp = make_inputs(T=T, d=d, E=E, k=k, f=f, seed=21)
    fwd = O.layer_forward(inp["x"], inp["w_router"], inp["bias"], inp["w_gate"], inp["w_up"],
                          inp["w_down"], k, bm=16)
    bwd = O.layer_backward(fwd, inp["d_out"], inp["x"], inp["w_router"], inp["w_gate"],
                           inp["w_up"], inp["w_down"], lb_coef=coef)
    x = _f(inp["x"]).requires_grad_()
    wr = _f(inp["w_router"]).requires_grad_()
    wg, wu, wd = _f(inp["w_gate"]), _f(inp["w_up"]), _f(inp["w_down"])
    wg.requires_grad_()
    bias = torch.from_numpy(inp["bias"].astype(np.float64))
    logits = x @ wr.T + bias
    logits.retain_grad()
    p = torch.softmax(logits, dim=-1)
    idx = torch.topk(logits, k, dim=-1).indices
    psel = torch.gather(p, 1, idx)
    g = psel / psel.sum(-1, keepdim=True)
    G = torch.zeros_like(logits).scatter(1, idx, g)
    out = torch.zeros_like(x)
    for e in range(E):
        out = out + G[:, e:e + 1] * ((torch.nn.functional.silu(x @ wg[e].T) * (x @ wu[e].T)) @ wd[e].T)
    loss = (out * _f(inp["d_out"])).sum() + _torch_lbl(logits, idx.numpy(), E, coef)
    loss.backward()
    rel = lambda a, b: np.abs(a - b).max() / max(np.abs(b).max(), 1e-300)
    assert rel(bwd["dlogits"], logits.grad.numpy()) < 1e-11
    assert rel(bwd["dx"], x.grad.numpy()) < 1e-11
    assert rel(bwd["dW_router"], wr.grad.numpy()) < 1e-11
    assert rel(bwd["dW_gate"], wg.grad.numpy()) < 1e-11
    # without the term the router gradients differ
    plain = O.layer_backward(fwd, inp["d_out"], inp["x"], inp["w_router"], inp["w_gate"],
                             inp["w_up"], inp["w_down"])
    assert rel(plain["dlogits"], logits.grad.numpy()) > 1e-6
