"""Load-balancing statistics and the loss term's gradient on the GPU, against
the oracle: moe_load_balance (and the layer forward's saved lb_stats), the
term added to dlogits in the combine backward, and the dense router backward
it implies for dx and dW_r.  GPU only."""
import numpy as np
import pytest
import torch

from oracle import cpp as O
from synth import make_inputs
from gpu_util import f64, max_abs_rel, to_dev_bf16

pytestmark = pytest.mark.gpu
TOL = 2e-2


@pytest.mark.parametrize("T,E,k", [(1000, 16, 4), (777, 128, 4), (50, 256, 32), (8192, 32, 4)])
def test_load_balance_statistics(moe_gpu, T, E, k):
    m, dev = moe_gpu
    rng = np.random.default_rng(T + E)
    L = (rng.standard_normal((T, E)) * 1.5).astype(np.float32)
    s = m.shape(T, 128, E, k, 128)
    buf = m.allocate(s, with_grads=False)
    buf.saved["logits"].copy_(torch.from_numpy(L))
    sv = buf.saved
    m.route(s, None, None, None, sv["logits"], sv["topk_idx"], sv["gates"], sv["counts"],
            sv["offsets"], sv["tile_offsets"], sv["slot_of_route"], sv["route_of_slot"], buf.ws)
    stats = torch.empty(E + 1, dtype=torch.float32, device=dev)
    m.load_balance(s, sv["logits"], sv["counts"], stats, buf.ws)
    lbl, P, f = O.load_balance(L, sv["topk_idx"].cpu().numpy(), E)
    got = stats.cpu().numpy().astype(np.float64)
    assert abs(got[0] - lbl) <= 1e-5 * lbl
    np.testing.assert_allclose(got[1:], P, rtol=0, atol=1e-6)
    assert m.read_error(buf.ws) == 0


def test_uniform_scores_give_one(moe_gpu):
    m, dev = moe_gpu
    T, E, k = 300, 12, 3
    s = m.shape(T, 128, E, k, 128)
    buf = m.allocate(s, with_grads=False)
    buf.saved["logits"].fill_(0.5)
    sv = buf.saved
    m.route(s, None, None, None, sv["logits"], sv["topk_idx"], sv["gates"], sv["counts"],
            sv["offsets"], sv["tile_offsets"], sv["slot_of_route"], sv["route_of_slot"], buf.ws)
    stats = torch.empty(E + 1, dtype=torch.float32, device=dev)
    m.load_balance(s, sv["logits"], sv["counts"], stats, buf.ws)
    got = stats.cpu().numpy()
    assert abs(got[0] - 1.0) < 1e-5
    np.testing.assert_allclose(got[1:], 1.0 / E, rtol=1e-6)


def run_layer_lb(m, dev, inp, k, coef, use_router, logits32=None):
    T, d, E, f = inp["T"], inp["d"], inp["E"], inp["f"]
    s = m.shape(T, d, E, k, f)
    buf = m.allocate(s, load_balance=True)
    t = {n: to_dev_bf16(inp[n], dev) for n in ("x", "w_router", "w_gate", "w_up", "w_down", "d_out")}
    bias = torch.from_numpy(inp["bias"]).to(dev) if use_router else None
    if not use_router:
        buf.saved["logits"].copy_(torch.from_numpy(logits32))
    wr = t["w_router"] if use_router else None
    out = torch.empty(T, d, dtype=torch.bfloat16, device=dev)
    m.clear_error(buf.ws)
    m.forward(buf, t["x"], wr, bias, t["w_gate"], t["w_up"], t["w_down"], out)
    m.backward(buf, t["d_out"], t["x"], wr, t["w_gate"], t["w_up"], t["w_down"], lb_coef=coef)
    assert m.read_error(buf.ws) == 0
    return buf


@pytest.mark.parametrize("T,d,E,k,f", [(1000, 256, 16, 4, 256), (513, 128, 64, 8, 128)],
                         ids=lambda v: str(v))
def test_loss_term_gradient_on_shared_logits(moe_gpu, T, d, E, k, f):
    """Routing bit-exact on shared logits; the forward's lb_stats and the term's
    gradient on the logits no route selects (where it is the only part) match the
    oracle; the other gradients keep the bf16 tolerance."""
    m, dev = moe_gpu
    coef = 0.7
    inp = make_inputs(T=T, d=d, E=E, k=k, f=f, seed=T + 3)
    L32 = O.router_logits(inp["x"], inp["w_router"], inp["bias"]).astype(np.float32)
    buf = run_layer_lb(m, dev, inp, k, coef, use_router=False, logits32=L32)
    fwd = O.layer_forward(inp["x"], None, None, inp["w_gate"], inp["w_up"], inp["w_down"], k,
                          logits=L32)
    np.testing.assert_array_equal(buf.saved["topk_idx"].cpu().numpy(), fwd["topk_idx"])
    lbl, P, _ = O.load_balance(L32, fwd["topk_idx"], E)
    stats = buf.saved["lb_stats"].cpu().numpy().astype(np.float64)
    assert abs(stats[0] - lbl) <= 1e-5 * lbl
    np.testing.assert_allclose(stats[1:], P, rtol=0, atol=1e-6)
    bwd = O.layer_backward(fwd, inp["d_out"], inp["x"], None, inp["w_gate"], inp["w_up"],
                           inp["w_down"], lb_coef=coef)
    dl = f64(buf.grads["dlogits"])
    unselected = np.ones((T, E), dtype=bool)
    unselected[np.arange(T)[:, None], fwd["topk_idx"]] = False
    term = O.load_balance_dlogits(L32, fwd["topk_idx"], E, coef)
    assert np.abs(term[unselected]).max() > 0
    assert max_abs_rel(dl[unselected], term[unselected]) <= 1e-4
    assert max_abs_rel(dl, bwd["dlogits"]) <= TOL
    for mine, ref in [("dx", "dx"), ("d_gates", "d_gates"), ("dw_gate", "dW_gate"),
                      ("dw_down", "dW_down")]:
        assert max_abs_rel(f64(buf.grads[mine]), bwd[ref]) <= TOL, mine


@pytest.mark.parametrize("T,d,E,k,f", [(1000, 256, 16, 4, 256), (300, 512, 128, 4, 128)],
                         ids=lambda v: str(v))
def test_dense_router_backward(moe_gpu, T, d, E, k, f):
    """With the router projection on the device and a coefficient large enough
    for the term to dominate, dx and dW_r (dense router backward) match the
    oracle; tokens at a near-tie of the oracle's logits are left out of dx."""
    m, dev = moe_gpu
    coef = 500.0 * T          # the term's scale coef * E / T = 500 E: it dominates dlogits
    inp = make_inputs(T=T, d=d, E=E, k=k, f=f, seed=T + 5)
    buf = run_layer_lb(m, dev, inp, k, coef, use_router=True)
    fwd = O.layer_forward(inp["x"], inp["w_router"], inp["bias"], inp["w_gate"], inp["w_up"],
                          inp["w_down"], k)
    same = (buf.saved["topk_idx"].cpu().numpy() == fwd["topk_idx"]).all(1)
    assert same.mean() > 0.99
    bwd = O.layer_backward(fwd, inp["d_out"], inp["x"], inp["w_router"], inp["w_gate"],
                           inp["w_up"], inp["w_down"], lb_coef=coef)
    assert max_abs_rel(f64(buf.grads["dlogits"])[same], bwd["dlogits"][same]) <= TOL
    assert max_abs_rel(f64(buf.grads["dx"])[same], bwd["dx"][same]) <= TOL
    if same.all():
        assert max_abs_rel(f64(buf.grads["dw_router"]), bwd["dW_router"]) <= 1e-3


def test_recompute_with_the_balance_term_is_bitwise_the_saved_one(moe_gpu):
    """Both options together: recomputed activations and the loss term give the
    same gradients, bit for bit, as the saving backward with the term."""
    m, dev = moe_gpu
    T, d, E, k, f = 1000, 256, 16, 4, 256
    inp = make_inputs(T=T, d=d, E=E, k=k, f=f, seed=31)
    buf = run_layer_lb(m, dev, inp, k, 3.0, use_router=True)
    names = ("dx", "dw_router", "dw_gate", "dw_up", "dw_down", "d_gates", "dlogits")
    saved = {n: buf.grads[n].clone() for n in names}
    for n in ("xd", "h", "u", "a", "y"):
        buf.saved[n].fill_(float("nan"))
    t = {n: to_dev_bf16(inp[n], dev) for n in ("x", "w_router", "w_gate", "w_up", "w_down", "d_out")}
    m.backward(buf, t["d_out"], t["x"], t["w_router"], t["w_gate"], t["w_up"], t["w_down"],
               recompute=True, lb_coef=3.0)
    assert m.read_error(buf.ws) == 0
    for n in names:
        assert torch.equal(buf.grads[n], saved[n]), n


def test_invalid_backward_options_are_rejected(moe_gpu):
    m, dev = moe_gpu
    T, d, E, k, f = 64, 128, 4, 2, 128
    inp = make_inputs(T=T, d=d, E=E, k=k, f=f, seed=2)
    buf = run_layer_lb(m, dev, inp, k, 0.0, use_router=True)
    t = {n: to_dev_bf16(inp[n], dev) for n in ("x", "w_router", "w_gate", "w_up", "w_down", "d_out")}
    with pytest.raises(m.MoEError):
        m.backward(buf, t["d_out"], t["x"], t["w_router"], t["w_gate"], t["w_up"], t["w_down"],
                   lb_coef=float("nan"))
    with pytest.raises(m.MoEError):
        m.backward(buf, t["d_out"], t["x"], t["w_router"], t["w_gate"], t["w_up"], t["w_down"],
                   lb_coef=float("inf"))
    # recompute is a 0/1 flag; any other value is refused before anything runs
    g = buf.grads
    ba = m.BwdArgs(d_out=t["d_out"].data_ptr(), x=t["x"].data_ptr(),
                   w_router=t["w_router"].data_ptr(), w_gate=t["w_gate"].data_ptr(),
                   w_up=t["w_up"].data_ptr(), w_down=t["w_down"].data_ptr(),
                   recompute=2, lb_coef=0.0, **{n: v.data_ptr() for n, v in g.items()})
    with pytest.raises(m.MoEError):
        m.layer_bwd(buf.shape, ba, buf.saved_struct(), buf.ws)
    assert m.read_error(buf.ws) == 0
