"""Whole-layer parity on random shapes (a fixed seed): BF16 and MXFP8 layers,
forward + backward on shared fp32 logits, against the oracle — routing, counts
and slots bit-exact, floating-point outputs within max-abs-rel 2e-2 (BF16) or
6e-2 (MXFP8, against the MXFP8 oracle).  The shapes span 1-1500 tokens, d and f
multiples of 128 up to 768 and 640, 1-100 experts (sometimes one left without
routes), top-1 to top-12.  GPU only."""
import numpy as np
import pytest
import torch

from oracle import cpp as O
from synth import make_inputs
from gpu_util import f64, max_abs_rel, to_dev_bf16

pytestmark = pytest.mark.gpu


def _shapes(n, seed=20261203):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        E = int(rng.choice([1, 2, 3, 5, 8, 12, 16, 33, 64, 100]))
        k = int(rng.integers(1, min(E, 12) + 1))
        T = int(rng.integers(1, 1500))
        d = 128 * int(rng.integers(1, 7))
        f = 128 * int(rng.integers(1, 6))
        empty = E > 2 and bool(rng.integers(0, 2))
        out.append((i % 2 == 1, T, d, E, k, f, empty))
    return out


@pytest.mark.parametrize("mx,T,d,E,k,f,empty", _shapes(16),
                         ids=lambda v: str(int(v)) if isinstance(v, (bool, np.bool_)) else str(v))
def test_layer_on_random_shapes(moe_gpu, mx, T, d, E, k, f, empty):
    m, dev = moe_gpu
    inp = make_inputs(T=T, d=d, E=E, k=k, f=f, seed=T + 13 * d + E)
    if empty:
        inp["bias"][:, E // 2] -= 100.0
    L32 = O.router_logits(inp["x"], inp["w_router"], inp["bias"]).astype(np.float32)
    s = m.shape(T, d, E, k, f, prec=m.MXFP8 if mx else m.BF16)
    buf = m.allocate(s)
    t = {n: to_dev_bf16(inp[n], dev) for n in ("x", "w_gate", "w_up", "w_down", "d_out")}
    if mx:
        m.build_mx_weights(s, t["w_gate"], t["w_up"], t["w_down"], buf.mx_weights)
    buf.saved["logits"].copy_(torch.from_numpy(L32))
    out = torch.empty(T, d, dtype=torch.bfloat16, device=dev)
    m.clear_error(buf.ws)
    m.forward(buf, t["x"], None, None, t["w_gate"], t["w_up"], t["w_down"], out)
    m.backward(buf, t["d_out"], t["x"], None, t["w_gate"], t["w_up"], t["w_down"])
    assert m.read_error(buf.ws) == 0
    fwd_fn = O.layer_forward_mxfp8 if mx else O.layer_forward
    bwd_fn = O.layer_backward_mxfp8 if mx else O.layer_backward
    fwd = fwd_fn(inp["x"], None, None, inp["w_gate"], inp["w_up"], inp["w_down"], k, logits=L32)
    bwd = bwd_fn(fwd, inp["d_out"], inp["x"], None, inp["w_gate"], inp["w_up"], inp["w_down"])
    for n in ("topk_idx", "counts", "offsets", "tile_offsets", "slot_of_route"):
        np.testing.assert_array_equal(buf.saved[n].cpu().numpy(), fwd[n], err_msg=n)
    tol = 6e-2 if mx else 2e-2
    pairs = [("out", f64(out), fwd["out"]), ("dx", f64(buf.grads["dx"]), bwd["dx"]),
             ("dw_gate", f64(buf.grads["dw_gate"]), bwd["dW_gate"]),
             ("dw_up", f64(buf.grads["dw_up"]), bwd["dW_up"]),
             ("dw_down", f64(buf.grads["dw_down"]), bwd["dW_down"]),
             ("d_gates", f64(buf.grads["d_gates"]), bwd["d_gates"]),
             ("dlogits", f64(buf.grads["dlogits"]), bwd["dlogits"])]
    for name, got, ref in pairs:
        assert max_abs_rel(got, ref) <= tol, (name, max_abs_rel(got, ref))
    if empty and (fwd["counts"] == 0).any():
        e0 = np.where(fwd["counts"] == 0)[0]
        assert (f64(buf.grads["dw_gate"])[e0] == 0).all()
