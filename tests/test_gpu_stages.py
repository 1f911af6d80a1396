"""Parity of every stage call (dispatch, grouped GEMMs, combine and the backward
stages) with the oracle.  Each stage gets the oracle's own intermediate results
as its inputs (rounded to the device storage type), so a failure points at one
kernel.  Floating-point outputs: max-abs-rel <= 2e-2 (bf16 tolerance of the
layer); index and copy outputs: bit-exact.  GPU only."""
import numpy as np
import pytest
import torch

from oracle import cpp as O
from synth import bf16_bits_from_f32, make_inputs
from gpu_util import bf16_bits_of, f64, max_abs_rel, to_dev_bf16

pytestmark = pytest.mark.gpu
TOL = 2e-2

SHAPES = [
    # T, d, E, k, f   (f = 384: N tiles of 128 in the f-wide GEMMs; expert 2 empty)
    (300, 256, 6, 2, 384),
    (1000, 512, 8, 4, 256),
    (129, 128, 3, 1, 128),
    (500, 256, 16, 8, 256),    # k = 8: the wider gather kernels
    # skewed: experts 5, 11 and 30 get 1446, 687 and 409 of the 4000 routes (more
    # than twice the mean), the weight gradients hand their tiles out first, and
    # 640 / 320 pair tiles run several rounds over the CTA pairs
    (2000, 1024, 40, 2, 512, "skew"),
]
SKEW_BIAS = ((5, 3.0), (11, 2.0), (30, 1.5))


def bf(a, dev):
    """fp64/fp32 numpy -> bf16 device tensor (round to nearest even)."""
    return to_dev_bf16(bf16_bits_from_f32(np.asarray(a, dtype=np.float32)), dev)


def i32(a, dev):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)


def f32(a, dev):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev)


@pytest.fixture(scope="module", params=SHAPES, ids=lambda s: "x".join(map(str, s)))
def case(request, moe_gpu):
    m, dev = moe_gpu
    T, d, E, k, f = request.param[:5]
    inp = make_inputs(T=T, d=d, E=E, k=k, f=f, seed=T + E)
    inp["bias"][:, min(2, E - 1) if E > 2 else 0] -= (100.0 if E > 2 else 0.0)
    if len(request.param) > 5:
        for e, b in SKEW_BIAS:
            inp["bias"][:, e] += b
    L32 = O.router_logits(inp["x"], inp["w_router"], inp["bias"]).astype(np.float32)
    fwd = O.layer_forward(inp["x"], inp["w_router"], None, inp["w_gate"], inp["w_up"],
                          inp["w_down"], k, logits=L32)
    bwd = O.layer_backward(fwd, inp["d_out"], inp["x"], inp["w_router"], inp["w_gate"],
                           inp["w_up"], inp["w_down"])
    s = m.shape(T, d, E, k, f)
    n = m.rows_max(s)
    used = int(fwd["row_offsets"][-1])
    ws = torch.zeros(m.workspace_size(s), dtype=torch.uint8, device=dev)

    def rows(a, width):          # oracle row buffer -> bf16 [n, width] device tensor
        full = np.zeros((n, width))
        full[:used] = a
        return bf(full, dev)

    return dict(m=m, dev=dev, T=T, d=d, E=E, k=k, f=f, s=s, n=n, used=used, ws=ws, inp=inp,
                fwd=fwd, bwd=bwd, rows=rows,
                to=lambda key: to_dev_bf16(inp[key], dev),
                tile_offsets=i32(fwd["tile_offsets"], dev), counts=i32(fwd["counts"], dev),
                slot=i32(fwd["slot_of_route"], dev), topk=i32(fwd["topk_idx"], dev),
                gates=f32(fwd["gates"], dev))


def test_dispatch_is_an_exact_row_copy(case):
    c = case
    m, dev = c["m"], c["dev"]
    xd = torch.full((c["n"], c["d"]), 3.0, dtype=torch.bfloat16, device=dev)  # garbage
    m.dispatch(c["s"], c["to"]("x"), c["slot"], c["counts"], c["tile_offsets"], xd)
    got = bf16_bits_of(xd)[: c["used"]]
    want = bf16_bits_from_f32(c["fwd"]["Xd"].astype(np.float32))
    np.testing.assert_array_equal(got, want)


def test_fwd1_swiglu(case):
    c = case
    m, dev, n, f = c["m"], c["dev"], c["n"], c["f"]
    H, U, A = (torch.empty(n, f, dtype=torch.bfloat16, device=dev) for _ in range(3))
    m.grouped_gemm(c["s"], m.GEMM_FWD1_SWIGLU, c["ws"], tile_offsets=c["tile_offsets"],
                   a0=c["rows"](c["fwd"]["Xd"], c["d"]), w0=c["to"]("w_gate"), w1=c["to"]("w_up"),
                   out0=H, out1=U, out2=A)
    u = c["used"]
    for name, t in (("H", H), ("U", U), ("A", A)):
        r = max_abs_rel(f64(t)[:u], c["fwd"][name])
        assert r <= TOL, (name, r)
    assert m.read_error(c["ws"]) == 0


def test_fwd2(case):
    c = case
    m, dev, n = c["m"], c["dev"], c["n"]
    Y = torch.empty(n, c["d"], dtype=torch.bfloat16, device=dev)
    m.grouped_gemm(c["s"], m.GEMM_FWD2, c["ws"], tile_offsets=c["tile_offsets"],
                   a0=c["rows"](c["fwd"]["A"], c["f"]), w0=c["to"]("w_down"), out0=Y)
    assert max_abs_rel(f64(Y)[: c["used"]], c["fwd"]["Y"]) <= TOL


def test_combine(case):
    c = case
    m, dev = c["m"], c["dev"]
    out = torch.empty(c["T"], c["d"], dtype=torch.bfloat16, device=dev)
    m.combine(c["s"], c["rows"](c["fwd"]["Y"], c["d"]), c["gates"], c["slot"], out)
    assert max_abs_rel(f64(out), c["fwd"]["out"]) <= TOL


def test_combine_bwd(case):
    c = case
    m, dev, n = c["m"], c["dev"], c["n"]
    dy = torch.full((n, c["d"]), 5.0, dtype=torch.bfloat16, device=dev)
    dg = torch.empty(c["T"], c["k"], dtype=torch.float32, device=dev)
    dl = torch.empty(c["T"], c["E"], dtype=torch.float32, device=dev)
    m.combine_bwd(c["s"], c["to"]("d_out"), c["rows"](c["fwd"]["Y"], c["d"]), c["gates"], c["topk"],
                  c["slot"], c["counts"], c["tile_offsets"], dy, dg, dl)
    b = c["bwd"]
    assert max_abs_rel(f64(dy)[: c["used"]], b["dY"]) <= TOL
    assert max_abs_rel(f64(dg), b["d_gates"]) <= TOL
    assert max_abs_rel(f64(dl), b["dlogits"]) <= TOL
    assert (f64(dl)[b["dlogits"] == 0] == 0).all()


def test_dgrad2_swiglu_bwd(case):
    c = case
    m, dev, n, f = c["m"], c["dev"], c["n"], c["f"]
    dH, dU = (torch.empty(n, f, dtype=torch.bfloat16, device=dev) for _ in range(2))
    m.grouped_gemm(c["s"], m.GEMM_DGRAD2_SWIGLU, c["ws"], tile_offsets=c["tile_offsets"],
                   a0=c["rows"](c["bwd"]["dY"], c["d"]), w0=c["to"]("w_down"),
                   aux0=c["rows"](c["fwd"]["H"], f), aux1=c["rows"](c["fwd"]["U"], f), out0=dH, out1=dU)
    u = c["used"]
    assert max_abs_rel(f64(dH)[:u], c["bwd"]["dH"]) <= TOL
    assert max_abs_rel(f64(dU)[:u], c["bwd"]["dU"]) <= TOL


def test_wgrad2(case):
    c = case
    m, dev = c["m"], c["dev"]
    dW = torch.full((c["E"], c["d"], c["f"]), 7.0, dtype=torch.float32, device=dev)
    m.grouped_gemm(c["s"], m.GEMM_WGRAD2, c["ws"], tile_offsets=c["tile_offsets"],
                   a0=c["rows"](c["bwd"]["dY"], c["d"]), a1=c["rows"](c["fwd"]["A"], c["f"]), out0=dW)
    got = f64(dW)
    assert max_abs_rel(got, c["bwd"]["dW_down"]) <= TOL
    empty = np.where(c["fwd"]["counts"] == 0)[0]
    assert (got[empty] == 0).all()


def test_dgrad1(case):
    c = case
    m, dev, n, f = c["m"], c["dev"], c["n"], c["f"]
    dXd = torch.empty(n, c["d"], dtype=torch.bfloat16, device=dev)
    m.grouped_gemm(c["s"], m.GEMM_DGRAD1, c["ws"], tile_offsets=c["tile_offsets"],
                   a0=c["rows"](c["bwd"]["dH"], f), a1=c["rows"](c["bwd"]["dU"], f),
                   w0=c["to"]("w_gate"), w1=c["to"]("w_up"), out0=dXd)
    assert max_abs_rel(f64(dXd)[: c["used"]], c["bwd"]["dXd"]) <= TOL


def test_wgrad1(case):
    c = case
    m, dev, f = c["m"], c["dev"], c["f"]
    dWg = torch.full((c["E"], f, c["d"]), 7.0, dtype=torch.float32, device=dev)
    dWu = torch.full((c["E"], f, c["d"]), 7.0, dtype=torch.float32, device=dev)
    m.grouped_gemm(c["s"], m.GEMM_WGRAD1, c["ws"], tile_offsets=c["tile_offsets"],
                   a0=c["rows"](c["bwd"]["dH"], f), a1=c["rows"](c["bwd"]["dU"], f),
                   aux0=c["rows"](c["fwd"]["Xd"], c["d"]), out0=dWg, out1=dWu)
    assert max_abs_rel(f64(dWg), c["bwd"]["dW_gate"]) <= TOL
    assert max_abs_rel(f64(dWu), c["bwd"]["dW_up"]) <= TOL
    empty = np.where(c["fwd"]["counts"] == 0)[0]
    assert (f64(dWg)[empty] == 0).all() and (f64(dWu)[empty] == 0).all()


def test_dispatch_bwd_with_router_term(case):
    c = case
    m, dev = c["m"], c["dev"]
    dx = torch.empty(c["T"], c["d"], dtype=torch.bfloat16, device=dev)
    m.dispatch_bwd(c["s"], c["rows"](c["bwd"]["dXd"], c["d"]), c["slot"], c["topk"],
                   f32(c["bwd"]["dlogits"], dev), c["to"]("w_router"), dx)
    assert max_abs_rel(f64(dx), c["bwd"]["dx"]) <= TOL


def test_router_bwd(case):
    c = case
    m, dev = c["m"], c["dev"]
    dW = torch.full((c["E"], c["d"]), 9.0, dtype=torch.float32, device=dev)
    ros = np.full(c["n"], -1, dtype=np.int32)
    ros[: c["used"]] = c["fwd"]["route_of_slot"]
    m.router_bwd(c["s"], c["to"]("x"), f32(c["bwd"]["dlogits"], dev), i32(ros, dev), c["counts"],
                 c["tile_offsets"], dW, c["ws"])
    got = f64(dW)
    assert max_abs_rel(got, c["bwd"]["dW_router"]) <= 1e-4
    empty = np.where(c["fwd"]["counts"] == 0)[0]
    assert (got[empty] == 0).all()


def test_profile_hook_times_each_launch(case):
    """moe_profile_start/stop record one event pair per launch of the chosen GEMM only."""
    c = case
    m, dev, n = c["m"], c["dev"], c["n"]
    Y = torch.empty(n, c["d"], dtype=torch.bfloat16, device=dev)
    a0 = c["rows"](c["fwd"]["A"], c["f"])
    w0 = c["to"]("w_down")
    m.profile_start(m.GEMM_FWD2)
    for _ in range(3):
        m.grouped_gemm(c["s"], m.GEMM_FWD2, c["ws"], tile_offsets=c["tile_offsets"], a0=a0, w0=w0,
                       out0=Y)
    dXd = torch.empty(n, c["d"], dtype=torch.bfloat16, device=dev)   # another op: not timed
    m.grouped_gemm(c["s"], m.GEMM_DGRAD1, c["ws"], tile_offsets=c["tile_offsets"],
                   a0=c["rows"](c["bwd"]["dH"], c["f"]), a1=c["rows"](c["bwd"]["dU"], c["f"]),
                   w0=c["to"]("w_gate"), w1=c["to"]("w_up"), out0=dXd)
    ms, launches = m.profile_stop()
    assert launches == 3 and ms > 0.0
    ms2, launches2 = m.profile_stop()          # stopped: nothing more recorded
    assert launches2 == 0 and ms2 == 0.0
    assert max_abs_rel(f64(Y)[: c["used"]], c["fwd"]["Y"]) <= TOL
