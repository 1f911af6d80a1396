"""Whole-layer parity: moe_layer_fwd + moe_layer_bwd through the C ABI against
the oracle, on small shapes and on the full-size workloads (the same calls and
launch configuration the benchmark times), plus CUDA-graph capture/replay.
GPU only."""
import warnings

import numpy as np
import pytest
import torch

from oracle import cpp as O
from synth import CONFIGS, make_inputs
from gpu_util import f64, max_abs_rel, near_tie_tokens, to_dev_bf16

pytestmark = pytest.mark.gpu
TOL = 2e-2


def run_layer(m, dev, inp, k, use_router, logits32=None, backward=True):
    T, d, E, f = inp["T"], inp["d"], inp["E"], inp["f"]
    s = m.shape(T, d, E, k, f)
    buf = m.allocate(s)
    t = {n: to_dev_bf16(inp[n], dev) for n in ("x", "w_router", "w_gate", "w_up", "w_down", "d_out")}
    bias = torch.from_numpy(inp["bias"]).to(dev) if (use_router and inp["bias"] is not None) else None
    if not use_router:
        buf.saved["logits"].copy_(torch.from_numpy(logits32))
    wr = t["w_router"] if use_router else None
    out = torch.empty(T, d, dtype=torch.bfloat16, device=dev)
    m.clear_error(buf.ws)
    m.forward(buf, t["x"], wr, bias, t["w_gate"], t["w_up"], t["w_down"], out)
    if backward:
        m.backward(buf, t["d_out"], t["x"], wr, t["w_gate"], t["w_up"], t["w_down"])
    err = m.read_error(buf.ws)
    res = {"out": f64(out), "err": err}
    res.update({n: v.cpu().numpy() for n, v in buf.saved.items()
                if n in ("logits", "topk_idx", "gates", "counts", "offsets", "tile_offsets",
                         "slot_of_route", "route_of_slot")})
    if backward:
        res.update({n: f64(v) for n, v in buf.grads.items()
                    if n in ("dx", "dw_router", "dw_gate", "dw_up", "dw_down", "d_gates", "dlogits")})
    res["_call"] = (buf, t, wr, bias)
    return res


def compare_grads(g, b, use_router, rows=None):
    pairs = [("dw_gate", "dW_gate"), ("dw_up", "dW_up"), ("dw_down", "dW_down")]
    for mine, ref in pairs:
        r = max_abs_rel(g[mine], b[ref])
        assert r <= TOL, (mine, r)
    sel = slice(None) if rows is None else rows
    for mine, ref in [("dx", "dx"), ("d_gates", "d_gates"), ("dlogits", "dlogits")]:
        r = max_abs_rel(g[mine][sel], b[ref][sel])
        assert r <= TOL, (mine, r)
    if use_router:
        r = max_abs_rel(g["dw_router"], b["dW_router"])
        assert r <= TOL, ("dw_router", r)


SMALL = [(256, 128, 8, 2, 256), (300, 256, 6, 2, 384), (1000, 512, 16, 4, 256), (77, 384, 4, 4, 128),
         (1, 128, 4, 2, 128),
         # k in 5..8 and k > 8 take the wider gather kernels; 256 experts and
         # top-32 are the envelope's maxima; T = 513 is not a multiple of the
         # 128-token routing block
         (513, 256, 64, 8, 256), (200, 128, 256, 32, 128), (129, 128, 3, 3, 128)]


@pytest.mark.parametrize("T,d,E,k,f", SMALL, ids=lambda v: str(v))
def test_layer_on_shared_logits(moe_gpu, T, d, E, k, f):
    """Routing bit-exact, every floating-point output within 2e-2."""
    m, dev = moe_gpu
    inp = make_inputs(T=T, d=d, E=E, k=k, f=f, seed=3 * T + d)
    L32 = O.router_logits(inp["x"], inp["w_router"], inp["bias"]).astype(np.float32)
    g = run_layer(m, dev, inp, k, use_router=False, logits32=L32)
    assert g["err"] == 0
    fwd = O.layer_forward(inp["x"], None, None, inp["w_gate"], inp["w_up"], inp["w_down"], k,
                          logits=L32)
    bwd = O.layer_backward(fwd, inp["d_out"], inp["x"], None, inp["w_gate"], inp["w_up"],
                           inp["w_down"])
    for n in ("topk_idx", "counts", "offsets", "tile_offsets", "slot_of_route"):
        np.testing.assert_array_equal(g[n], fwd[n], err_msg=n)
    assert max_abs_rel(g["out"], fwd["out"]) <= TOL
    compare_grads(g, bwd, use_router=False)


def check_full_path(m, dev, inp, k, backward=True):
    """Router projection on the device; tokens at a near-tie of the oracle's
    logits may choose differently and are left out of the per-token checks."""
    g = run_layer(m, dev, inp, k, use_router=True, backward=backward)
    assert g["err"] == 0
    fwd = O.layer_forward(inp["x"], inp["w_router"], inp["bias"], inp["w_gate"], inp["w_up"],
                          inp["w_down"], k)
    assert max_abs_rel(g["logits"], fwd["logits"]) < 1e-5
    tol = 1e-5 * np.abs(fwd["logits"]).max()
    tie = near_tie_tokens(fwd["logits"], k, 2 * tol)
    same = (g["topk_idx"] == fwd["topk_idx"]).all(1)
    assert same[~tie].all()
    if same.all():
        for n in ("counts", "offsets", "tile_offsets", "slot_of_route"):
            np.testing.assert_array_equal(g[n], fwd[n], err_msg=n)
    else:
        # the routing metadata then differs by construction; the bit-exact
        # routing tests (shared logits) cover it
        warnings.warn(f"{int((~same).sum())} near-tie token(s) routed differently from the "
                      "oracle: counts/offsets/slots not compared, those tokens left out")
    assert max_abs_rel(g["out"][same], fwd["out"][same]) <= TOL
    g["_oracle"] = (fwd, None, same)
    if backward:
        bwd = O.layer_backward(fwd, inp["d_out"], inp["x"], inp["w_router"], inp["w_gate"],
                               inp["w_up"], inp["w_down"])
        compare_grads(g, bwd, use_router=True, rows=same)
        g["_oracle"] = (fwd, bwd, same)
    return g


def recompute_matches(m, g, use_router):
    """Backward again with recompute after overwriting every saved activation
    and gradient with NaN; the gradients must match the oracle's backward."""
    buf, t, wr, bias = g["_call"]
    fwd, bwd, rows = g["_oracle"]
    for n in ("xd", "h", "u", "a", "y"):
        buf.saved[n].fill_(float("nan"))
    for n in GRAD_NAMES:
        buf.grads[n].fill_(float("nan"))
    m.backward(buf, t["d_out"], t["x"], wr, t["w_gate"], t["w_up"], t["w_down"], recompute=True)
    assert m.read_error(buf.ws) == 0
    got = {n: f64(buf.grads[n]) for n in GRAD_NAMES}
    compare_grads(got, bwd, use_router=use_router, rows=rows)


@pytest.mark.parametrize("T,d,E,k,f", SMALL[:3] + SMALL[5:7], ids=lambda v: str(v))
def test_layer_with_router_projection(moe_gpu, T, d, E, k, f):
    m, dev = moe_gpu
    inp = make_inputs(T=T, d=d, E=E, k=k, f=f, seed=5 * T + d)
    check_full_path(m, dev, inp, k)


def test_tiny_forward_workload(moe_gpu):
    """The 256-token, d=128, 8-expert top-2 forward (routing from x.W_r alone, seed 0)."""
    m, dev = moe_gpu
    cfg = CONFIGS["tiny_fwd"]
    inp = make_inputs(cfg, seed=0)
    check_full_path(m, dev, inp, cfg.k, backward=False)


@pytest.mark.parametrize("name", ["fine_grained", "large_pool", "skewed"])
def test_full_size_workload(moe_gpu, name):
    """Full-size bf16 workloads, forward and backward, same calls as the benchmark;
    on the fine-grained workload also the backward with per-layer recompute."""
    m, dev = moe_gpu
    cfg = CONFIGS[name]
    inp = make_inputs(cfg, seed=0)
    g = check_full_path(m, dev, inp, cfg.k)
    if name == "skewed":
        assert (g["counts"] == 0).sum() >= 4
        empty = np.where(g["counts"] == 0)[0]
        assert (g["dw_gate"][empty] == 0).all() and (g["dw_down"][empty] == 0).all()
    if name == "fine_grained":
        recompute_matches(m, g, use_router=True)


@pytest.mark.parametrize("T,d,E,k,f", [(1000, 512, 16, 4, 256), (513, 256, 64, 8, 256)],
                         ids=lambda v: str(v))
def test_recompute_backward_matches_the_oracle(moe_gpu, T, d, E, k, f):
    """Per-layer recompute (the report's Section 24.3, Evidence 11): the backward
    rebuilds Xd, H, U, A, Y from x and the routing metadata; its gradients match
    the oracle's backward."""
    m, dev = moe_gpu
    inp = make_inputs(T=T, d=d, E=E, k=k, f=f, seed=23 + T)
    g = check_full_path(m, dev, inp, k)
    recompute_matches(m, g, use_router=True)


def test_two_batch_overlap_on_two_streams_matches_the_oracle(moe_gpu):
    """Two halves of the batch, each a whole layer forward + backward with its
    own buffers, run on two streams at once (the single-GPU analogue of the
    report's two-batch overlap, Section 24.2, Evidence 5): each half's out and dx
    match the oracle's whole-batch rows, and the two halves' weight gradients
    add up to the oracle's."""
    m, dev = moe_gpu
    T, d, E, k, f = 2048, 512, 16, 4, 512
    inp = make_inputs(T=T, d=d, E=E, k=k, f=f, seed=29)
    L32 = O.router_logits(inp["x"], inp["w_router"], inp["bias"]).astype(np.float32)
    fwd = O.layer_forward(inp["x"], None, None, inp["w_gate"], inp["w_up"], inp["w_down"], k,
                          logits=L32)
    bwd = O.layer_backward(fwd, inp["d_out"], inp["x"], None, inp["w_gate"], inp["w_up"],
                           inp["w_down"])
    t = {n: to_dev_bf16(inp[n], dev) for n in ("x", "w_gate", "w_up", "w_down", "d_out")}
    h = T // 2
    s2 = m.shape(h, d, E, k, f)
    bufs = [m.allocate(s2) for _ in range(2)]
    outs = [torch.empty(h, d, dtype=torch.bfloat16, device=dev) for _ in range(2)]
    streams = [torch.cuda.Stream(device=dev) for _ in range(2)]
    main = torch.cuda.current_stream()
    for i in range(2):
        bufs[i].saved["logits"].copy_(torch.from_numpy(L32[i * h:(i + 1) * h]))
        m.clear_error(bufs[i].ws)
    torch.cuda.synchronize()
    for i in range(2):
        streams[i].wait_stream(main)
        with torch.cuda.stream(streams[i]):
            sl = slice(i * h, (i + 1) * h)
            m.forward(bufs[i], t["x"][sl], None, None, t["w_gate"], t["w_up"], t["w_down"], outs[i],
                      stream=streams[i])
            m.backward(bufs[i], t["d_out"][sl], t["x"][sl], None, t["w_gate"], t["w_up"],
                       t["w_down"], stream=streams[i])
    for st in streams:
        main.wait_stream(st)
    torch.cuda.synchronize()
    for i in range(2):
        assert m.read_error(bufs[i].ws) == 0
    assert max_abs_rel(np.concatenate([f64(o) for o in outs]), fwd["out"]) <= TOL
    assert max_abs_rel(np.concatenate([f64(b.grads["dx"]) for b in bufs]), bwd["dx"]) <= TOL
    for mine, ref in [("dw_gate", "dW_gate"), ("dw_up", "dW_up"), ("dw_down", "dW_down")]:
        tot = f64(bufs[0].grads[mine]) + f64(bufs[1].grads[mine])
        assert max_abs_rel(tot, bwd[ref]) <= TOL, mine


def test_graph_capture_replays_bitwise(moe_gpu):
    """The whole fwd+bwd captures into one CUDA graph (no host sync inside) and
    replays deterministically."""
    m, dev = moe_gpu
    T, d, E, k, f = 512, 256, 8, 2, 256
    inp = make_inputs(T=T, d=d, E=E, k=k, f=f, seed=11)
    s = m.shape(T, d, E, k, f)
    buf = m.allocate(s)
    t = {n: to_dev_bf16(inp[n], dev) for n in ("x", "w_router", "w_gate", "w_up", "w_down", "d_out")}
    bias = torch.from_numpy(inp["bias"]).to(dev)
    out = torch.empty(T, d, dtype=torch.bfloat16, device=dev)

    def step():
        m.forward(buf, t["x"], t["w_router"], bias, t["w_gate"], t["w_up"], t["w_down"], out)
        m.backward(buf, t["d_out"], t["x"], t["w_router"], t["w_gate"], t["w_up"], t["w_down"])

    names = ("dx", "dw_router", "dw_gate", "dw_up", "dw_down", "d_gates", "dlogits")
    step()
    torch.cuda.synchronize()
    eager = [out.clone()] + [buf.grads[n].clone() for n in names]
    graph = torch.cuda.CUDAGraph()
    s_cap = torch.cuda.Stream()
    s_cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s_cap):
        with torch.cuda.graph(graph, stream=s_cap, capture_error_mode="global"):
            step()
    torch.cuda.current_stream().wait_stream(s_cap)
    for _ in range(3):
        out.zero_()
        for n in names:
            buf.grads[n].zero_()
        graph.replay()
        torch.cuda.synchronize()
        now = [out] + [buf.grads[n] for n in names]
        for a, b in zip(eager, now):
            assert torch.equal(a, b)
    assert m.read_error(buf.ws) == 0


GRAD_NAMES = ("dx", "dw_router", "dw_gate", "dw_up", "dw_down", "d_gates", "dlogits")


@pytest.mark.parametrize("T,d,E,k,f", [(1000, 512, 16, 4, 256), (8192, 2048, 32, 4, 1024)],
                         ids=lambda v: str(v))
def test_recompute_backward_is_bitwise_the_saved_one(moe_gpu, T, d, E, k, f):
    """moe_layer_bwd with recompute re-runs dispatch and both expert GEMMs from
    x and the routing metadata: with every saved activation overwritten by NaN
    in between, the gradients equal those of the saving backward bit for bit."""
    m, dev = moe_gpu
    inp = make_inputs(T=T, d=d, E=E, k=k, f=f, seed=17)
    s = m.shape(T, d, E, k, f)
    buf = m.allocate(s)
    t = {n: to_dev_bf16(inp[n], dev) for n in ("x", "w_router", "w_gate", "w_up", "w_down", "d_out")}
    bias = torch.from_numpy(inp["bias"]).to(dev)
    out = torch.empty(T, d, dtype=torch.bfloat16, device=dev)
    m.clear_error(buf.ws)
    m.forward(buf, t["x"], t["w_router"], bias, t["w_gate"], t["w_up"], t["w_down"], out)
    m.backward(buf, t["d_out"], t["x"], t["w_router"], t["w_gate"], t["w_up"], t["w_down"])
    saved_grads = {n: buf.grads[n].clone() for n in GRAD_NAMES}
    for n in ("xd", "h", "u", "a", "y"):
        buf.saved[n].fill_(float("nan"))
    for n in GRAD_NAMES:
        buf.grads[n].fill_(float("nan"))
    m.backward(buf, t["d_out"], t["x"], t["w_router"], t["w_gate"], t["w_up"], t["w_down"],
               recompute=True)
    assert m.read_error(buf.ws) == 0
    for n in GRAD_NAMES:
        assert torch.equal(buf.grads[n], saved_grads[n]), n
