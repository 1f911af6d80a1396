"""MXFP8 parity (GPU): the quantiser is bit-exact against the oracle (codes and
E8M0 scales, both orientations, the interleaved and transposed weight caches),
dequantisation is exact, the MXFP8 dispatch writes the oracle's codes, every
MXFP8 GEMM stage and the whole MXFP8 layer are within max-abs-rel 6e-2 of the
MXFP8 oracle, and the full-size MXFP8 workload is checked on sampled outputs."""
import numpy as np
import pytest
import torch

from oracle import cpp as O
from synth import CONFIGS, bf16_bits_from_f32, make_inputs
from gpu_util import (bf16_bits_of, f64, max_abs_rel, sf_index, sf_pack, sf_unpack,
                      to_dev_bf16)

pytestmark = pytest.mark.gpu
TOL = 6e-2


def u8(a, dev):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8)).to(dev)


def bf(a, dev):
    return to_dev_bf16(bf16_bits_from_f32(np.asarray(a, dtype=np.float32)), dev)


def q_rows(a):
    """oracle quantisation along the last axis -> (codes, row-major scales)"""
    return O.quantize_mxfp8(a)


def test_quantize_rows_bit_exact(moe_gpu):
    m, dev = moe_gpu
    rng = np.random.default_rng(0)
    vals = rng.standard_normal((2, 256, 384)).astype(np.float32) * 3
    vals[0, 0] = 0.0                                              # all-zero blocks
    vals[0, 1] = -0.0
    vals[0, 2, :32] = O.E4M3_VALUES[rng.integers(0, 126, 32)] * 8.0   # on the grid
    vals[0, 2, 0] = 448.0 * 8.0
    vals[0, 3] = rng.standard_normal(384) * 1e-30                 # tiny
    vals[0, 4] = rng.standard_normal(384) * 1e30                  # huge
    vals[1, 5, ::7] = -3.0e38
    bits = bf16_bits_from_f32(vals)
    x = to_dev_bf16(bits, dev)
    q = torch.empty(2, 256, 384, dtype=torch.uint8, device=dev)
    s = torch.empty(2 * 256 * 12, dtype=torch.uint8, device=dev)
    m.quantize_mxfp8(2, 256, 384, 1, x, q, s)
    torch.cuda.synchronize()
    codes, scales = q_rows(O.as_f64(bits))
    np.testing.assert_array_equal(q.cpu().numpy(), codes)
    sb = s.cpu().numpy().reshape(2, -1)
    for i in range(2):
        np.testing.assert_array_equal(sf_unpack(sb[i], 256, 12), scales[i])


def test_quantize_cols_writes_the_transpose(moe_gpu):
    m, dev = moe_gpu
    rng = np.random.default_rng(1)
    vals = (rng.standard_normal((3, 256, 384)) * np.exp(rng.standard_normal((3, 256, 1)))).astype(np.float32)
    bits = bf16_bits_from_f32(vals)
    q = torch.empty(3, 384, 256, dtype=torch.uint8, device=dev)
    s = torch.empty(3 * 384 * 8, dtype=torch.uint8, device=dev)
    m.quantize_mxfp8(3, 256, 384, 0, to_dev_bf16(bits, dev), q, s)
    torch.cuda.synchronize()
    sb = s.cpu().numpy().reshape(3, -1)
    for i in range(3):
        codes, scales = q_rows(O.as_f64(bits[i]).T)
        np.testing.assert_array_equal(q[i].cpu().numpy(), codes)
        np.testing.assert_array_equal(sf_unpack(sb[i], 384, 8), scales)


def oracle_caches(inp):
    """The five MXFP8 weight caches, built from the oracle's quantiser."""
    E, f, d = inp["E"], inp["f"], inp["d"]
    wg, wu, wd = (O.as_f64(inp[n]) for n in ("w_gate", "w_up", "w_down"))
    gu_q = np.zeros((E, 2 * f, d), np.uint8)
    gu_s = np.zeros((E, 2 * f, d // 32), np.uint8)
    for e in range(E):
        cg, sg = q_rows(wg[e])
        cu, su = q_rows(wu[e])
        for j in range(f // 64):
            gu_q[e, 128 * j:128 * j + 64] = cg[64 * j:64 * j + 64]
            gu_s[e, 128 * j:128 * j + 64] = sg[64 * j:64 * j + 64]
            gu_q[e, 128 * j + 64:128 * j + 128] = cu[64 * j:64 * j + 64]
            gu_s[e, 128 * j + 64:128 * j + 128] = su[64 * j:64 * j + 64]
    out = {"gu": (gu_q, gu_s)}
    out["down"] = tuple(np.stack(z) for z in zip(*[q_rows(wd[e]) for e in range(E)]))
    out["downT"] = tuple(np.stack(z) for z in zip(*[q_rows(wd[e].T) for e in range(E)]))
    out["gateT"] = tuple(np.stack(z) for z in zip(*[q_rows(wg[e].T) for e in range(E)]))
    out["upT"] = tuple(np.stack(z) for z in zip(*[q_rows(wu[e].T) for e in range(E)]))
    return out


def pack_cache(c, dev):
    res = {}
    for name, (q, s) in c.items():
        E, rows, kb = s.shape
        res[name + "_q"] = u8(q, dev)
        res[name + "_s"] = u8(np.concatenate([sf_pack(s[e]) for e in range(E)]), dev)
    return res


def test_weight_caches_bit_exact(moe_gpu):
    m, dev = moe_gpu
    inp = make_inputs(T=8, d=384, E=3, k=2, f=256, seed=21, with_grad=False)
    s = m.shape(8, 384, 3, 2, 256, prec=m.MXFP8)
    buf = m.allocate(s, with_grads=False)
    m.build_mx_weights(s, *(to_dev_bf16(inp[n], dev) for n in ("w_gate", "w_up", "w_down")),
                       buf.mx_weights)
    torch.cuda.synchronize()
    ref = oracle_caches(inp)
    for name, (q, sc) in ref.items():
        got_q = buf.mx_weights[name + "_q"].cpu().numpy()
        np.testing.assert_array_equal(got_q, q, err_msg=name)
        E, rows, kb = sc.shape
        gs = buf.mx_weights[name + "_s"].cpu().numpy().reshape(E, -1)
        for e in range(E):
            np.testing.assert_array_equal(sf_unpack(gs[e], rows, kb), sc[e], err_msg=name)


def test_dequantize_is_exact(moe_gpu):
    m, dev = moe_gpu
    rng = np.random.default_rng(2)
    a = rng.standard_normal((256, 512)) * np.exp(rng.standard_normal((256, 1)) * 3)
    codes, scales = q_rows(a)
    out = torch.empty(256, 512, dtype=torch.bfloat16, device=dev)
    m.dequantize_mxfp8(256, 512, u8(codes, dev), u8(sf_pack(scales), dev), out)
    np.testing.assert_array_equal(f64(out), O.dequantize_mxfp8(codes, scales))


# ------------------------------------------------------------------ stages
# f = 384: DGRAD2 (N = f) on the single-CTA MXFP8 kernel; d = 384: FWD2 and
# DGRAD1 (N = d) there; the other GEMMs on CTA pairs; top-12 takes the k > 8
# gathers (the combine backward's fused dY quantisation included)
SHAPES = [(300, 256, 6, 2, 256), (1000, 512, 8, 8, 384), (200, 384, 4, 2, 256),
          (160, 256, 16, 12, 256),
          # skewed: experts 5, 11 and 30 take 1492, 806 and 447 of the 4000 routes
          # (more than twice the mean), so the weight gradients, natural layout
          # included, hand their tiles out first, over several rounds of pairs
          (2000, 512, 40, 2, 512, "skew")]
SKEW_BIAS = ((5, 3.0), (11, 2.0), (30, 1.5))


@pytest.fixture(scope="module", params=SHAPES, ids=lambda v: "x".join(map(str, v)))
def mcase(request, moe_gpu):
    m, dev = moe_gpu
    T, d, E, k, f = request.param[:5]
    inp = make_inputs(T=T, d=d, E=E, k=k, f=f, seed=T + 7)
    inp["bias"][:, 2] -= 100.0                  # one empty expert
    if len(request.param) > 5:
        for e, b in SKEW_BIAS:
            inp["bias"][:, e] += b
    L32 = O.router_logits(inp["x"], inp["w_router"], inp["bias"]).astype(np.float32)
    fwd = O.layer_forward_mxfp8(inp["x"], None, None, inp["w_gate"], inp["w_up"], inp["w_down"],
                                k, logits=L32)
    bwd = O.layer_backward_mxfp8(fwd, inp["d_out"], inp["x"], None, inp["w_gate"], inp["w_up"],
                                 inp["w_down"])
    s = m.shape(T, d, E, k, f, prec=m.MXFP8)
    n = m.rows_max(s)
    used = int(fwd["row_offsets"][-1])

    def rows_q(a, width):              # oracle rows -> quantised [n, width] codes + packed scales
        full = np.zeros((n, width))
        full[:used] = a
        c, sc = q_rows(full)
        return u8(c, dev), u8(sf_pack(sc), dev)

    def rows_bf(a, width):
        full = np.zeros((n, width))
        full[:used] = a
        return bf(full, dev)

    return dict(m=m, dev=dev, T=T, d=d, E=E, k=k, f=f, s=s, n=n, used=used, inp=inp, L32=L32,
                fwd=fwd, bwd=bwd, rows_q=rows_q, rows_bf=rows_bf,
                ws=torch.zeros(m.workspace_size(s), dtype=torch.uint8, device=dev),
                cache=pack_cache(oracle_caches(inp), dev),
                tile_offsets=torch.from_numpy(fwd["tile_offsets"].astype(np.int32)).to(dev),
                counts=torch.from_numpy(fwd["counts"].astype(np.int32)).to(dev),
                slot=torch.from_numpy(fwd["slot_of_route"].astype(np.int32)).to(dev))


def test_mx_dispatch_writes_the_oracle_codes(mcase):
    c = mcase
    m, dev, n, d = c["m"], c["dev"], c["n"], c["d"]
    xq = torch.full((n, d), 0x55, dtype=torch.uint8, device=dev)
    xs = torch.full((n * d // 32,), 0x66, dtype=torch.uint8, device=dev)
    m.dispatch(c["s"], to_dev_bf16(c["inp"]["x"], dev), c["slot"], c["counts"], c["tile_offsets"],
               xq, xs)
    torch.cuda.synchronize()
    codes, scales = q_rows(O.as_f64(c["inp"]["x"]))
    used = c["used"]
    ros = c["fwd"]["route_of_slot"]
    want_q = np.zeros((used, d), np.uint8)
    want_s = np.full((used, d // 32), 127, np.uint8)
    real = ros >= 0
    want_q[real] = codes[ros[real] // c["k"]]
    want_s[real] = scales[ros[real] // c["k"]]
    np.testing.assert_array_equal(xq.cpu().numpy()[:used], want_q)
    np.testing.assert_array_equal(sf_unpack(xs.cpu().numpy(), n, d // 32)[:used], want_s)
    # with the dequantised copy: the same codes, and that copy bit for bit the dequantiser's
    xq2 = torch.full((n, d), 0x55, dtype=torch.uint8, device=dev)
    xs2 = torch.full((n * d // 32,), 0x66, dtype=torch.uint8, device=dev)
    xdq = torch.full((n, d), 7.0, dtype=torch.bfloat16, device=dev)
    m.dispatch(c["s"], to_dev_bf16(c["inp"]["x"], dev), c["slot"], c["counts"], c["tile_offsets"],
               xq2, xs2, xd_dq=xdq)
    assert torch.equal(xq2[:used], xq[:used]) and torch.equal(xs2, xs)
    ref = torch.empty(n, d, dtype=torch.bfloat16, device=dev)
    m.dequantize_mxfp8(n, d, xq2, xs2, ref)
    assert torch.equal(xdq[:used].view(torch.int16), ref[:used].view(torch.int16))


def test_mx_fwd1_swiglu(mcase):
    c = mcase
    m, dev, n, f = c["m"], c["dev"], c["n"], c["f"]
    H, U = (torch.empty(n, f, dtype=torch.bfloat16, device=dev) for _ in range(2))
    Aq = torch.empty(n, f, dtype=torch.uint8, device=dev)
    As = torch.empty(n * f // 32, dtype=torch.uint8, device=dev)
    Adq = torch.empty(n, f, dtype=torch.bfloat16, device=dev)
    xq, xs = c["rows_q"](c["fwd"]["Xd"], c["d"])
    m.grouped_gemm(c["s"], m.GEMM_FWD1_SWIGLU, c["ws"], tile_offsets=c["tile_offsets"], a0=xq,
                   sfa0=xs, w0=c["cache"]["gu_q"], sfb0=c["cache"]["gu_s"], out0=H, out1=U,
                   out2=Aq, osf0=As, out3=Adq)
    u = c["used"]
    assert m.read_error(c["ws"]) == 0
    assert max_abs_rel(f64(H)[:u], c["fwd"]["H"]) <= TOL
    assert max_abs_rel(f64(U)[:u], c["fwd"]["U"]) <= TOL
    a_deq = O.dequantize_mxfp8(Aq.cpu().numpy(), sf_unpack(As.cpu().numpy(), n, f // 32))
    assert max_abs_rel(a_deq[:u], c["fwd"]["Aq"]) <= TOL
    # the dequantised copy is bit for bit the dequantiser's
    ref = torch.empty(n, f, dtype=torch.bfloat16, device=dev)
    m.dequantize_mxfp8(n, f, Aq, As, ref)
    assert torch.equal(Adq[:u].view(torch.int16), ref[:u].view(torch.int16))


def test_mx_fwd2(mcase):
    c = mcase
    m, dev, n = c["m"], c["dev"], c["n"]
    Y = torch.empty(n, c["d"], dtype=torch.bfloat16, device=dev)
    aq, as_ = c["rows_q"](c["fwd"]["Aq"], c["f"])
    m.grouped_gemm(c["s"], m.GEMM_FWD2, c["ws"], tile_offsets=c["tile_offsets"], a0=aq, sfa0=as_,
                   w0=c["cache"]["down_q"], sfb0=c["cache"]["down_s"], out0=Y)
    assert max_abs_rel(f64(Y)[: c["used"]], c["fwd"]["Y"]) <= TOL


def test_mx_dgrad2_swiglu_bwd(mcase):
    c = mcase
    m, dev, n, f = c["m"], c["dev"], c["n"], c["f"]
    dH, dU = (torch.empty(n, f, dtype=torch.bfloat16, device=dev) for _ in range(2))
    dHq, dUq = (torch.empty(n, f, dtype=torch.uint8, device=dev) for _ in range(2))
    dHs, dUs = (torch.empty(n * f // 32, dtype=torch.uint8, device=dev) for _ in range(2))
    yq, ys = c["rows_q"](c["bwd"]["dY"], c["d"])
    m.grouped_gemm(c["s"], m.GEMM_DGRAD2_SWIGLU, c["ws"], tile_offsets=c["tile_offsets"], a0=yq,
                   sfa0=ys, w0=c["cache"]["downT_q"], sfb0=c["cache"]["downT_s"],
                   aux0=c["rows_bf"](c["fwd"]["H"], f), aux1=c["rows_bf"](c["fwd"]["U"], f),
                   out0=dH, out1=dU, out2=dHq, out3=dUq, osf0=dHs, osf1=dUs)
    u = c["used"]
    assert max_abs_rel(f64(dH)[:u], c["bwd"]["dH"]) <= TOL
    assert max_abs_rel(f64(dU)[:u], c["bwd"]["dU"]) <= TOL
    for q, sc, val, ref in ((dHq, dHs, dH, "dH"), (dUq, dUs, dU, "dU")):
        sf = sf_unpack(sc.cpu().numpy(), n, f // 32)
        dq = O.dequantize_mxfp8(q.cpu().numpy(), sf)
        assert max_abs_rel(dq[:u], c["bwd"][ref]) <= TOL, ref
        # every code sits in its own row and column: within E4M3 rounding (2^-4
        # relative, half a subnormal step 2^(s-10) absolute) of the kernel's own
        # bf16 value, plus that value's bf16 rounding (2^-8 relative)
        x = f64(val)[:u]
        step = np.repeat(np.exp2(sf[:u].astype(np.float64) - 127.0 - 10.0), 32, axis=1)
        assert np.all(np.abs(dq[:u] - x) <= (2.0 ** -4 + 2.0 ** -8) * np.abs(x) + step), ref


def test_mx_combine_bwd_quantises_dy_in_the_same_pass(mcase):
    # the fused quantisation writes byte for byte what the row quantiser gives
    # for the dy rows the same call wrote (padding rows: zero codes, scale 2^0)
    c = mcase
    m, dev, n, d, T, k, E = c["m"], c["dev"], c["n"], c["d"], c["T"], c["k"], c["E"]
    fwd = c["fwd"]
    gates = torch.from_numpy(fwd["gates"].astype(np.float32)).to(dev)
    topk = torch.from_numpy(fwd["topk_idx"].astype(np.int32)).to(dev)
    y = c["rows_bf"](fwd["Y"], d)
    dO = to_dev_bf16(c["inp"]["d_out"], dev)

    def run(quant):
        dy = torch.full((n, d), 5.0, dtype=torch.bfloat16, device=dev)
        dg = torch.empty(T, k, dtype=torch.float32, device=dev)
        dl = torch.empty(T, E, dtype=torch.float32, device=dev)
        q = torch.full((n, d), 0x55, dtype=torch.uint8, device=dev) if quant else None
        sc = torch.full((n * d // 32,), 0x66, dtype=torch.uint8, device=dev) if quant else None
        m.combine_bwd(c["s"], dO, y, gates, topk, c["slot"], c["counts"], c["tile_offsets"], dy,
                      dg, dl, dy_q=q, dy_scales=sc)
        return dy, dg, dl, q, sc

    dy, dg, dl, q, sc = run(True)
    dy0, dg0, dl0, _, _ = run(False)
    u = c["used"]
    assert torch.equal(dy[:u].view(torch.int16), dy0[:u].view(torch.int16))
    assert torch.equal(dg, dg0) and torch.equal(dl, dl0)
    rq = torch.empty(n, d, dtype=torch.uint8, device=dev)
    rs = torch.empty(n * d // 32, dtype=torch.uint8, device=dev)
    m.quantize_mxfp8(1, n, d, 1, dy, rq, rs)
    np.testing.assert_array_equal(q.cpu().numpy()[:u], rq.cpu().numpy()[:u])
    np.testing.assert_array_equal(sf_unpack(sc.cpu().numpy(), n, d // 32)[:u],
                                  sf_unpack(rs.cpu().numpy(), n, d // 32)[:u])
    assert max_abs_rel(f64(dy)[:u], c["bwd"]["dY"]) <= TOL
    with pytest.raises(m.MoEError):     # codes without scales
        m.combine_bwd(c["s"], dO, y, gates, topk, c["slot"], c["counts"], c["tile_offsets"], dy,
                      dg, dl, dy_q=q)


def test_mx_dgrad1(mcase):
    c = mcase
    m, dev, n, f = c["m"], c["dev"], c["n"], c["f"]
    dXd = torch.empty(n, c["d"], dtype=torch.bfloat16, device=dev)
    hq, hs = c["rows_q"](c["bwd"]["dH"], f)
    uq, us = c["rows_q"](c["bwd"]["dU"], f)
    m.grouped_gemm(c["s"], m.GEMM_DGRAD1, c["ws"], tile_offsets=c["tile_offsets"], a0=hq, sfa0=hs,
                   a1=uq, sfa1=us, w0=c["cache"]["gateT_q"], sfb0=c["cache"]["gateT_s"],
                   w1=c["cache"]["upT_q"], sfb1=c["cache"]["upT_s"], out0=dXd)
    assert max_abs_rel(f64(dXd)[: c["used"]], c["bwd"]["dXd"]) <= TOL


def run_mx_layer(m, dev, inp, k, L32, backward=True):
    T, d, E, f = inp["T"], inp["d"], inp["E"], inp["f"]
    s = m.shape(T, d, E, k, f, prec=m.MXFP8)
    buf = m.allocate(s, with_grads=backward)
    t = {nm: to_dev_bf16(inp[nm], dev) for nm in ("x", "w_gate", "w_up", "w_down", "d_out")}
    m.build_mx_weights(s, t["w_gate"], t["w_up"], t["w_down"], buf.mx_weights)
    buf.saved["logits"].copy_(torch.from_numpy(L32))
    out = torch.empty(T, d, dtype=torch.bfloat16, device=dev)
    m.clear_error(buf.ws)
    m.forward(buf, t["x"], None, None, t["w_gate"], t["w_up"], t["w_down"], out)
    if backward:
        m.backward(buf, t["d_out"], t["x"], None, t["w_gate"], t["w_up"], t["w_down"])
    return buf, out, m.read_error(buf.ws)


def test_mx_layer_small(mcase):
    c = mcase
    m, dev = c["m"], c["dev"]
    buf, out, err = run_mx_layer(m, dev, c["inp"], c["k"], c["L32"])
    assert err == 0
    f, b = c["fwd"], c["bwd"]
    for nm in ("topk_idx", "counts", "offsets", "tile_offsets", "slot_of_route"):
        np.testing.assert_array_equal(buf.saved[nm].cpu().numpy(), f[nm], err_msg=nm)
    assert max_abs_rel(f64(out), f["out"]) <= TOL
    g = buf.grads
    for mine, ref in [("dx", "dx"), ("dw_gate", "dW_gate"), ("dw_up", "dW_up"),
                      ("dw_down", "dW_down"), ("d_gates", "d_gates"), ("dlogits", "dlogits")]:
        r = max_abs_rel(f64(g[mine]), b[ref])
        assert r <= TOL, (mine, r)
    empty = np.where(f["counts"] == 0)[0]
    assert (f64(g["dw_gate"])[empty] == 0).all() and (f64(g["dw_down"])[empty] == 0).all()


def test_mx_full_size_workload_sampled(moe_gpu):
    """32768 tokens, d=4096, 64 experts, top-8, f=2048 (the benchmark's workload
    and launch configuration): routing and the dispatched codes in full; eight
    experts in full (H and Y rows, dXd rows and all three weight gradients) and
    the out, dx and d_gates rows of 256 seeded tokens against the C++ oracle's
    MXFP8 layer; the natural-layout weight gradients bit for bit against the
    layer's."""
    m, dev = moe_gpu
    cfg = CONFIGS["mxfp8"]
    k, E = cfg.k, cfg.E
    inp = make_inputs(cfg, seed=0)
    L32 = O.router_logits(inp["x"], inp["w_router"], inp["bias"]).astype(np.float32)
    buf, out, err = run_mx_layer(m, dev, inp, k, L32)
    assert err == 0
    idx, gates = O.softmax_topk_gates(L32, k)
    counts = O.expert_counts(idx, E)
    tile_offsets, row_offsets = O.tile_layout(counts, 128)
    sor, ros = O.assign_slots(idx, row_offsets)
    np.testing.assert_array_equal(buf.saved["topk_idx"].cpu().numpy(), idx)
    np.testing.assert_array_equal(buf.saved["slot_of_route"].cpu().numpy(), sor)
    n = buf.rows_max
    xq_all = buf.mx["xd_q"].cpu().numpy()
    xs_all = sf_unpack(buf.mx["xd_s"].cpu().numpy(), n, cfg.d // 32)
    codes, scales = q_rows(O.as_f64(inp["x"]))
    real = ros >= 0
    np.testing.assert_array_equal(xq_all[: len(ros)][real], codes[ros[real] // k])
    np.testing.assert_array_equal(xs_all[: len(ros)][real], scales[ros[real] // k])
    xq = O.dequantize_mxfp8(codes, scales)          # the quantised tokens, [T, d]
    del xq_all, xs_all, codes, scales
    dO = O.as_f64(inp["d_out"])
    g = buf.grads
    rng = np.random.default_rng(0)
    # ---- eight experts in full
    big, small = int(np.argmax(counts)), int(np.argmin(counts))
    others = [int(e) for e in rng.permutation(E) if e not in (big, small)][:6]
    for e in [big, small] + others:
        a, c = int(row_offsets[e]), int(counts[e])
        routes = ros[a:a + c]
        tok = routes // k
        ro1 = np.array([0, c])
        w = [inp[nm][e:e + 1] for nm in ("w_gate", "w_up", "w_down")]
        H, U, A, Aq, Y = O.expert_ffn_forward_mxfp8(xq[tok], *w, ro1)
        assert max_abs_rel(f64(buf.saved["h"][a:a + c]), H) <= TOL, ("H", e)
        assert max_abs_rel(f64(buf.saved["u"][a:a + c]), U) <= TOL, ("U", e)
        assert max_abs_rel(f64(buf.saved["y"][a:a + c]), Y) <= TOL, ("Y", e)
        dY = gates.reshape(-1)[routes][:, None] * dO[tok]
        gb = O.expert_ffn_backward_mxfp8(dY, xq[tok], H, U, Aq, *w, ro1)
        assert max_abs_rel(f64(g["dxd"][a:a + c]), gb["dXd"]) <= TOL, ("dXd", e)
        for mine, ref in (("dw_gate", "dW_gate"), ("dw_up", "dW_up"), ("dw_down", "dW_down")):
            assert max_abs_rel(f64(g[mine][e]), gb[ref][0]) <= TOL, (mine, e)
    # ---- out, dx and d_gates of 256 seeded tokens, through all their experts
    ts = np.sort(rng.choice(cfg.T, 256, replace=False))
    idx_s, g_s = idx[ts], gates[ts]
    _, ro_s = O.tile_layout(O.expert_counts(idx_s, E), 1)
    sor_s, _ = O.assign_slots(idx_s, ro_s)
    rows_s = int(ro_s[-1])
    Xd_s = O.dispatch(xq[ts], sor_s, k, rows_s)
    H, U, A, Aq, Y = O.expert_ffn_forward_mxfp8(Xd_s, inp["w_gate"], inp["w_up"], inp["w_down"], ro_s)
    assert max_abs_rel(f64(out)[ts], O.combine(Y, g_s, sor_s, 256, k)) <= TOL
    dg, dY = O.combine_backward(dO[ts], Y, g_s, sor_s, 256, k, rows_s)
    assert max_abs_rel(f64(g["d_gates"])[ts], dg) <= TOL
    gb = O.expert_ffn_backward_mxfp8(dY, Xd_s, H, U, Aq, inp["w_gate"], inp["w_up"], inp["w_down"],
                                     ro_s)
    assert max_abs_rel(f64(g["dx"])[ts], O.dispatch_backward(gb["dXd"], sor_s, 256, k)) <= TOL
    # the natural-layout weight gradients on the layer's own codes and scales
    # equal, bit for bit, the layer's (global dequantisation + BF16) ones
    s = m.shape(cfg.T, cfg.d, cfg.E, cfg.k, cfg.f, prec=m.MXFP8)
    to = buf.saved["tile_offsets"]
    dWd = torch.empty_like(g["dw_down"])
    m.grouped_gemm(s, m.GEMM_WGRAD2_NATURAL, buf.ws, tile_offsets=to, a0=g["dy"],
                   a1=buf.mx["a_q"], sfb0=buf.mx["a_s"], out0=dWd)
    dWg, dWu = torch.empty_like(g["dw_gate"]), torch.empty_like(g["dw_up"])
    m.grouped_gemm(s, m.GEMM_WGRAD1_NATURAL, buf.ws, tile_offsets=to, a0=g["dh"], a1=g["du"],
                   aux0=buf.mx["xd_q"], sfb0=buf.mx["xd_s"], out0=dWg, out1=dWu)
    assert m.read_error(buf.ws) == 0
    assert torch.equal(dWd, g["dw_down"])
    assert torch.equal(dWg, g["dw_gate"]) and torch.equal(dWu, g["dw_up"])


def test_mx_recompute_backward_matches_the_oracle(mcase):
    """MXFP8 backward with recompute (saved activations overwritten with NaN
    first) against the C++ oracle's MXFP8 backward."""
    c = mcase
    m, dev = c["m"], c["dev"]
    buf, out, err = run_mx_layer(m, dev, c["inp"], c["k"], c["L32"])
    assert err == 0
    for n in ("h", "u", "y"):
        buf.saved[n].fill_(float("nan"))
    for n in ("xd_q", "a_q"):
        buf.mx[n].fill_(0x7F)
    for n in ("dx", "dw_gate", "dw_up", "dw_down", "d_gates", "dlogits"):
        buf.grads[n].fill_(float("nan"))
    t = {nm: to_dev_bf16(c["inp"][nm], dev) for nm in ("x", "w_gate", "w_up", "w_down", "d_out")}
    m.backward(buf, t["d_out"], t["x"], None, t["w_gate"], t["w_up"], t["w_down"], recompute=True)
    assert m.read_error(buf.ws) == 0
    b = c["bwd"]
    for mine, ref in [("dx", "dx"), ("dw_gate", "dW_gate"), ("dw_up", "dW_up"),
                      ("dw_down", "dW_down"), ("d_gates", "d_gates"), ("dlogits", "dlogits")]:
        assert max_abs_rel(f64(buf.grads[mine]), b[ref]) <= TOL, mine


def test_mx_graph_capture_replays_bitwise(mcase):
    """Weight caches + MXFP8 forward + backward capture into one CUDA graph (no
    host sync inside), replay bit for bit, and match the MXFP8 oracle."""
    c = mcase
    m, dev = c["m"], c["dev"]
    T, d, E, k, f = c["T"], c["d"], c["E"], c["k"], c["f"]
    s = c["s"]
    buf = m.allocate(s)
    t = {nm: to_dev_bf16(c["inp"][nm], dev) for nm in ("x", "w_gate", "w_up", "w_down", "d_out")}
    buf.saved["logits"].copy_(torch.from_numpy(c["L32"]))
    out = torch.empty(T, d, dtype=torch.bfloat16, device=dev)
    names = ("dx", "dw_gate", "dw_up", "dw_down", "d_gates", "dlogits")

    def step():
        m.build_mx_weights(s, t["w_gate"], t["w_up"], t["w_down"], buf.mx_weights)
        m.forward(buf, t["x"], None, None, t["w_gate"], t["w_up"], t["w_down"], out)
        m.backward(buf, t["d_out"], t["x"], None, t["w_gate"], t["w_up"], t["w_down"])

    m.clear_error(buf.ws)
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
        for a, b in zip(eager, [out] + [buf.grads[n] for n in names]):
            assert torch.equal(a, b)
    assert m.read_error(buf.ws) == 0
    assert max_abs_rel(f64(out), c["fwd"]["out"]) <= TOL
    assert max_abs_rel(f64(buf.grads["dx"]), c["bwd"]["dx"]) <= TOL
    assert max_abs_rel(f64(buf.grads["dw_gate"]), c["bwd"]["dW_gate"]) <= TOL


def test_mx_recompute_backward_is_bitwise_the_saved_one(mcase):
    """MXFP8 recompute: the quantised Xd and A and the bf16 H, U, Y are rebuilt
    from x; with them overwritten in between, the gradients are bit for bit
    those of the saving backward."""
    c = mcase
    m, dev = c["m"], c["dev"]
    buf, out, err = run_mx_layer(m, dev, c["inp"], c["k"], c["L32"])
    assert err == 0
    names = ("dx", "dw_gate", "dw_up", "dw_down", "d_gates", "dlogits")
    saved_grads = {n: buf.grads[n].clone() for n in names}
    for n in ("h", "u", "y"):
        buf.saved[n].fill_(float("nan"))
    for n in ("xd_q", "a_q"):
        buf.mx[n].fill_(0x7F)          # E4M3 NaN codes
    for n in ("xd_s", "a_s"):
        buf.mx[n].fill_(0xFF)          # E8M0 NaN scale
    for n in names:
        buf.grads[n].fill_(float("nan"))
    t = {nm: to_dev_bf16(c["inp"][nm], dev) for nm in ("x", "w_gate", "w_up", "w_down", "d_out")}
    m.backward(buf, t["d_out"], t["x"], None, t["w_gate"], t["w_up"], t["w_down"], recompute=True)
    assert m.read_error(buf.ws) == 0
    for n in names:
        assert torch.equal(buf.grads[n], saved_grads[n]), n


# ------------------------------------------------ weight gradients, natural layout
def natural_wgrads(m, s, ws, tile_offsets, dY, A_q, A_s, dH, dU, Xd_q, Xd_s, n, d, f, E):
    """(dW_down, dW_gate, dW_up) from the natural-layout ops, and the same from
    the global dequantisation followed by the BF16 weight-gradient GEMMs."""
    dev = dY.device
    out = {}
    for arm in ("natural", "dq_bf16"):
        dWd = torch.full((E, d, f), float("nan"), dtype=torch.float32, device=dev)
        dWg, dWu = (torch.full((E, f, d), float("nan"), dtype=torch.float32, device=dev)
                    for _ in range(2))
        if arm == "natural":
            if f % 256 == 0:
                m.grouped_gemm(s, m.GEMM_WGRAD2_NATURAL, ws, tile_offsets=tile_offsets, a0=dY,
                               a1=A_q, sfb0=A_s, out0=dWd)
            m.grouped_gemm(s, m.GEMM_WGRAD1_NATURAL, ws, tile_offsets=tile_offsets, a0=dH, a1=dU,
                           aux0=Xd_q, sfb0=Xd_s, out0=dWg, out1=dWu)
        else:
            a_dq = torch.empty(n, f, dtype=torch.bfloat16, device=dev)
            x_dq = torch.empty(n, d, dtype=torch.bfloat16, device=dev)
            m.dequantize_mxfp8(n, f, A_q, A_s, a_dq)
            m.dequantize_mxfp8(n, d, Xd_q, Xd_s, x_dq)
            m.grouped_gemm(s, m.GEMM_WGRAD2, ws, tile_offsets=tile_offsets, a0=dY, a1=a_dq,
                           out0=dWd)
            m.grouped_gemm(s, m.GEMM_WGRAD1, ws, tile_offsets=tile_offsets, a0=dH, a1=dU,
                           aux0=x_dq, out0=dWg, out1=dWu)
        out[arm] = (dWd, dWg, dWu)
    return out


def test_natural_wgrad_is_bitwise_the_dequantised_one(mcase):
    """The weight gradients on the forward's MXFP8 codes (dequantised inside the
    GEMM) equal, bit for bit, global dequantisation + BF16 GEMM, and match the
    MXFP8 oracle; an expert without rows gets exact zeros."""
    c = mcase
    m, dev, n, d, f, E = c["m"], c["dev"], c["n"], c["d"], c["f"], c["E"]
    if d % 256:
        pytest.skip("the natural-layout weight gradients take d a multiple of 256 "
                    "(test_natural_wgrad_refuses_unsupported_shapes covers the refusal)")
    aq, as_ = c["rows_q"](c["fwd"]["Aq"], f)
    xq, xs = c["rows_q"](c["fwd"]["Xd"], d)
    dY = c["rows_bf"](c["bwd"]["dY"], d)
    dH = c["rows_bf"](c["bwd"]["dH"], f)
    dU = c["rows_bf"](c["bwd"]["dU"], f)
    got = natural_wgrads(m, c["s"], c["ws"], c["tile_offsets"], dY, aq, as_, dH, dU, xq, xs, n, d,
                         f, E)
    assert m.read_error(c["ws"]) == 0
    nat, ref = got["natural"], got["dq_bf16"]
    if f % 256 == 0:
        assert torch.equal(nat[0], ref[0])
        assert max_abs_rel(f64(nat[0]), c["bwd"]["dW_down"]) <= TOL
    assert torch.equal(nat[1], ref[1]) and torch.equal(nat[2], ref[2])
    assert max_abs_rel(f64(nat[1]), c["bwd"]["dW_gate"]) <= TOL
    assert max_abs_rel(f64(nat[2]), c["bwd"]["dW_up"]) <= TOL
    empty = np.where(c["fwd"]["counts"] == 0)[0]   # none when top-k selects every expert
    assert (f64(nat[1])[empty] == 0).all() and (f64(nat[2])[empty] == 0).all()


def test_natural_wgrad_refuses_unsupported_shapes(mcase):
    c = mcase
    m, dev, n, d, f, E = c["m"], c["dev"], c["n"], c["d"], c["f"], c["E"]
    if f % 256 == 0 and d % 256 == 0:
        pytest.skip("both natural ops support this shape")
    aq, as_ = c["rows_q"](c["fwd"]["Aq"], f)
    dW = torch.empty(E, d, f, dtype=torch.float32, device=dev)
    with pytest.raises(m.MoEError):
        m.grouped_gemm(c["s"], m.GEMM_WGRAD2_NATURAL, c["ws"], tile_offsets=c["tile_offsets"],
                       a0=c["rows_bf"](c["bwd"]["dY"], d), a1=aq, sfb0=as_, out0=dW)
    with pytest.raises(m.MoEError):   # scales missing
        m.grouped_gemm(c["s"], m.GEMM_WGRAD1_NATURAL, c["ws"], tile_offsets=c["tile_offsets"],
                       a0=dW, a1=dW, aux0=aq, out0=dW, out1=dW)
    assert m.read_error(c["ws"]) == 0


@pytest.mark.parametrize("T,d,E,k,f", [(4096, 512, 8, 4, 512), (3000, 768, 5, 2, 256)],
                         ids=lambda v: str(v))
def test_natural_wgrad_long_k(moe_gpu, T, d, E, k, f):
    """Many K steps per expert (the ring and both B slots wrap many times) and a
    ragged last tile: still bit for bit the dequantised BF16 result."""
    m, dev = moe_gpu
    rng = np.random.default_rng(T)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    counts = O.expert_counts(idx, E)
    tile_offsets, row_offsets = O.tile_layout(counts, 128)
    s = m.shape(T, d, E, k, f, prec=m.MXFP8)
    n = m.rows_max(s)
    used = int(row_offsets[-1])
    ws = torch.zeros(m.workspace_size(s), dtype=torch.uint8, device=dev)

    def qrows(width, scale):
        a = np.zeros((n, width))
        a[:used] = rng.standard_normal((used, width)) * scale
        # zero rows between each expert's count and its tile boundary
        for e in range(E):
            a[int(row_offsets[e]) + int(counts[e]): int(tile_offsets[e + 1]) * 128] = 0.0
        codes, sc = q_rows(a)
        return a, u8(codes, dev), u8(sf_pack(sc), dev)

    def brows(width):
        a = np.zeros((n, width))
        a[:used] = rng.standard_normal((used, width))
        for e in range(E):
            a[int(row_offsets[e]) + int(counts[e]): int(tile_offsets[e + 1]) * 128] = 0.0
        return bf(a, dev)

    _, aq, as_ = qrows(f, 0.5)
    _, xq, xs = qrows(d, np.exp(rng.standard_normal((1, d))))
    dY, dH, dU = brows(d), brows(f), brows(f)
    to = torch.from_numpy(tile_offsets.astype(np.int32)).to(dev)
    got = natural_wgrads(m, s, ws, to, dY, aq, as_, dH, dU, xq, xs, n, d, f, E)
    assert m.read_error(ws) == 0
    for a, b in zip(got["natural"], got["dq_bf16"]):
        assert torch.equal(a, b)
    assert torch.isfinite(got["natural"][1]).all()
