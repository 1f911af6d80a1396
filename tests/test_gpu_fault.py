"""Failure detection without a GPU fault: a host-set test hook makes the grouped
GEMM's producer issue nothing, so the MMA issuer's bounded mbarrier wait runs
out (about one second).  The kernel must report MOE_DEVERR_TIMEOUT through the
error word, free its tensor memory and return, and the context must stay usable:
the same GEMM run again afterwards gives the oracle's result.  GPU only."""
import numpy as np
import pytest
import torch

from oracle import cpp as O
from synth import bf16_bits_from_f32, make_inputs
from gpu_util import f64, max_abs_rel, to_dev_bf16

pytestmark = pytest.mark.gpu


def test_stalled_gemm_times_out_and_context_survives(moe_gpu):
    m, dev = moe_gpu
    T, d, E, k, f = 300, 256, 4, 2, 256
    inp = make_inputs(T=T, d=d, E=E, k=k, f=f, seed=77)
    L32 = O.router_logits(inp["x"], inp["w_router"], inp["bias"]).astype(np.float32)
    fwd = O.layer_forward(inp["x"], None, None, inp["w_gate"], inp["w_up"], inp["w_down"], k,
                          logits=L32)
    s = m.shape(T, d, E, k, f)
    n = m.rows_max(s)
    used = int(fwd["row_offsets"][-1])
    ws = torch.zeros(m.workspace_size(s), dtype=torch.uint8, device=dev)
    xd = np.zeros((n, d), dtype=np.float32)
    xd[:used] = fwd["Xd"]
    xd_t = to_dev_bf16(bf16_bits_from_f32(xd), dev)
    tile_offsets = torch.from_numpy(fwd["tile_offsets"].astype(np.int32)).to(dev)
    H, U, A = (torch.zeros(n, f, dtype=torch.bfloat16, device=dev) for _ in range(3))

    def run():
        m.grouped_gemm(s, m.GEMM_FWD1_SWIGLU, ws, tile_offsets=tile_offsets, a0=xd_t,
                       w0=to_dev_bf16(inp["w_gate"], dev), w1=to_dev_bf16(inp["w_up"], dev),
                       out0=H, out1=U, out2=A)

    prev = m.debug_inject_stall(1)
    try:
        m.clear_error(ws)
        run()
        err = m.read_error(ws)              # synchronises: the kernel has returned
    finally:
        m.debug_inject_stall(prev)
    assert err & m.DEVERR_TIMEOUT
    # the context is still usable and the kernel is correct again
    m.clear_error(ws)
    run()
    assert m.read_error(ws) == 0
    assert max_abs_rel(f64(H)[:used], fwd["H"]) <= 2e-2
    assert max_abs_rel(f64(A)[:used], fwd["A"]) <= 2e-2


def test_stalled_natural_wgrad_times_out_and_context_survives(moe_gpu):
    """The same hook on the weight gradient that dequantises its MXFP8 operand
    inside the kernel: the converter warps' bounded waits (for codes that never
    arrive) run out as well, the kernel reports the timeout and returns, and the
    next launch equals global dequantisation + the BF16 weight gradient."""
    m, dev = moe_gpu
    T, d, E, k, f = 300, 256, 4, 2, 256
    rng = np.random.default_rng(78)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    counts = O.expert_counts(idx, E)
    tile_offsets, row_offsets = O.tile_layout(counts, 128)
    s = m.shape(T, d, E, k, f, prec=m.MXFP8)
    n = m.rows_max(s)
    used = int(row_offsets[-1])
    ws = torch.zeros(m.workspace_size(s), dtype=torch.uint8, device=dev)
    dY = torch.zeros(n, d, dtype=torch.bfloat16, device=dev)
    A = torch.zeros(n, f, dtype=torch.bfloat16, device=dev)
    dY[:used] = torch.from_numpy(rng.standard_normal((used, d)).astype(np.float32)).to(dev)
    A[:used] = torch.from_numpy(rng.standard_normal((used, f)).astype(np.float32)).to(dev)
    Aq = torch.empty(n, f, dtype=torch.uint8, device=dev)
    As = torch.empty(n * f // 32, dtype=torch.uint8, device=dev)
    m.quantize_mxfp8(1, n, f, 1, A, Aq, As)
    to = torch.from_numpy(tile_offsets.astype(np.int32)).to(dev)
    dW = torch.zeros(E, d, f, dtype=torch.float32, device=dev)

    def run():
        m.grouped_gemm(s, m.GEMM_WGRAD2_NATURAL, ws, tile_offsets=to, a0=dY, a1=Aq, sfb0=As,
                       out0=dW)

    prev = m.debug_inject_stall(1)
    try:
        m.clear_error(ws)
        run()
        err = m.read_error(ws)
    finally:
        m.debug_inject_stall(prev)
    assert err & m.DEVERR_TIMEOUT
    m.clear_error(ws)
    run()
    assert m.read_error(ws) == 0
    Adq = torch.empty(n, f, dtype=torch.bfloat16, device=dev)
    m.dequantize_mxfp8(n, f, Aq, As, Adq)
    ref = torch.zeros_like(dW)
    m.grouped_gemm(s, m.GEMM_WGRAD2, ws, tile_offsets=to, a0=dY, a1=Adq, out0=ref)
    assert m.read_error(ws) == 0
    assert torch.equal(dW, ref)


def test_stalled_mxfp8_pair_gemm_times_out_and_context_survives(moe_gpu):
    """The same hook on the MXFP8 CTA-pair GEMM in its SwiGLU-backward form,
    where two mover threads per CTA also wait on mbarriers (for dH/dU written by
    the epilogue): every role gives up within its bound, the kernel reports the
    timeout, and the next launch equals a clean launch made before, bit for bit."""
    m, dev = moe_gpu
    T, d, E, k, f = 300, 256, 4, 2, 256
    rng = np.random.default_rng(79)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    counts = O.expert_counts(idx, E)
    tile_offsets, row_offsets = O.tile_layout(counts, 128)
    s = m.shape(T, d, E, k, f, prec=m.MXFP8)
    n = m.rows_max(s)
    used = int(row_offsets[-1])
    ws = torch.zeros(m.workspace_size(s), dtype=torch.uint8, device=dev)
    bf = lambda *sh: torch.from_numpy(rng.standard_normal(sh).astype(np.float32)).to(dev).to(torch.bfloat16)
    dY = torch.zeros(n, d, dtype=torch.bfloat16, device=dev)
    dY[:used] = bf(used, d)
    H, U = bf(n, f), bf(n, f)
    dYq = torch.empty(n, d, dtype=torch.uint8, device=dev)
    dYs = torch.empty(n * d // 32, dtype=torch.uint8, device=dev)
    m.quantize_mxfp8(1, n, d, 1, dY, dYq, dYs)
    buf = m.allocate(s, with_grads=False)
    w = buf.mx_weights
    m.build_mx_weights(s, 0.02 * bf(E, f, d), 0.02 * bf(E, f, d), 0.02 * bf(E, d, f), w)
    to = torch.from_numpy(tile_offsets.astype(np.int32)).to(dev)

    def run():
        o = dict(out0=torch.zeros(n, f, dtype=torch.bfloat16, device=dev),
                 out1=torch.zeros(n, f, dtype=torch.bfloat16, device=dev),
                 out2=torch.zeros(n, f, dtype=torch.uint8, device=dev),
                 out3=torch.zeros(n, f, dtype=torch.uint8, device=dev),
                 osf0=torch.zeros(n * f // 32, dtype=torch.uint8, device=dev),
                 osf1=torch.zeros(n * f // 32, dtype=torch.uint8, device=dev))
        m.grouped_gemm(s, m.GEMM_DGRAD2_SWIGLU, ws, tile_offsets=to, a0=dYq, sfa0=dYs,
                       w0=w["downT_q"], sfb0=w["downT_s"], aux0=H, aux1=U, **o)
        return o

    m.clear_error(ws)
    clean = run()
    assert m.read_error(ws) == 0
    prev = m.debug_inject_stall(1)
    try:
        m.clear_error(ws)
        run()
        err = m.read_error(ws)
    finally:
        m.debug_inject_stall(prev)
    assert err & m.DEVERR_TIMEOUT
    m.clear_error(ws)
    again = run()
    assert m.read_error(ws) == 0
    for key in clean:
        assert torch.equal(clean[key][:used] if clean[key].dim() == 2 else clean[key],
                           again[key][:used] if again[key].dim() == 2 else again[key]), key
