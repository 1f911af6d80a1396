"""Failure detection without a GPU fault: a host-set test hook makes the grouped
GEMM's producer issue nothing, so the MMA issuer's bounded mbarrier wait runs
out (about one second).  The kernel must report MOE_DEVERR_TIMEOUT through the
error word, free its tensor memory and return, and the context must stay usable:
the same GEMM run again afterwards gives the oracle's result.  GPU only."""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
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
