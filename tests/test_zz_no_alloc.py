"""moe_route_noalloc against moe_route (GPU).

moe_route_noalloc serves callers that cannot allocate device memory (plugins
whose host owns all device memory, fixed memory budgets, loops that must stay
out of cudaMalloc because it can synchronise the device): it takes no workspace
and keeps its scratch in a static device array of the library.  Its
results must equal those of moe_route, the call it stands in for, on two calls
in a row (the array keeps the previous call's contents, so the second call
checks that nothing stale leaks through).  This file is collected last on
purpose and also passes when run alone in a fresh process.
"""
import numpy as np
import pytest
import torch

from synth import make_inputs
from gpu_util import to_dev_bf16

pytestmark = pytest.mark.gpu


def _outputs(dev, T, E, k, n):
    i32 = dict(dtype=torch.int32, device=dev)
    return {
        "logits": torch.empty(T, E, dtype=torch.float32, device=dev),
        "topk_idx": torch.empty(T, k, **i32), "gates": torch.empty(T, k, dtype=torch.float32, device=dev),
        "counts": torch.empty(E, **i32), "offsets": torch.empty(E + 1, **i32),
        "tile_offsets": torch.empty(E + 1, **i32), "slot_of_route": torch.empty(T * k, **i32),
        "route_of_slot": torch.full((n,), -9, **i32),
    }


def _args(o):
    return (o["logits"], o["topk_idx"], o["gates"], o["counts"], o["offsets"], o["tile_offsets"],
            o["slot_of_route"], o["route_of_slot"])


@pytest.mark.parametrize("T,d,E,k,use_router", [(3000, 512, 64, 8, True), (777, 128, 16, 3, False),
                                                (8192, 2048, 32, 4, True), (50, 128, 256, 32, False),
                                                (300, 128, 1, 1, False), (5000, 128, 250, 8, False)])
def test_noalloc_route_matches_route_twice(moe_gpu, T, d, E, k, use_router):
    m, dev = moe_gpu
    inp = make_inputs(T=T, d=d, E=E, k=k, f=128, seed=T + E, with_grad=False)
    s = m.shape(T, d, E, k, 128)
    n = m.rows_max(s)
    x = to_dev_bf16(inp["x"], dev)
    wr = to_dev_bf16(inp["w_router"], dev) if use_router else None
    bias = torch.from_numpy(inp["bias"]).to(dev)
    given = torch.from_numpy(np.random.default_rng(T).standard_normal((T, E)).astype(np.float32)).to(dev)

    ref = _outputs(dev, T, E, k, n)
    if not use_router:
        ref["logits"].copy_(given)
    ws = torch.zeros(m.workspace_size(s), dtype=torch.uint8, device=dev)
    m.route(s, x, wr, bias, *_args(ref), ws)
    assert m.read_error(ws) == 0
    used = int(ref["tile_offsets"][-1].item()) * 128

    for call in range(2):
        got = _outputs(dev, T, E, k, n)
        if not use_router:
            got["logits"].copy_(given)
        dev_err = torch.full((4,), 123, dtype=torch.int32, device=dev)
        m.route_noalloc(s, x, wr, bias, *_args(got), dev_err)
        torch.cuda.synchronize()
        assert int(dev_err[0].item()) == 0, call
        for name in ("topk_idx", "counts", "offsets", "tile_offsets", "slot_of_route"):
            assert torch.equal(got[name], ref[name]), (call, name)
        assert torch.equal(got["route_of_slot"][:used], ref["route_of_slot"][:used]), call
        # same kernels on the same inputs: gates and logits are identical, which
        # is inside the 1e-6 gate tolerance the routing tests use
        assert torch.equal(got["gates"], ref["gates"]), call
        assert torch.equal(got["logits"], ref["logits"]), call


def test_noalloc_reports_device_errors_and_clears_them(moe_gpu):
    m, dev = moe_gpu
    T, E, k = 100, 8, 2
    s = m.shape(T, 128, E, k, 128)
    n = m.rows_max(s)
    bad = np.random.default_rng(0).standard_normal((T, E)).astype(np.float32)
    bad[5, 3] = np.nan
    for logits, want in ((bad, m.DEVERR_NONFINITE_LOGIT), (np.nan_to_num(bad), 0)):
        o = _outputs(dev, T, E, k, n)
        o["logits"].copy_(torch.from_numpy(logits))
        dev_err = torch.zeros(4, dtype=torch.int32, device=dev)
        m.route_noalloc(s, None, None, None, *_args(o), dev_err)
        torch.cuda.synchronize()
        assert int(dev_err[0].item()) == want


def test_noalloc_rejects_shapes_beyond_its_scratch(moe_gpu):
    m, dev = moe_gpu
    T, E, k = 1 << 20, 64, 8             # 32 MiB of route ranks: more than the 2 MiB array
    s = m.shape(T, 128, E, k, 128)
    dummy = torch.empty(16, dtype=torch.int32, device=dev)
    with pytest.raises(m.MoEError) as ei:
        m.route_noalloc(s, None, None, None, dummy, dummy, dummy, dummy, dummy, dummy, dummy, dummy)
    assert ei.value.code == m.ERR_SCRATCH_LIMIT
