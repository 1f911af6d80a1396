"""Parity of moe_route (router projection, softmax/top-k, counts, offsets, slots)
with the oracle.  Index outputs are compared bit for bit on shared fp32 logits;
gates within 1e-6.  GPU only."""
import numpy as np
import pytest
import torch

from oracle import cpp as O
from synth import CONFIGS, make_inputs
from gpu_util import max_abs_rel, near_tie_tokens, to_dev_bf16

pytestmark = pytest.mark.gpu


def gpu_route(m, dev, T, E, k, logits32=None, x=None, w_router=None, bias=None, d=128):
    s = m.shape(T, d, E, k, 128)
    n = m.rows_max(s)
    i32 = dict(dtype=torch.int32, device=dev)
    out = {
        "logits": (torch.from_numpy(np.ascontiguousarray(logits32)).to(dev) if logits32 is not None
                   else torch.empty(T, E, dtype=torch.float32, device=dev)),
        "topk_idx": torch.empty(T, k, **i32), "gates": torch.empty(T, k, dtype=torch.float32, device=dev),
        "counts": torch.empty(E, **i32), "offsets": torch.empty(E + 1, **i32),
        "tile_offsets": torch.empty(E + 1, **i32), "slot_of_route": torch.empty(T * k, **i32),
        "route_of_slot": torch.full((n,), -7, **i32),
    }
    ws = torch.zeros(m.workspace_size(s), dtype=torch.uint8, device=dev)
    bias_t = torch.from_numpy(bias).to(dev) if bias is not None else None
    m.route(s, x, w_router, bias_t, out["logits"], out["topk_idx"], out["gates"], out["counts"],
            out["offsets"], out["tile_offsets"], out["slot_of_route"], out["route_of_slot"], ws)
    err = m.read_error(ws)
    res = {kk: v.cpu().numpy() for kk, v in out.items()}
    res["err"] = err
    return res


def check_routing(g, logits32, k):
    idx, gates = O.softmax_topk_gates(logits32, k)
    E = logits32.shape[1]
    counts = O.expert_counts(idx, E)
    offsets = O.exclusive_scan(counts)
    tile_offsets, row_offsets = O.tile_layout(counts, 128)
    sor, ros = O.assign_slots(idx, row_offsets)
    assert g["err"] == 0
    np.testing.assert_array_equal(g["topk_idx"], idx)
    np.testing.assert_array_equal(g["counts"], counts)
    np.testing.assert_array_equal(g["offsets"], offsets)
    np.testing.assert_array_equal(g["tile_offsets"], tile_offsets)
    np.testing.assert_array_equal(g["slot_of_route"], sor)
    used = int(row_offsets[-1])
    np.testing.assert_array_equal(g["route_of_slot"][:used], ros)
    assert np.abs(g["gates"] - gates).max() <= 1e-6


@pytest.mark.parametrize("T,E,k", [(256, 8, 2), (1000, 32, 4), (777, 128, 4), (3000, 64, 8),
                                   (50, 256, 32), (300, 1, 1), (100, 8, 8), (1, 16, 3), (65, 40, 5),
                                   # E not a multiple of 4 over many 128-token blocks
                                   (20000, 7, 3), (5000, 250, 8)])
def test_random_logits(moe_gpu, T, E, k):
    m, dev = moe_gpu
    rng = np.random.default_rng(T * 7 + E)
    L = rng.standard_normal((T, E)).astype(np.float32)
    check_routing(gpu_route(m, dev, T, E, k, L), L, k)


def test_ties_go_to_the_lowest_expert(moe_gpu):
    m, dev = moe_gpu
    rng = np.random.default_rng(1)
    L = (rng.integers(-2, 3, size=(500, 16)) * 0.25).astype(np.float32)
    check_routing(gpu_route(m, dev, 500, 16, 4, L), L, 4)
    L = np.full((130, 16), 0.5, dtype=np.float32)
    g = gpu_route(m, dev, 130, 16, 3, L)
    check_routing(g, L, 3)
    assert (g["topk_idx"] == np.arange(3)).all()
    assert np.allclose(g["gates"], 1 / 3, atol=1e-7)


def test_empty_experts_and_tile_boundaries(moe_gpu):
    m, dev = moe_gpu
    rng = np.random.default_rng(2)
    L = rng.standard_normal((129, 4)).astype(np.float32)
    L[:, 0] += 100.0          # every token picks expert 0 first: 129 routes = one tile + 1
    L[:, 3] -= 100.0          # expert 3 never picked
    g = gpu_route(m, dev, 129, 4, 2, L)
    check_routing(g, L, 2)
    assert g["counts"][0] == 129 and g["counts"][3] == 0
    assert g["tile_offsets"][1] == 2


@pytest.mark.parametrize("name", ["fine_grained", "large_pool", "skewed", "mxfp8"])
def test_full_size_workload_logits(moe_gpu, name):
    """Routing of the full-size workloads on the oracle's fp32 logits."""
    m, dev = moe_gpu
    cfg = CONFIGS[name]
    inp = make_inputs(cfg, seed=0, with_grad=False)
    L = O.router_logits(inp["x"], inp["w_router"], inp["bias"]).astype(np.float32)
    g = gpu_route(m, dev, cfg.T, cfg.E, cfg.k, L)
    check_routing(g, L, cfg.k)
    if name == "skewed":
        assert (g["counts"] == 0).sum() >= 4
        assert abs(g["counts"].max() / (cfg.T * cfg.k) - 0.15) < 0.01


def test_nonfinite_logits_flag_and_zero_gates(moe_gpu):
    m, dev = moe_gpu
    rng = np.random.default_rng(3)
    L = rng.standard_normal((100, 8)).astype(np.float32)
    L[3, 5] = np.nan
    L[7, 1] = np.inf
    g = gpu_route(m, dev, 100, 8, 2, L)
    assert g["err"] & m.DEVERR_NONFINITE_LOGIT
    assert (g["gates"][[3, 7]] == 0).all()
    idx = g["topk_idx"]
    assert ((idx >= 0) & (idx < 8)).all() and (idx[:, 0] != idx[:, 1]).all()
    ok = np.ones(100, dtype=bool)
    ok[[3, 7]] = False
    ref_idx, ref_g = O.softmax_topk_gates(L[ok], 2)
    np.testing.assert_array_equal(idx[ok], ref_idx)
    assert np.abs(g["gates"][ok] - ref_g).max() <= 1e-6
    # slots stay a valid permutation
    assert sorted(g["slot_of_route"].tolist()) == sorted(set(g["slot_of_route"].tolist()))


@pytest.mark.parametrize("T,d,E,k,routing", [(300, 256, 8, 2, "none"), (1000, 512, 32, 4, "normal"),
                                             (2048, 2048, 128, 4, "normal"), (257, 128, 16, 16, "normal"),
                                             (10000, 256, 12, 2, "normal"), (10000, 256, 16, 4, "normal")])
def test_router_projection(moe_gpu, T, d, E, k, routing):
    """tcgen05 router GEMM: logits within 1e-5 of the fp64 oracle (relative to the
    largest logit); the selection equals the oracle's except at near-ties.  The
    10000-token cases have more row tiles than half the SMs, so the K loop is
    not split and the epilogue stores directly (E = 12: column by column,
    E = 16: 4-wide)."""
    m, dev = moe_gpu
    inp = make_inputs(T=T, d=d, E=E, k=k, f=128, seed=T + d, routing=routing, with_grad=False)
    x = to_dev_bf16(inp["x"], dev)
    wr = to_dev_bf16(inp["w_router"], dev)
    g = gpu_route(m, dev, T, E, k, None, x=x, w_router=wr, bias=inp["bias"], d=d)
    ref = O.router_logits(inp["x"], inp["w_router"], inp["bias"])
    assert max_abs_rel(g["logits"], ref) < 1e-5
    idx, _ = O.softmax_topk_gates(ref, k)
    tol = 1e-5 * np.abs(ref).max()
    tie = near_tie_tokens(ref, k, 2 * tol)
    same = (np.sort(g["topk_idx"], 1) == np.sort(idx, 1)).all(1)
    assert same[~tie].all()
    # validity on the device's own logits: the chosen k are the k largest, in order
    gl = g["logits"].astype(np.float64)
    chosen = np.take_along_axis(gl, g["topk_idx"].astype(np.int64), axis=1)
    assert (np.diff(chosen, axis=1) <= 0).all()
    kth = np.sort(gl, axis=1)[:, ::-1][:, k - 1]
    assert (chosen[:, -1] == kth).all()
    assert (g["counts"].sum() == T * k) and g["err"] == 0


@pytest.mark.parametrize("T,d,E,k", [(10000, 256, 64, 8), (12000, 128, 250, 4), (9999, 128, 1, 1),
                                     (20000, 512, 128, 2), (32768, 256, 256, 8), (3000, 128, 40, 12)],
                         ids=lambda v: str(v))
def test_routing_with_router_projection_large(moe_gpu, T, d, E, k):
    """Router GEMM, top-k (four threads per token for k <= 8, a warp per token
    above), scan and slots on many routing blocks, a ragged last block and E
    not a multiple of 4: bit for bit the oracle's routing of the logits the call
    wrote, which agree with the oracle's own logits to 1e-5."""
    m, dev = moe_gpu
    inp = make_inputs(T=T, d=d, E=E, k=k, f=128, seed=T + E, with_grad=False)
    g = gpu_route(m, dev, T, E, k, x=to_dev_bf16(inp["x"], dev),
                  w_router=to_dev_bf16(inp["w_router"], dev), bias=inp["bias"], d=d)
    check_routing(g, g["logits"], k)
    ref = O.router_logits(inp["x"], inp["w_router"], inp["bias"])
    assert max_abs_rel(g["logits"], ref) < 1e-5


def test_non_finite_logit_from_the_router_projection(moe_gpu):
    """A NaN in the bias makes one token's logits non-finite: the error bit is
    set and only that token's gates are zeroed (its neighbours in the same warp
    and block keep theirs); its k experts are still distinct."""
    m, dev = moe_gpu
    T, d, E, k = 10000, 128, 32, 4
    inp = make_inputs(T=T, d=d, E=E, k=k, f=128, seed=5, with_grad=False)
    bias = inp["bias"].copy()
    bias[1234, 7] = np.nan
    g = gpu_route(m, dev, T, E, k, x=to_dev_bf16(inp["x"], dev),
                  w_router=to_dev_bf16(inp["w_router"], dev), bias=bias, d=d)
    assert g["err"] & m.DEVERR_NONFINITE_LOGIT
    assert (g["gates"][1234] == 0).all()
    ok = np.ones(T, dtype=bool)
    ok[1234] = False
    assert np.abs(g["gates"][ok].sum(1) - 1).max() < 1e-5
    assert (np.sort(g["topk_idx"], axis=1)[:, 1:] != np.sort(g["topk_idx"], axis=1)[:, :-1]).all()
