"""Python face of the C++ oracle (oracle/moe_oracle.cpp): TEST INFRASTRUCTURE.

Only the tests, the package smoke check and the benchmark's CPU-baseline leg
import this module.  The CUDA library never imports, links or calls it.

The functions have the names, arguments and results of the float64 numpy
restatement in moe_oracle.py (kept as an independent cross-check): every
floating-point step runs in the C++ library in double; this module only widens
inputs exactly to float64 (bf16 bit patterns -> float64), allocates the result
arrays and walks the experts of the layer in order.  The library is compiled
with g++ (-O2, OpenMP, no FMA contraction) on first use, or by build().
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(_HERE, "moe_oracle.cpp")
LIB = os.path.join(_HERE, "libmoe_oracle.so")
FLAGS = ["-O2", "-std=c++17", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared"]

__all__ = [
    "build", "threads", "as_f64", "router_logits", "softmax_topk_gates", "expert_counts",
    "exclusive_scan", "tile_layout", "assign_slots", "dispatch", "silu", "silu_grad",
    "expert_ffn_forward", "combine", "combine_backward", "expert_ffn_backward",
    "expert_ffn_forward_mxfp8", "expert_ffn_backward_mxfp8",
    "dispatch_backward", "router_backward", "load_balance", "load_balance_dlogits",
    "layer_forward", "layer_backward", "dense_forward", "E4M3_VALUES", "E4M3_MAX",
    "e4m3_encode", "mx_scale_exponent", "quantize_mxfp8", "dequantize_mxfp8",
    "layer_forward_mxfp8", "layer_backward_mxfp8",
]

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile libmoe_oracle.so next to its source (when missing or older)."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    tmp = LIB + f".{os.getpid()}.tmp"
    cmd = [os.environ.get("CXX", "g++"), *FLAGS, "-o", tmp, SRC]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("building the C++ oracle failed:\n" + r.stdout + r.stderr)
    os.replace(tmp, LIB)
    return LIB


_P = ctypes.c_void_p
_I = ctypes.c_int64
_C = ctypes.c_int
_D = ctypes.c_double
_SIG = {
    "mo_num_threads": ([], _C),
    "mo_widen_bf16": ([_P, _I, _P], _C),
    "mo_silu": ([_P, _I, _P], _C),
    "mo_silu_grad": ([_P, _I, _P], _C),
    "mo_router_logits": ([_P, _P, _P, _I, _I, _I, _P], _C),
    "mo_softmax_topk_gates": ([_P, _I, _C, _C, _P, _P], _C),
    "mo_expert_counts": ([_P, _I, _C, _P], _C),
    "mo_exclusive_scan": ([_P, _C, _P], _C),
    "mo_tile_layout": ([_P, _C, _C, _P, _P], _C),
    "mo_assign_slots": ([_P, _I, _C, _C, _P, _P, _P], _C),
    "mo_dispatch": ([_P, _I, _I, _C, _P, _I, _P], _C),
    "mo_expert_forward": ([_P, _I, _I, _I, _P, _P, _P, _C, _P, _P, _P, _P, _P], _C),
    "mo_combine": ([_P, _I, _P, _P, _I, _C, _P], _C),
    "mo_combine_backward": ([_P, _P, _I, _P, _P, _I, _C, _I, _P, _P], _C),
    "mo_expert_backward": ([_P, _P, _P, _P, _P, _I, _I, _I, _P, _P, _P, _C,
                            _P, _P, _P, _P, _P, _P], _C),
    "mo_dispatch_backward": ([_P, _I, _P, _I, _C, _P], _C),
    "mo_router_backward": ([_P, _P, _P, _I, _C, _C, _P, _P, _P, _I, _P, _P, _P], _C),
    "mo_load_balance": ([_P, _P, _I, _C, _C, _P, _P, _P], _C),
    "mo_load_balance_dlogits": ([_P, _P, _I, _C, _C, _D, _P], _C),
    "mo_e4m3_value": ([_C], _D),
    "mo_e4m3_encode": ([_P, _I, _P], _C),
    "mo_mx_scale_exponent": ([_P, _I, _P], _C),
    "mo_quantize_mxfp8": ([_P, _I, _I, _P, _P], _C),
    "mo_dequantize_mxfp8": ([_P, _P, _I, _I, _P], _C),
    "mo_qdq_rows": ([_P, _I, _I], _C),
}


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(LIB)
            for name, (args, res) in _SIG.items():
                fn = getattr(L, name)
                fn.argtypes = args
                fn.restype = res
            _lib = L
    return _lib


def threads() -> int:
    """OpenMP threads the library runs on."""
    return int(lib().mo_num_threads())


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _ok(rc, what):
    if rc != 0:
        raise ValueError(f"{what}: invalid argument")


# --------------------------------------------------------------------------
# input widening (data conversion only)
# --------------------------------------------------------------------------
def as_f64(a) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64, exactly; float arrays as they are."""
    a = np.asarray(a)
    if a.dtype == np.uint16:
        bits = np.ascontiguousarray(a)
        out = np.empty(bits.shape, dtype=np.float64)
        lib().mo_widen_bf16(_ptr(bits), bits.size, _ptr(out))
        return out
    return np.ascontiguousarray(a, dtype=np.float64)


# --------------------------------------------------------------------------
# a1-a3
# --------------------------------------------------------------------------
def router_logits(x, w_router, bias=None) -> np.ndarray:
    X, W = as_f64(x), as_f64(w_router)
    T, d = X.shape
    E = W.shape[0]
    B = None if bias is None else as_f64(bias)
    out = np.empty((T, E))
    lib().mo_router_logits(_ptr(X), _ptr(W), _ptr(B), T, d, E, _ptr(out))
    return out


def softmax_topk_gates(logits, k: int):
    L = as_f64(logits)
    T, E = L.shape
    if not 1 <= k <= E:
        raise ValueError("need 1 <= k <= E")
    idx = np.empty((T, k), dtype=np.int32)
    gates = np.empty((T, k))
    if lib().mo_softmax_topk_gates(_ptr(L), T, E, k, _ptr(idx), _ptr(gates)) != 0:
        raise FloatingPointError("non-finite router logit")
    return idx, gates


def expert_counts(topk_idx, E: int) -> np.ndarray:
    idx = _c(topk_idx, np.int32)
    out = np.empty(E, dtype=np.int64)
    _ok(lib().mo_expert_counts(_ptr(idx), idx.size, E, _ptr(out)), "expert_counts")
    return out


def exclusive_scan(counts) -> np.ndarray:
    c = _c(counts, np.int64)
    out = np.empty(c.size + 1, dtype=np.int64)
    lib().mo_exclusive_scan(_ptr(c), c.size, _ptr(out))
    return out


def tile_layout(counts, bm: int):
    c = _c(counts, np.int64)
    to = np.empty(c.size + 1, dtype=np.int64)
    ro = np.empty(c.size + 1, dtype=np.int64)
    _ok(lib().mo_tile_layout(_ptr(c), c.size, bm, _ptr(to), _ptr(ro)), "tile_layout")
    return to, ro


def assign_slots(topk_idx, row_offsets):
    idx = _c(topk_idx, np.int32)
    T, k = idx.shape
    ro = _c(row_offsets, np.int64)
    sor = np.empty(T * k, dtype=np.int64)
    ros = np.empty(int(ro[-1]), dtype=np.int64)
    lib().mo_assign_slots(_ptr(idx), T, k, ro.size - 1, _ptr(ro), _ptr(sor), _ptr(ros))
    return sor, ros


def dispatch(x, slot_of_route, k: int, n_rows: int) -> np.ndarray:
    X = as_f64(x)
    T, d = X.shape
    s = _c(slot_of_route, np.int64)
    out = np.empty((n_rows, d))
    lib().mo_dispatch(_ptr(X), T, d, k, _ptr(s), n_rows, _ptr(out))
    return out


# --------------------------------------------------------------------------
# a5-a7
# --------------------------------------------------------------------------
def silu(h):
    h = as_f64(h)
    out = np.empty_like(h)
    lib().mo_silu(_ptr(h), h.size, _ptr(out))
    return out


def silu_grad(h):
    h = as_f64(h)
    out = np.empty_like(h)
    lib().mo_silu_grad(_ptr(h), h.size, _ptr(out))
    return out


def _expert_forward(Xd, w_gate, w_up, w_down, row_offsets, mx: bool):
    Xd = as_f64(Xd)
    ro = [int(v) for v in np.asarray(row_offsets).tolist()]
    E = len(ro) - 1
    f = np.asarray(w_gate).shape[1]
    n, d = Xd.shape
    H, U, A, Y = np.zeros((n, f)), np.zeros((n, f)), np.zeros((n, f)), np.zeros((n, d))
    Aq = np.zeros((n, f)) if mx else None
    for e in range(E):
        a, b = ro[e], ro[e + 1]
        if a == b:
            continue
        wg, wu, wd = as_f64(w_gate[e]), as_f64(w_up[e]), as_f64(w_down[e])
        h, u, act, y = (np.empty((b - a, f)), np.empty((b - a, f)), np.empty((b - a, f)),
                        np.empty((b - a, d)))
        aq = np.empty((b - a, f)) if mx else None
        lib().mo_expert_forward(_ptr(np.ascontiguousarray(Xd[a:b])), b - a, d, f, _ptr(wg),
                                _ptr(wu), _ptr(wd), int(mx), _ptr(h), _ptr(u), _ptr(act),
                                _ptr(aq), _ptr(y))
        H[a:b], U[a:b], A[a:b], Y[a:b] = h, u, act, y
        if mx:
            Aq[a:b] = aq
    return H, U, A, Aq, Y


def expert_ffn_forward(Xd, w_gate, w_up, w_down, row_offsets):
    H, U, A, _, Y = _expert_forward(Xd, w_gate, w_up, w_down, row_offsets, False)
    return H, U, A, Y


def expert_ffn_forward_mxfp8(Xd, w_gate, w_up, w_down, row_offsets):
    """The MXFP8 forward's per-expert part on dispatched (already quantised)
    rows: returns H, U, A, Aq, Y."""
    return _expert_forward(Xd, w_gate, w_up, w_down, row_offsets, True)


def combine(Y, gates, slot_of_route, T: int, k: int) -> np.ndarray:
    Y = as_f64(Y)
    g = _c(as_f64(gates).reshape(T, k), np.float64)
    s = _c(slot_of_route, np.int64)
    out = np.empty((T, Y.shape[1]))
    lib().mo_combine(_ptr(Y), Y.shape[1], _ptr(g), _ptr(s), T, k, _ptr(out))
    return out


# --------------------------------------------------------------------------
# a8-a14
# --------------------------------------------------------------------------
def combine_backward(d_out, Y, gates, slot_of_route, T: int, k: int, n_rows: int):
    dO, Y = as_f64(d_out), as_f64(Y)
    g = _c(as_f64(gates).reshape(T, k), np.float64)
    s = _c(slot_of_route, np.int64)
    d = dO.shape[1]
    dg = np.empty((T, k))
    dY = np.empty((n_rows, d))
    lib().mo_combine_backward(_ptr(dO), _ptr(Y), d, _ptr(g), _ptr(s), T, k, n_rows, _ptr(dg),
                              _ptr(dY))
    return dg, dY


def _expert_backward(dY, Xd, H, U, A, w_gate, w_up, w_down, row_offsets, mx: bool):
    dY, Xd, H, U, A = (as_f64(v) for v in (dY, Xd, H, U, A))
    ro = [int(v) for v in np.asarray(row_offsets).tolist()]
    E = len(ro) - 1
    f, d = np.asarray(w_gate).shape[1:]
    n = Xd.shape[0]
    dH, dU, dXd = np.zeros((n, f)), np.zeros((n, f)), np.zeros((n, d))
    dWg, dWu, dWd = np.zeros((E, f, d)), np.zeros((E, f, d)), np.zeros((E, d, f))
    for e in range(E):
        a, b = ro[e], ro[e + 1]
        if a == b:
            continue
        m = b - a
        wg, wu, wd = as_f64(w_gate[e]), as_f64(w_up[e]), as_f64(w_down[e])
        sl = lambda v: np.ascontiguousarray(v[a:b])
        gh, gu, gx = np.empty((m, f)), np.empty((m, f)), np.empty((m, d))
        lib().mo_expert_backward(_ptr(sl(dY)), _ptr(sl(Xd)), _ptr(sl(H)), _ptr(sl(U)), _ptr(sl(A)),
                                 m, d, f, _ptr(wg), _ptr(wu), _ptr(wd), int(mx), _ptr(gh),
                                 _ptr(gu), _ptr(gx), _ptr(dWg[e]), _ptr(dWu[e]), _ptr(dWd[e]))
        dH[a:b], dU[a:b], dXd[a:b] = gh, gu, gx
    return {"dH": dH, "dU": dU, "dXd": dXd, "dW_gate": dWg, "dW_up": dWu, "dW_down": dWd}


def expert_ffn_backward(dY, Xd, H, U, A, w_gate, w_up, w_down, row_offsets):
    return _expert_backward(dY, Xd, H, U, A, w_gate, w_up, w_down, row_offsets, False)


def expert_ffn_backward_mxfp8(dY, Xd, H, U, Aq, w_gate, w_up, w_down, row_offsets):
    """The MXFP8 backward's per-expert part (Aq: the forward's quantised A)."""
    return _expert_backward(dY, Xd, H, U, Aq, w_gate, w_up, w_down, row_offsets, True)


def dispatch_backward(dXd, slot_of_route, T: int, k: int) -> np.ndarray:
    dXd = as_f64(dXd)
    s = _c(slot_of_route, np.int64)
    out = np.empty((T, dXd.shape[1]))
    lib().mo_dispatch_backward(_ptr(dXd), dXd.shape[1], _ptr(s), T, k, _ptr(out))
    return out


def load_balance(logits, topk_idx, E: int):
    L = as_f64(logits)
    idx = _c(topk_idx, np.int32)
    T, k = idx.shape
    P, f = np.empty(E), np.empty(E)
    lbl = ctypes.c_double()
    lib().mo_load_balance(_ptr(L), _ptr(idx), T, k, E, ctypes.byref(lbl), _ptr(P), _ptr(f))
    return float(lbl.value), P, f


def load_balance_dlogits(logits, topk_idx, E: int, coef: float) -> np.ndarray:
    L = as_f64(logits)
    idx = _c(topk_idx, np.int32)
    T, k = idx.shape
    out = np.empty((T, E))
    lib().mo_load_balance_dlogits(_ptr(L), _ptr(idx), T, k, E, float(coef), _ptr(out))
    return out


def router_backward(d_gates, gates, topk_idx, E: int, x=None, w_router=None, dlogits_extra=None):
    dg = _c(as_f64(d_gates), np.float64)
    g = _c(as_f64(gates), np.float64)
    idx = _c(topk_idx, np.int32)
    T, k = idx.shape
    extra = None if dlogits_extra is None else as_f64(dlogits_extra)
    dl = np.empty((T, E))
    out = {"dlogits": dl}
    if w_router is not None:
        W, X = as_f64(w_router), as_f64(x)
        d = W.shape[1]
        dxr, dwr = np.empty((T, d)), np.empty((E, d))
        lib().mo_router_backward(_ptr(dg), _ptr(g), _ptr(idx), T, k, E, _ptr(extra), _ptr(X),
                                 _ptr(W), d, _ptr(dl), _ptr(dxr), _ptr(dwr))
        out["dx_router"], out["dW_router"] = dxr, dwr
    else:
        lib().mo_router_backward(_ptr(dg), _ptr(g), _ptr(idx), T, k, E, _ptr(extra), None, None,
                                 0, _ptr(dl), None, None)
    return out


# --------------------------------------------------------------------------
# the whole layer
# --------------------------------------------------------------------------
def _route(x, w_router, bias, k, bm, logits):
    if logits is None:
        logits = router_logits(x, w_router, bias)
    logits = as_f64(logits)
    T, E = logits.shape
    idx, gates = softmax_topk_gates(logits, k)
    counts = expert_counts(idx, E)
    tile_offsets, row_offsets = tile_layout(counts, bm)
    slot_of_route, route_of_slot = assign_slots(idx, row_offsets)
    return {"logits": logits, "topk_idx": idx, "gates": gates, "counts": counts,
            "offsets": exclusive_scan(counts), "tile_offsets": tile_offsets,
            "row_offsets": row_offsets, "slot_of_route": slot_of_route,
            "route_of_slot": route_of_slot, "k": k, "bm": bm}


def layer_forward(x, w_router, bias, w_gate, w_up, w_down, k: int, bm: int = 128, logits=None):
    """route -> dispatch -> per-expert SwiGLU -> combine (all arithmetic in C++)."""
    r = _route(x, w_router, bias, k, bm, logits)
    T = r["logits"].shape[0]
    Xd = dispatch(x, r["slot_of_route"], k, int(r["row_offsets"][-1]))
    H, U, A, _, Y = _expert_forward(Xd, w_gate, w_up, w_down, r["row_offsets"], False)
    r.update(Xd=Xd, H=H, U=U, A=A, Y=Y, out=combine(Y, r["gates"], r["slot_of_route"], T, k))
    return r


def _layer_backward(fwd, d_out, x, w_router, w_gate, w_up, w_down, lb_coef, mx):
    T, k = fwd["topk_idx"].shape
    E = fwd["logits"].shape[1]
    n_rows = fwd["Xd"].shape[0]
    d_gates, dY = combine_backward(d_out, fwd["Y"], fwd["gates"], fwd["slot_of_route"], T, k, n_rows)
    act = fwd["Aq"] if mx else fwd["A"]
    g = _expert_backward(dY, fwd["Xd"], fwd["H"], fwd["U"], act, w_gate, w_up, w_down,
                         fwd["row_offsets"], mx)
    dx = dispatch_backward(g["dXd"], fwd["slot_of_route"], T, k)
    extra = (load_balance_dlogits(fwd["logits"], fwd["topk_idx"], E, lb_coef)
             if lb_coef != 0.0 else None)
    rb = router_backward(d_gates, fwd["gates"], fwd["topk_idx"], E,
                         x if w_router is not None else None, w_router, extra)
    if w_router is not None:
        dx = dx + rb["dx_router"]
    out = {"d_gates": d_gates, "dY": dY, "dx": dx, "dlogits": rb["dlogits"]}
    out.update(g)
    if w_router is not None:
        out["dW_router"] = rb["dW_router"]
    return out


def layer_backward(fwd, d_out, x, w_router, w_gate, w_up, w_down, lb_coef: float = 0.0):
    return _layer_backward(fwd, d_out, x, w_router, w_gate, w_up, w_down, lb_coef, False)


def dense_forward(x, w_router, bias, w_gate, w_up, w_down, k: int, logits=None):
    """Every expert on every token, masked by the [T, E] gate matrix (tiny shapes)."""
    if logits is None:
        logits = router_logits(x, w_router, bias)
    idx, gates = softmax_topk_gates(logits, k)
    X = as_f64(x)
    T, E = as_f64(logits).shape
    f = np.asarray(w_gate).shape[1]
    d = X.shape[1]
    out = np.zeros_like(X)
    for e in range(E):
        h, u, a, y = np.empty((T, f)), np.empty((T, f)), np.empty((T, f)), np.empty((T, d))
        lib().mo_expert_forward(_ptr(X), T, d, f, _ptr(as_f64(w_gate[e])), _ptr(as_f64(w_up[e])),
                                _ptr(as_f64(w_down[e])), 0, _ptr(h), _ptr(u), _ptr(a), None,
                                _ptr(y))
        G = np.zeros((T, 1))
        for j in range(k):
            G[idx[:, j] == e, 0] = gates[idx[:, j] == e, j]
        out += G * y
    return out


# --------------------------------------------------------------------------
# a15: MXFP8
# --------------------------------------------------------------------------
def _e4m3_table() -> np.ndarray:
    return np.array([lib().mo_e4m3_value(c) for c in range(256)], dtype=np.float64)


class _LazyTable:
    """The E4M3 value of every code, from the C++ decoder (built on first use)."""

    _v = None

    def get(self):
        if _LazyTable._v is None:
            _LazyTable._v = _e4m3_table()
        return _LazyTable._v


E4M3_MAX = 448.0


def __getattr__(name):
    if name == "E4M3_VALUES":
        return _LazyTable().get()
    raise AttributeError(name)


def e4m3_encode(v) -> np.ndarray:
    v = as_f64(v)
    out = np.empty(v.shape, dtype=np.uint8)
    lib().mo_e4m3_encode(_ptr(v), v.size, _ptr(out))
    return out


def mx_scale_exponent(amax) -> np.ndarray:
    a = as_f64(amax)
    out = np.empty(a.shape, dtype=np.int64)
    lib().mo_mx_scale_exponent(_ptr(a), a.size, _ptr(out))
    return out


def quantize_mxfp8(a, block: int = 32):
    if block != 32:
        raise ValueError("MXFP8 blocks hold 32 values")
    a = as_f64(a)
    K = a.shape[-1]
    if K % 32:
        raise ValueError("last axis must be a multiple of the block size")
    codes = np.empty(a.shape, dtype=np.uint8)
    scales = np.empty(a.shape[:-1] + (K // 32,), dtype=np.uint8)
    lib().mo_quantize_mxfp8(_ptr(a), a.size // K, K, _ptr(codes), _ptr(scales))
    return codes, scales


def dequantize_mxfp8(codes, scales, block: int = 32) -> np.ndarray:
    c = _c(codes, np.uint8)
    s = _c(scales, np.uint8)
    K = c.shape[-1]
    out = np.empty(c.shape, dtype=np.float64)
    _ok(lib().mo_dequantize_mxfp8(_ptr(c), _ptr(s), c.size // K, K, _ptr(out)), "dequantize")
    return out


def _qdq(a):
    a = np.array(as_f64(a), dtype=np.float64, copy=True, order="C")
    _ok(lib().mo_qdq_rows(_ptr(a), a.size // a.shape[-1], a.shape[-1]), "qdq")
    return a


def layer_forward_mxfp8(x, w_router, bias, w_gate, w_up, w_down, k: int, bm: int = 128, logits=None):
    """MXFP8 forward: x quantised once per token along d before the dispatch;
    per expert, W_gate/W_up quantised along d and W_down along f, A along f."""
    r = _route(x, w_router, bias, k, bm, logits)
    T = r["logits"].shape[0]
    Xd = dispatch(_qdq(x), r["slot_of_route"], k, int(r["row_offsets"][-1]))
    H, U, A, Aq, Y = _expert_forward(Xd, w_gate, w_up, w_down, r["row_offsets"], True)
    r.update(Xd=Xd, H=H, U=U, A=A, Aq=Aq, Y=Y,
             out=combine(Y, r["gates"], r["slot_of_route"], T, k))
    return r


def layer_backward_mxfp8(fwd, d_out, x, w_router, w_gate, w_up, w_down, lb_coef: float = 0.0):
    """MXFP8 data-gradient GEMMs (dY along d, dH/dU along f, second weight cache)
    and BF16 weight gradients on the dequantised activations."""
    return _layer_backward(fwd, d_out, x, w_router, w_gate, w_up, w_down, lb_coef, True)
