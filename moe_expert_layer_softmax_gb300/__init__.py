"""Python binding of libmoe_gb300.so, the sm_103a MoE expert layer library.

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  Tensors are torch CUDA tensors (used for device memory and streams);
the C entry points have the same names without the `moe_` prefix.  There is no
fallback: if the library is missing or cannot be loaded, every call raises.

Shapes follow include/moe.h: x [T, d] bf16, W_r [E, d] bf16, W_gate/W_up
[E, f, d] bf16, W_down [E, d, f] bf16; dispatched row buffers have
`rows_max(shape)` rows.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

_PKG = os.path.dirname(os.path.abspath(__file__))
# MOE_GB300_CHECKS=1 selects the checks build (device-side bounds checks, see
# moe_checks_read) and guard bands around every buffer allocate() hands out
CHECKS = os.environ.get("MOE_GB300_CHECKS", "") == "1"
LIB_PATH = os.path.join(_PKG, "libmoe_gb300_checks.so" if CHECKS else "libmoe_gb300.so")

BF16, MXFP8 = 0, 1
TILE_M = 128

GEMM_FWD1_SWIGLU = 0
GEMM_FWD2 = 1
GEMM_DGRAD2_SWIGLU = 2
GEMM_DGRAD1 = 3
GEMM_WGRAD2 = 4
GEMM_WGRAD1 = 5
GEMM_WGRAD2_NATURAL = 6   # activation operand as MXFP8 codes + scales, dequantised in the kernel
GEMM_WGRAD1_NATURAL = 7

DEVERR_NONFINITE_LOGIT = 0x1
DEVERR_TIMEOUT = 0x2
DEVERR_BOUNDS = 0x4

_ERRORS = {-1: "MOE_ERR_INVALID", -2: "MOE_ERR_UNSUPPORTED", -3: "MOE_ERR_ALIGN",
           -4: "MOE_ERR_CUDA", -5: "MOE_ERR_NOT_INIT", -6: "MOE_ERR_SCRATCH_LIMIT"}
ERR_SCRATCH_LIMIT = -6

# every symbol the C header declares
EXPORTS = (
    "moe_init", "moe_rows_max", "moe_workspace_size", "moe_clear_error", "moe_read_error",
    "moe_route", "moe_dispatch", "moe_quantize_mxfp8", "moe_grouped_gemm", "moe_combine",
    "moe_combine_bwd", "moe_dispatch_bwd", "moe_router_bwd", "moe_layer_fwd", "moe_layer_bwd",
    "moe_route_noalloc", "moe_dequantize_mxfp8", "moe_build_mx_weights",
    "moe_debug_inject_stall", "moe_profile_start", "moe_profile_stop", "moe_load_balance",
    "moe_checks_read",
)


class MoEError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} returned {code} ({_ERRORS.get(code, 'unknown')})")
        self.code = code


class Shape(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("d_model", ctypes.c_int32), ("n_experts", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("d_ff", ctypes.c_int32), ("prec", ctypes.c_int32)]


_vp = ctypes.c_void_p


class GemmArgs(ctypes.Structure):
    _fields_ = [(n, _vp) for n in ("tile_offsets", "a0", "a1", "w0", "w1", "aux0", "aux1",
                                   "out0", "out1", "out2", "sfa0", "sfa1", "sfb0", "sfb1",
                                   "out3", "osf0", "osf1")]


MX_WEIGHT_FIELDS = ("gu_q", "gu_s", "down_q", "down_s", "downT_q", "downT_s", "gateT_q",
                    "gateT_s", "upT_q", "upT_s")
MX_BUFFER_FIELDS = ("xd_q", "xd_s", "a_q", "a_s", "dy_q", "dy_s", "dh_q", "dh_s", "du_q",
                    "du_s", "xd_dq", "a_dq")


class MxWeights(ctypes.Structure):
    _fields_ = [(n, _vp) for n in MX_WEIGHT_FIELDS]


class MxBuffers(ctypes.Structure):
    _fields_ = [(n, _vp) for n in MX_BUFFER_FIELDS]


class Saved(ctypes.Structure):
    _fields_ = [(n, _vp) for n in ("logits", "topk_idx", "gates", "counts", "offsets",
                                   "tile_offsets", "slot_of_route", "route_of_slot", "xd", "h",
                                   "u", "a", "y", "lb_stats")]


class FwdArgs(ctypes.Structure):
    _fields_ = [(n, _vp) for n in ("x", "w_router", "logit_bias", "w_gate", "w_up", "w_down",
                                   "out", "mx_weights", "mx")]


class BwdArgs(ctypes.Structure):
    _fields_ = [(n, _vp) for n in ("d_out", "x", "w_router", "w_gate", "w_up", "w_down", "dx",
                                   "dw_router", "dw_gate", "dw_up", "dw_down", "d_gates",
                                   "dlogits", "dy", "dh", "du", "dxd", "mx_weights", "mx")] + \
        [("recompute", ctypes.c_int32), ("lb_coef", ctypes.c_float)]


_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the library (once).  Raises if it is missing: there is no fallback."""
    global _lib
    if _lib is not None:
        return _lib
    if CHECKS and path == LIB_PATH:
        from . import _build
        _build.build(checks=True)
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with __graft_entry__.build() "
                           "(the MoE layer has no CPU or eager fallback)")
    lib = ctypes.CDLL(path)
    P = ctypes.POINTER
    i32 = ctypes.c_int32
    sig = {
        "moe_init": [ctypes.c_int],
        "moe_rows_max": [P(Shape), P(ctypes.c_int64)],
        "moe_workspace_size": [P(Shape), P(ctypes.c_size_t)],
        "moe_clear_error": [_vp, _vp],
        "moe_read_error": [_vp, P(i32), _vp],
        "moe_debug_inject_stall": [i32],
        "moe_profile_start": [i32],
        "moe_load_balance": [P(Shape), _vp, _vp, _vp, _vp, _vp],
        "moe_profile_stop": [_vp, _vp],
        "moe_route": [P(Shape)] + [_vp] * 11 + [_vp, _vp],
        "moe_route_noalloc": [P(Shape)] + [_vp] * 11 + [_vp, _vp],
        "moe_dispatch": [P(Shape)] + [_vp] * 7 + [_vp],
        "moe_quantize_mxfp8": [i32, i32, i32, i32, _vp, _vp, _vp, _vp],
        "moe_dequantize_mxfp8": [ctypes.c_int64, i32, _vp, _vp, _vp, _vp],
        "moe_build_mx_weights": [P(Shape), _vp, _vp, _vp, P(MxWeights), _vp],
        "moe_grouped_gemm": [P(Shape), i32, P(GemmArgs), _vp, _vp],
        "moe_combine": [P(Shape)] + [_vp] * 4 + [_vp],
        "moe_combine_bwd": [P(Shape)] + [_vp] * 12 + [_vp],
        "moe_dispatch_bwd": [P(Shape)] + [_vp] * 6 + [_vp],
        "moe_router_bwd": [P(Shape)] + [_vp] * 7 + [_vp],
        "moe_layer_fwd": [P(Shape), P(FwdArgs), P(Saved), _vp, _vp],
        "moe_layer_bwd": [P(Shape), P(BwdArgs), P(Saved), _vp, _vp],
        "moe_checks_read": [P(i32), i32],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    _lib = lib
    return lib


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn: str, rc: int):
    if rc != 0:
        raise MoEError(fn, rc)


def shape(T, d, E, k, f, prec=BF16) -> Shape:
    return Shape(int(T), int(d), int(E), int(k), int(f), int(prec))


# ------------------------------------------------------------------ set-up
_inited = set()


def init(device: int | None = None):
    import torch
    dev = torch.cuda.current_device() if device is None else int(device)
    if dev in _inited:
        return
    with torch.cuda.device(dev):
        _check("moe_init", load().moe_init(dev))
    _inited.add(dev)


def rows_max(s: Shape) -> int:
    v = ctypes.c_int64()
    _check("moe_rows_max", load().moe_rows_max(ctypes.byref(s), ctypes.byref(v)))
    return v.value


def workspace_size(s: Shape) -> int:
    v = ctypes.c_size_t()
    _check("moe_workspace_size", load().moe_workspace_size(ctypes.byref(s), ctypes.byref(v)))
    return v.value


def checks_read(reset: bool = True) -> int:
    """moe_checks_read: the OR of the checks build's bounds-check words (0 when
    no index left its buffer); raises MoEError(MOE_ERR_UNSUPPORTED) on the
    normal build."""
    v = ctypes.c_int32()
    _check("moe_checks_read", load().moe_checks_read(ctypes.byref(v), int(bool(reset))))
    return v.value


# ---- guard bands (checks mode): every buffer of allocate() sits between two
# 4 KB bands of a known byte pattern, verified by check_canaries()
GUARD_BYTES = 4096
GUARD_BYTE = 0xA5
_guarded = {}   # id of a handed-out buffer -> its whole allocation (bands included)


def _alloc(shape, dtype, device, zero=False):
    import torch
    if not CHECKS:
        return (torch.zeros if zero else torch.empty)(shape, dtype=dtype, device=device)
    import math
    import weakref
    n = math.prod(shape) * torch.empty((), dtype=dtype).element_size()
    base = torch.full((n + 2 * GUARD_BYTES,), GUARD_BYTE, dtype=torch.uint8, device=device)
    mid = base[GUARD_BYTES:GUARD_BYTES + n]
    if zero:
        mid.zero_()
    out = mid.view(dtype).view(shape)
    key = id(out)
    _guarded[key] = base
    weakref.finalize(out, _guarded.pop, key, None)   # forgotten with the buffer
    return out


def check_canaries() -> list:
    """Checks mode: the guard bands of every live buffer from allocate() still
    hold their pattern.  Returns a description of each band that was written."""
    bad = []
    for base in list(_guarded.values()):
        for name, band in (("front", base[:GUARD_BYTES]), ("back", base[-GUARD_BYTES:])):
            changed = int((band != GUARD_BYTE).sum().item())
            if changed:
                bad.append(f"{changed} byte(s) of the {name} guard of a {base.numel() - 2 * GUARD_BYTES}"
                           f"-byte buffer were written")
    return bad


def clear_error(ws, stream=None):
    _check("moe_clear_error", load().moe_clear_error(_ptr(ws), _stream(stream)))


def debug_inject_stall(mode: int) -> int:
    """Test hook: 1 makes the next grouped-GEMM launches stall on purpose (their
    bounded waits time out and report MOE_DEVERR_TIMEOUT); 0 turns it off."""
    rc = load().moe_debug_inject_stall(int(mode))
    if rc < 0:
        raise MoEError("moe_debug_inject_stall", rc)
    return rc


def load_balance(s: Shape, logits, counts, lb_stats, ws, stream=None):
    """moe_load_balance: lb_stats[0] = LBL, lb_stats[1 + e] = P_e."""
    _check("moe_load_balance", load().moe_load_balance(ctypes.byref(s), _ptr(logits), _ptr(counts),
                                                       _ptr(lb_stats), _ptr(ws), _stream(stream)))


def profile_start(op: int):
    """moe_profile_start: time every following launch of grouped-GEMM `op`."""
    _check("moe_profile_start", load().moe_profile_start(int(op)))


def profile_stop():
    """moe_profile_stop: (summed milliseconds, number of timed launches)."""
    ms = ctypes.c_float(0.0)
    n = ctypes.c_int32(0)
    _check("moe_profile_stop", load().moe_profile_stop(ctypes.byref(ms), ctypes.byref(n)))
    return float(ms.value), int(n.value)


def read_error(ws, stream=None) -> int:
    v = ctypes.c_int32()
    _check("moe_read_error", load().moe_read_error(_ptr(ws), ctypes.byref(v), _stream(stream)))
    return v.value


# ------------------------------------------------------------------ stage calls
def route(s, x, w_router, logit_bias, logits, topk_idx, gates, counts, offsets, tile_offsets,
          slot_of_route, route_of_slot, ws, stream=None):
    _check("moe_route", load().moe_route(
        ctypes.byref(s), _ptr(x), _ptr(w_router), _ptr(logit_bias), _ptr(logits), _ptr(topk_idx),
        _ptr(gates), _ptr(counts), _ptr(offsets), _ptr(tile_offsets), _ptr(slot_of_route),
        _ptr(route_of_slot), _ptr(ws), _stream(stream)))


def route_noalloc(s, x, w_router, logit_bias, logits, topk_idx, gates, counts, offsets,
                  tile_offsets, slot_of_route, route_of_slot, dev_error=None, stream=None):
    """moe_route without a workspace: for callers that cannot allocate device
    memory (see include/moe.h); scratch lives in the library's static array."""
    _check("moe_route_noalloc", load().moe_route_noalloc(
        ctypes.byref(s), _ptr(x), _ptr(w_router), _ptr(logit_bias), _ptr(logits), _ptr(topk_idx),
        _ptr(gates), _ptr(counts), _ptr(offsets), _ptr(tile_offsets), _ptr(slot_of_route),
        _ptr(route_of_slot), _ptr(dev_error), _stream(stream)))


def dispatch(s, x, slot_of_route, counts, tile_offsets, xd, xd_scales=None, stream=None,
             xd_dq=None):
    _check("moe_dispatch", load().moe_dispatch(
        ctypes.byref(s), _ptr(x), _ptr(slot_of_route), _ptr(counts), _ptr(tile_offsets), _ptr(xd),
        _ptr(xd_scales), _ptr(xd_dq), _stream(stream)))


def quantize_mxfp8(batch, rows, cols, block_axis, src, q, scales, stream=None):
    _check("moe_quantize_mxfp8", load().moe_quantize_mxfp8(
        int(batch), int(rows), int(cols), int(block_axis), _ptr(src), _ptr(q), _ptr(scales),
        _stream(stream)))


def dequantize_mxfp8(rows, K, q, scales, out, stream=None):
    _check("moe_dequantize_mxfp8", load().moe_dequantize_mxfp8(
        int(rows), int(K), _ptr(q), _ptr(scales), _ptr(out), _stream(stream)))


def build_mx_weights(s, w_gate, w_up, w_down, cache: dict, stream=None):
    c = MxWeights(**{k: _ptr(cache[k]) for k in MX_WEIGHT_FIELDS})
    _check("moe_build_mx_weights", load().moe_build_mx_weights(
        ctypes.byref(s), _ptr(w_gate), _ptr(w_up), _ptr(w_down), ctypes.byref(c), _stream(stream)))


def grouped_gemm(s, op, ws, stream=None, **kw):
    a = GemmArgs(**{k: _ptr(v) for k, v in kw.items()})
    _check("moe_grouped_gemm", load().moe_grouped_gemm(ctypes.byref(s), int(op), ctypes.byref(a),
                                                       _ptr(ws), _stream(stream)))


def combine(s, y, gates, slot_of_route, out, stream=None):
    _check("moe_combine", load().moe_combine(ctypes.byref(s), _ptr(y), _ptr(gates),
                                             _ptr(slot_of_route), _ptr(out), _stream(stream)))


def combine_bwd(s, d_out, y, gates, topk_idx, slot_of_route, counts, tile_offsets, dy, d_gates,
                dlogits, stream=None, dy_q=None, dy_scales=None):
    _check("moe_combine_bwd", load().moe_combine_bwd(
        ctypes.byref(s), _ptr(d_out), _ptr(y), _ptr(gates), _ptr(topk_idx), _ptr(slot_of_route),
        _ptr(counts), _ptr(tile_offsets), _ptr(dy), _ptr(d_gates), _ptr(dlogits), _ptr(dy_q),
        _ptr(dy_scales), _stream(stream)))


def dispatch_bwd(s, dxd, slot_of_route, topk_idx, dlogits, w_router, dx, stream=None):
    _check("moe_dispatch_bwd", load().moe_dispatch_bwd(
        ctypes.byref(s), _ptr(dxd), _ptr(slot_of_route), _ptr(topk_idx), _ptr(dlogits),
        _ptr(w_router), _ptr(dx), _stream(stream)))


def router_bwd(s, x, dlogits, route_of_slot, counts, tile_offsets, dw_router, ws, stream=None):
    _check("moe_router_bwd", load().moe_router_bwd(
        ctypes.byref(s), _ptr(x), _ptr(dlogits), _ptr(route_of_slot), _ptr(counts),
        _ptr(tile_offsets), _ptr(dw_router), _ptr(ws), _stream(stream)))


def layer_fwd(s, fwd: FwdArgs, saved: Saved, ws, stream=None):
    _check("moe_layer_fwd", load().moe_layer_fwd(ctypes.byref(s), ctypes.byref(fwd),
                                                 ctypes.byref(saved), _ptr(ws), _stream(stream)))


def layer_bwd(s, bwd: BwdArgs, saved: Saved, ws, stream=None):
    _check("moe_layer_bwd", load().moe_layer_bwd(ctypes.byref(s), ctypes.byref(bwd),
                                                 ctypes.byref(saved), _ptr(ws), _stream(stream)))


# ------------------------------------------------------------------ buffers
@dataclass
class LayerBuffers:
    """Caller-owned device buffers of one layer shape (torch allocates them)."""

    shape: Shape
    rows_max: int
    ws: object
    saved: dict
    grads: dict
    mx_weights: dict | None = None
    mx: dict | None = None

    def saved_struct(self) -> Saved:
        return Saved(**{k: _ptr(v) for k, v in self.saved.items()})

    def mx_structs(self):
        """(MxWeights, MxBuffers) ctypes structs, or (None, None) in BF16 mode.
        The structs are kept on the object so their addresses stay valid."""
        if self.mx is None:
            return None, None
        self._mxw = MxWeights(**{k: _ptr(self.mx_weights[k]) for k in MX_WEIGHT_FIELDS})
        self._mxb = MxBuffers(**{k: _ptr(self.mx.get(k)) for k in MX_BUFFER_FIELDS})
        return ctypes.addressof(self._mxw), ctypes.addressof(self._mxb)


def allocate(s: Shape, device=None, with_grads: bool = True,
             load_balance: bool = False) -> LayerBuffers:
    """Allocate every buffer moe_layer_fwd / moe_layer_bwd need for shape `s`
    (with load_balance, saved["lb_stats"] receives the forward's
    load-balancing statistics)."""
    import torch
    dev = torch.device("cuda", torch.cuda.current_device() if device is None else device)
    T, d, E, k, f = s.T, s.d_model, s.n_experts, s.top_k, s.d_ff
    n = rows_max(s)
    bf = dict(dtype=torch.bfloat16, device=dev)
    i32 = dict(dtype=torch.int32, device=dev)
    f32 = dict(dtype=torch.float32, device=dev)
    ws = _alloc((workspace_size(s),), torch.uint8, dev, zero=True)
    u8 = dict(dtype=torch.uint8, device=dev)
    mx = s.prec == MXFP8

    def new(*shape, dtype, device):   # guard bands around it in checks mode
        return _alloc(shape, dtype, device)

    saved = {
        "logits": new(T, E, **f32), "topk_idx": new(T, k, **i32),
        "gates": new(T, k, **f32), "counts": new(E, **i32),
        "offsets": new(E + 1, **i32), "tile_offsets": new(E + 1, **i32),
        "slot_of_route": new(T * k, **i32), "route_of_slot": new(n, **i32),
        "xd": None if mx else new(n, d, **bf), "h": new(n, f, **bf),
        "u": new(n, f, **bf), "a": None if mx else new(n, f, **bf),
        "y": new(n, d, **bf),
        "lb_stats": new(E + 1, **f32) if load_balance else None,
    }
    grads = {}
    if with_grads:
        grads = {
            "dx": new(T, d, **bf), "dw_router": new(E, d, **f32),
            "dw_gate": new(E, f, d, **f32), "dw_up": new(E, f, d, **f32),
            "dw_down": new(E, d, f, **f32), "d_gates": new(T, k, **f32),
            "dlogits": new(T, E, **f32), "dy": new(n, d, **bf),
            "dh": new(n, f, **bf), "du": new(n, f, **bf),
            "dxd": new(n, d, **bf),
        }
    mxw = mxb = None
    if mx:
        mxw = {"gu_q": new(E, 2 * f, d, **u8), "gu_s": new(E * 2 * f * d // 32, **u8),
               "down_q": new(E, d, f, **u8), "down_s": new(E * d * f // 32, **u8),
               "downT_q": new(E, f, d, **u8), "downT_s": new(E * f * d // 32, **u8),
               "gateT_q": new(E, d, f, **u8), "gateT_s": new(E * d * f // 32, **u8),
               "upT_q": new(E, d, f, **u8), "upT_s": new(E * d * f // 32, **u8)}
        mxb = {"xd_q": new(n, d, **u8), "xd_s": new(n * d // 32, **u8),
               "a_q": new(n, f, **u8), "a_s": new(n * f // 32, **u8)}
        if with_grads:
            mxb.update({"dy_q": new(n, d, **u8), "dy_s": new(n * d // 32, **u8),
                        "dh_q": new(n, f, **u8), "dh_s": new(n * f // 32, **u8),
                        "du_q": new(n, f, **u8), "du_s": new(n * f // 32, **u8),
                        "xd_dq": new(n, d, **bf), "a_dq": new(n, f, **bf)})
    return LayerBuffers(s, n, ws, saved, grads, mxw, mxb)


def forward(buf: LayerBuffers, x, w_router, logit_bias, w_gate, w_up, w_down, out, stream=None):
    """moe_layer_fwd.  MXFP8 shapes use buf.mx_weights (fill them with
    build_mx_weights whenever the bf16 weights change)."""
    mw, mb = buf.mx_structs()
    fa = FwdArgs(x=_ptr(x), w_router=_ptr(w_router), logit_bias=_ptr(logit_bias),
                 w_gate=_ptr(w_gate), w_up=_ptr(w_up), w_down=_ptr(w_down), out=_ptr(out),
                 mx_weights=mw, mx=mb)
    layer_fwd(buf.shape, fa, buf.saved_struct(), buf.ws, stream)


def backward(buf: LayerBuffers, d_out, x, w_router, w_gate, w_up, w_down, stream=None,
             recompute: bool = False, lb_coef: float = 0.0):
    """moe_layer_bwd.  recompute=True re-runs dispatch and both expert GEMMs
    from x and the saved routing metadata instead of reading the saved
    activations; lb_coef adds lb_coef * LBL (the load-balancing scalar) to the
    loss."""
    g = buf.grads
    mw, mb = buf.mx_structs()
    ba = BwdArgs(d_out=_ptr(d_out), x=_ptr(x), w_router=_ptr(w_router), w_gate=_ptr(w_gate),
                 w_up=_ptr(w_up), w_down=_ptr(w_down), mx_weights=mw, mx=mb,
                 recompute=1 if recompute else 0, lb_coef=float(lb_coef),
                 **{k: _ptr(v) for k, v in g.items()})
    layer_bwd(buf.shape, ba, buf.saved_struct(), buf.ws, stream)
