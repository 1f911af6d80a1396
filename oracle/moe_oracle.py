"""Oracle for the MoE expert layer: a plain, slow CPU definition (TEST INFRASTRUCTURE).

This module is test infrastructure, not product code.  Only the tests, the
package smoke check and the benchmark's CPU-baseline leg may import it.  The
CUDA library never imports, links or calls it, and it shares no code with the
CUDA library.

What it computes (sources)
--------------------------
"Supercharging Olmo-core for Efficient and Scalable MoE Training" (Abstract)
states the problem: a router sends every token to a few experts, a rowwise
dispatch writes each token row straight into its expert's buffer with no
permutation pass, routing counts/offsets stay on the device, a device-scheduled
grouped GEMM runs the uneven per-expert shapes, and the results are combined.
Section 24.1 of the report adds that keeping the metadata on the device does not
change the routing calculation.  The blog "Olmo-core 3: an open training stack
for trillion-parameter MoE" (section "Olmo-core 3's answer: experts resident,
data routed") repeats this, adds that the grouped GEMM runs without padding every
expert to a common capacity, and that MXFP8 is an 8-bit format with shared block
scales.  Section 24 Evidence 10 gives the MXFP8 row payload (33/32 byte per
value, i.e. one 1-byte scale per 32 one-byte values) and the two weight caches.

The pages never write the layer's arithmetic out.  The readings used here (the
plainest ones the pages support) are:

* router: logits = x . W_r^T + bias, in fp32 on the device (here fp64);
* softmax over all experts, top-k chosen by logit (descending; equal logits go
  to the lower expert id), gates = the selected softmax probabilities
  renormalised to sum to one;
* expert e is a SwiGLU MLP without biases:
  y = (silu(x W_gate_e^T) * (x W_up_e^T)) W_down_e^T, silu(h) = h / (1 + e^-h);
* the gate multiplies in the combine: out[t] = sum_j g_tj * y_{e_tj}(x[t]);
* expert buffers are contiguous and expert e starts at row
  row_offsets[e] = BM * (number of BM-row tiles of the experts before e); with
  BM = 1 this is the plain exclusive scan of the counts.  Within an expert,
  rows are in ascending route order (token t, then choice j);
* load balancing (optional): the Switch-style scalar LBL = E * sum_e f_e P_e,
  f_e = fraction of routes of expert e (hard counts, not differentiated),
  P_e = mean full-softmax probability of expert e (Section 24.2, Evidence 9);
* backward: the exact gradient for a fixed top-k selection (the selection
  itself is piecewise constant);
* MXFP8: E4M3 values with one E8M0 (power-of-two) scale per 32 consecutive
  values along the contraction axis; the scale is the smallest power of two
  2^s with amax <= 448 * 2^s (s clamped to [-127, 127], s = 0 for an all-zero
  block), values are x / 2^s rounded to nearest-even E4M3, saturating at 448.

Precision: every input (bf16 bits or fp32 values) is widened exactly to float64
and all arithmetic is float64.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "as_f64",
    "router_logits",
    "softmax_topk_gates",
    "expert_counts",
    "exclusive_scan",
    "tile_layout",
    "assign_slots",
    "dispatch",
    "silu",
    "silu_grad",
    "expert_ffn_forward",
    "combine",
    "combine_backward",
    "expert_ffn_backward",
    "dispatch_backward",
    "router_backward",
    "layer_forward",
    "layer_backward",
    "dense_forward",
    "E4M3_VALUES",
    "e4m3_encode",
    "mx_scale_exponent",
    "quantize_mxfp8",
    "dequantize_mxfp8",
    "layer_forward_mxfp8",
    "layer_backward_mxfp8",
]


# --------------------------------------------------------------------------
# input widening
# --------------------------------------------------------------------------
def as_f64(a) -> np.ndarray:
    """Widen an input exactly to float64.

    uint16 arrays are bfloat16 bit patterns (the upper half of an IEEE fp32);
    float arrays are taken as they are.
    """
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


# --------------------------------------------------------------------------
# a1-a3: router, top-k, counts, offsets, slots
# --------------------------------------------------------------------------
def router_logits(x, w_router, bias=None) -> np.ndarray:
    """Router projection: logits[t, e] = sum_i x[t, i] * W_r[e, i] + bias[t, e].

    Routing is named as a subsystem of the stack ("Olmo-core DDP training
    stack", Section 2 closing paragraph: routing and sparse routing) but not
    written out; this is the plain linear router.  W_r is [E, d].
    """
    logits = as_f64(x) @ as_f64(w_router).T
    if bias is not None:
        logits = logits + as_f64(bias)
    return logits


def softmax_topk_gates(logits, k: int):
    """Softmax over all experts, top-k by logit, renormalised gates.

    Returns (topk_idx [T, k] int32, gates [T, k] float64).  Choice j of token t
    is the j-th largest logit; equal logits are ordered by ascending expert id
    (a stable sort of the negated logits).  gates = p_sel / sum(p_sel) where p
    is the softmax over all E experts.  Non-finite logits raise.
    """
    L = as_f64(logits)
    if not np.all(np.isfinite(L)):
        raise FloatingPointError("non-finite router logit")
    T, E = L.shape
    if not 1 <= k <= E:
        raise ValueError("need 1 <= k <= E")
    m = L.max(axis=1, keepdims=True)
    p = np.exp(L - m)
    p = p / p.sum(axis=1, keepdims=True)
    order = np.argsort(-L, axis=1, kind="stable")
    idx = order[:, :k]
    p_sel = np.take_along_axis(p, idx, axis=1)
    gates = p_sel / p_sel.sum(axis=1, keepdims=True)
    return idx.astype(np.int32), gates


def expert_counts(topk_idx, E: int) -> np.ndarray:
    """counts[e] = number of routes (t, j) whose expert is e.

    These are the routing counts the original path copied to the host
    (Section 24, Evidence 3 / Figure 74) and the new path keeps on the device.
    """
    counts = np.zeros(E, dtype=np.int64)
    for e in np.asarray(topk_idx).ravel().tolist():
        counts[e] += 1
    return counts


def exclusive_scan(counts) -> np.ndarray:
    """offsets[0] = 0, offsets[e + 1] = offsets[e] + counts[e]  (length E + 1)."""
    c = np.asarray(counts, dtype=np.int64)
    out = np.zeros(c.size + 1, dtype=np.int64)
    run = 0
    for e, v in enumerate(c.tolist()):
        run += v
        out[e + 1] = run
    return out


def tile_layout(counts, bm: int):
    """Tile-aligned expert buffers for a grouped GEMM with BM-row tiles.

    tiles[e] = ceil(counts[e] / BM); tile_offsets = exclusive scan of tiles;
    row_offsets = BM * tile_offsets.  Expert e owns rows
    [row_offsets[e], row_offsets[e + 1]) of the dispatched buffer; the last
    row_offsets[e + 1] - row_offsets[e] - counts[e] of them are zero padding.
    This is not padding to a common capacity (the blog, section "Olmo-core 3's
    answer"): each expert is padded by less than one tile.
    """
    c = np.asarray(counts, dtype=np.int64)
    tiles = (c + bm - 1) // bm
    tile_offsets = exclusive_scan(tiles)
    return tile_offsets, bm * tile_offsets


def assign_slots(topk_idx, row_offsets):
    """Stable rowwise slot assignment.

    Walk the routes in ascending (token, choice) order; route r = t * k + j of
    expert e gets slot row_offsets[e] + (number of earlier routes of e).
    Returns slot_of_route [T*k] and route_of_slot [row_offsets[E]] (-1 marks a
    padding row).  Abstract: each token row is written directly into its
    expert's buffer.
    """
    idx = np.asarray(topk_idx)
    T, k = idx.shape
    ro = [int(v) for v in np.asarray(row_offsets).tolist()]
    cursor = [0] * (len(ro) - 1)
    slot_of_route = np.empty(T * k, dtype=np.int64)
    route_of_slot = np.full(ro[-1], -1, dtype=np.int64)
    for r, e in enumerate(idx.ravel().tolist()):
        s = ro[e] + cursor[e]
        cursor[e] += 1
        slot_of_route[r] = s
        route_of_slot[s] = r
    return slot_of_route, route_of_slot


def dispatch(x, slot_of_route, k: int, n_rows: int) -> np.ndarray:
    """Rowwise dispatch: Xd[slot_of_route[t*k + j]] = x[t]; padding rows are 0."""
    X = as_f64(x)
    Xd = np.zeros((n_rows, X.shape[1]), dtype=np.float64)
    for r, s in enumerate(np.asarray(slot_of_route).tolist()):
        Xd[s] = X[r // k]
    return Xd


# --------------------------------------------------------------------------
# a5-a7: expert SwiGLU MLPs and the weighted combine
# --------------------------------------------------------------------------
def silu(h):
    """silu(h) = h / (1 + exp(-h))."""
    with np.errstate(over="ignore"):
        return h / (1.0 + np.exp(-h))


def silu_grad(h):
    """d silu / dh = sigma(h) * (1 + h * (1 - sigma(h)))."""
    with np.errstate(over="ignore"):
        s = 1.0 / (1.0 + np.exp(-h))
    return s * (1.0 + h * (1.0 - s))


def expert_ffn_forward(Xd, w_gate, w_up, w_down, row_offsets):
    """Per-expert SwiGLU on the expert's contiguous rows.

    H_e = Xd_e W_gate_e^T, U_e = Xd_e W_up_e^T, A_e = silu(H_e) * U_e,
    Y_e = A_e W_down_e^T.  W_gate, W_up are [E, f, d]; W_down is [E, d, f].
    Returns H, U, A [rows, f] and Y [rows, d].
    """
    Xd = as_f64(Xd)
    ro = np.asarray(row_offsets).tolist()
    E = len(ro) - 1
    f = np.asarray(w_gate).shape[1]
    n = Xd.shape[0]
    H = np.zeros((n, f))
    U = np.zeros((n, f))
    A = np.zeros((n, f))
    Y = np.zeros((n, Xd.shape[1]))
    for e in range(E):
        a, b = ro[e], ro[e + 1]
        if a == b:
            continue
        Xe = Xd[a:b]
        H[a:b] = Xe @ as_f64(w_gate[e]).T
        U[a:b] = Xe @ as_f64(w_up[e]).T
        A[a:b] = silu(H[a:b]) * U[a:b]
        Y[a:b] = A[a:b] @ as_f64(w_down[e]).T
    return H, U, A, Y


def combine(Y, gates, slot_of_route, T: int, k: int) -> np.ndarray:
    """Weighted combine: out[t] = sum_j gates[t, j] * Y[slot_of_route[t*k + j]]."""
    Y = as_f64(Y)
    g = as_f64(gates).reshape(T, k)
    slots = np.asarray(slot_of_route).reshape(T, k)
    out = np.zeros((T, Y.shape[1]))
    for j in range(k):
        out += g[:, j:j + 1] * Y[slots[:, j]]
    return out


# --------------------------------------------------------------------------
# a8-a14: backward
# --------------------------------------------------------------------------
def combine_backward(d_out, Y, gates, slot_of_route, T: int, k: int, n_rows: int):
    """Gradient of the combine.

    d_gates[t, j] = <dOut[t], Y[slot(t, j)]>, dY[slot(t, j)] = gates[t, j] * dOut[t]
    (padding rows of dY are zero).
    """
    dO = as_f64(d_out)
    Y = as_f64(Y)
    g = as_f64(gates).reshape(T, k)
    slots = np.asarray(slot_of_route).reshape(T, k)
    d_gates = np.zeros((T, k))
    dY = np.zeros((n_rows, dO.shape[1]))
    for j in range(k):
        d_gates[:, j] = np.einsum("td,td->t", dO, Y[slots[:, j]])
        dY[slots[:, j]] = g[:, j:j + 1] * dO
    return d_gates, dY


def expert_ffn_backward(dY, Xd, H, U, A, w_gate, w_up, w_down, row_offsets):
    """Per-expert SwiGLU backward.

    dA_e = dY_e W_down_e; dH = dA * U * silu'(H); dU = dA * silu(H);
    dXd_e = dH_e W_gate_e + dU_e W_up_e;
    dW_down_e = dY_e^T A_e; dW_gate_e = dH_e^T Xd_e; dW_up_e = dU_e^T Xd_e.
    Experts without rows get exact-zero weight gradients.
    """
    dY = as_f64(dY)
    Xd = as_f64(Xd)
    ro = np.asarray(row_offsets).tolist()
    E = len(ro) - 1
    f, d = np.asarray(w_gate).shape[1:]
    n = Xd.shape[0]
    dH = np.zeros((n, f))
    dU = np.zeros((n, f))
    dXd = np.zeros((n, d))
    dWg = np.zeros((E, f, d))
    dWu = np.zeros((E, f, d))
    dWd = np.zeros((E, d, f))
    for e in range(E):
        a, b = ro[e], ro[e + 1]
        if a == b:
            continue
        Wg, Wu, Wd = as_f64(w_gate[e]), as_f64(w_up[e]), as_f64(w_down[e])
        dA = dY[a:b] @ Wd
        h = H[a:b]
        dH[a:b] = dA * U[a:b] * silu_grad(h)
        dU[a:b] = dA * silu(h)
        dXd[a:b] = dH[a:b] @ Wg + dU[a:b] @ Wu
        dWd[e] = dY[a:b].T @ A[a:b]
        dWg[e] = dH[a:b].T @ Xd[a:b]
        dWu[e] = dU[a:b].T @ Xd[a:b]
    return {"dH": dH, "dU": dU, "dXd": dXd, "dW_gate": dWg, "dW_up": dWu, "dW_down": dWd}


def dispatch_backward(dXd, slot_of_route, T: int, k: int) -> np.ndarray:
    """Gradient of the dispatch (a gather-sum): dx[t] = sum_j dXd[slot(t, j)]."""
    dXd = as_f64(dXd)
    slots = np.asarray(slot_of_route).reshape(T, k)
    dx = np.zeros((T, dXd.shape[1]))
    for j in range(k):
        dx += dXd[slots[:, j]]
    return dx


def load_balance(logits, topk_idx, E: int):
    """Switch-style load-balancing scalar of a top-k router.

    "Section 24: Conclusion" of the report (Section 24.2, Evidence 9) describes
    the Switch-style scalar as a cross-term between soft router scores and hard
    expert counts.  Reading: the hard part is the fraction of routes each expert
    receives, f_e = count_e / (T k); the soft part is the mean router
    probability, P_e = mean over tokens of the softmax over all E experts; the
    scalar is LBL = E * sum_e f_e P_e (1 when the scores are uniform).
    Returns (LBL, P [E], f [E]).
    """
    L = as_f64(logits)
    idx = np.asarray(topk_idx)
    T, k = idx.shape
    p = np.exp(L - L.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    f = np.bincount(idx.ravel(), minlength=E).astype(np.float64) / (T * k)
    P = p.mean(axis=0)
    return float(E * np.dot(f, P)), P, f


def load_balance_dlogits(logits, topk_idx, E: int, coef: float) -> np.ndarray:
    """d(coef * LBL)/dlogits, the counts held fixed (they are not differentiable):
    coef * E / T * p[t, e] * (f_e - sum_e' f_e' p[t, e'])."""
    L = as_f64(logits)
    T = L.shape[0]
    _, _, f = load_balance(L, topk_idx, E)
    p = np.exp(L - L.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    s = p @ f
    return coef * E / T * p * (f[None, :] - s[:, None])


def router_backward(d_gates, gates, topk_idx, E: int, x=None, w_router=None, dlogits_extra=None):
    """Gradient through the renormalised softmax and the router projection.

    For the selected experts g_j = exp(l_j) / sum_sel exp(l_i), so
    dl_j = g_j * (dg_j - sum_i g_i dg_i); unselected logits get zero (the full
    softmax denominator cancels in the renormalisation).  With a router weight,
    dx_router = dlogits W_r and dW_r = dlogits^T x.  `dlogits_extra` (a dense
    [T, E] term, e.g. the load-balancing loss's) is added to dlogits first.
    Returns dlogits [T, E] and, when W_r is given, (dx_router [T, d], dW_r [E, d]).
    """
    dg = as_f64(d_gates)
    g = as_f64(gates)
    idx = np.asarray(topk_idx)
    T, k = idx.shape
    inner = np.sum(g * dg, axis=1, keepdims=True)
    dl_sel = g * (dg - inner)
    dlogits = np.zeros((T, E))
    for j in range(k):
        dlogits[np.arange(T), idx[:, j]] += dl_sel[:, j]
    if dlogits_extra is not None:
        dlogits = dlogits + as_f64(dlogits_extra)
    out = {"dlogits": dlogits}
    if w_router is not None:
        out["dx_router"] = dlogits @ as_f64(w_router)
        out["dW_router"] = dlogits.T @ as_f64(x)
    return out


# --------------------------------------------------------------------------
# the whole layer
# --------------------------------------------------------------------------
def layer_forward(x, w_router, bias, w_gate, w_up, w_down, k: int, bm: int = 128, logits=None):
    """Forward of the layer: route, dispatch, grouped SwiGLU, combine.

    If `logits` is given it replaces the router projection (used to compare the
    routing of a device run on the device's own fp32 logits).
    """
    if logits is None:
        logits = router_logits(x, w_router, bias)
    logits = as_f64(logits)
    T, E = logits.shape
    idx, gates = softmax_topk_gates(logits, k)
    counts = expert_counts(idx, E)
    offsets = exclusive_scan(counts)
    tile_offsets, row_offsets = tile_layout(counts, bm)
    slot_of_route, route_of_slot = assign_slots(idx, row_offsets)
    n_rows = int(row_offsets[-1])
    Xd = dispatch(x, slot_of_route, k, n_rows)
    H, U, A, Y = expert_ffn_forward(Xd, w_gate, w_up, w_down, row_offsets)
    out = combine(Y, gates, slot_of_route, T, k)
    return {
        "logits": logits, "topk_idx": idx, "gates": gates, "counts": counts,
        "offsets": offsets, "tile_offsets": tile_offsets, "row_offsets": row_offsets,
        "slot_of_route": slot_of_route, "route_of_slot": route_of_slot,
        "Xd": Xd, "H": H, "U": U, "A": A, "Y": Y, "out": out, "k": k, "bm": bm,
    }


def layer_backward(fwd, d_out, x, w_router, w_gate, w_up, w_down, lb_coef: float = 0.0):
    """Backward of the layer for upstream gradient dOut [T, d], plus lb_coef
    times the load-balancing scalar's gradient when lb_coef is not 0."""
    T, k = fwd["topk_idx"].shape
    E = fwd["logits"].shape[1]
    n_rows = fwd["Xd"].shape[0]
    d_gates, dY = combine_backward(d_out, fwd["Y"], fwd["gates"], fwd["slot_of_route"], T, k, n_rows)
    g = expert_ffn_backward(dY, fwd["Xd"], fwd["H"], fwd["U"], fwd["A"], w_gate, w_up, w_down,
                            fwd["row_offsets"])
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


def dense_forward(x, w_router, bias, w_gate, w_up, w_down, k: int, logits=None):
    """Brute-force restatement without dispatch: every expert on every token.

    out[t] = sum_e G[t, e] * FFN_e(x[t]) with G the [T, E] gate matrix (zero for
    unselected experts).  Only for tiny shapes.
    """
    if logits is None:
        logits = router_logits(x, w_router, bias)
    idx, gates = softmax_topk_gates(logits, k)
    X = as_f64(x)
    T, E = logits.shape
    G = np.zeros((T, E))
    for j in range(k):
        G[np.arange(T), idx[:, j]] = gates[:, j]
    out = np.zeros_like(X)
    for e in range(E):
        h = X @ as_f64(w_gate[e]).T
        u = X @ as_f64(w_up[e]).T
        out += G[:, e:e + 1] * ((silu(h) * u) @ as_f64(w_down[e]).T)
    return out


# --------------------------------------------------------------------------
# a15: MXFP8 (OCP MX: E4M3 elements, E8M0 block scales, 32 values per block)
# --------------------------------------------------------------------------
def _e4m3_table() -> np.ndarray:
    vals = np.empty(256, dtype=np.float64)
    for c in range(256):
        s = -1.0 if c & 0x80 else 1.0
        e = (c >> 3) & 0xF
        m = c & 0x7
        if e == 0xF and m == 0x7:
            vals[c] = np.nan
        elif e == 0:
            vals[c] = s * (m / 8.0) * 2.0 ** -6
        else:
            vals[c] = s * (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return vals


E4M3_VALUES = _e4m3_table()
_E4M3_POS = E4M3_VALUES[:127]          # codes 0..126: 0 .. 448, ascending
E4M3_MAX = 448.0


def e4m3_encode(v) -> np.ndarray:
    """Round to the nearest E4M3 value, ties to the even code, saturating at +-448.

    The sign bit is copied from the input (so -0.0 and negative values that
    round to zero give code 0x80).
    """
    v = as_f64(v)
    a = np.abs(v)
    sat = a >= E4M3_MAX
    i = np.searchsorted(_E4M3_POS, np.minimum(a, E4M3_MAX), side="left")
    i = np.clip(i, 0, 126)
    hi = i
    lo = np.maximum(i - 1, 0)
    exact = _E4M3_POS[hi] == a
    d_lo = a - _E4M3_POS[lo]
    d_hi = _E4M3_POS[hi] - a
    pick = np.where(d_lo < d_hi, lo, np.where(d_hi < d_lo, hi, np.where(lo % 2 == 0, lo, hi)))
    code = np.where(exact, hi, pick)
    code = np.where(sat, 126, code)
    code = np.where(a == 0, 0, code)
    sign = np.signbit(v)
    return (code.astype(np.uint8) | np.where(sign, 0x80, 0).astype(np.uint8)).astype(np.uint8)


def mx_scale_exponent(amax) -> np.ndarray:
    """Smallest integer s with amax <= 448 * 2^s, clamped to [-127, 127]; 0 when amax == 0."""
    amax = as_f64(amax)
    _, e = np.frexp(np.where(amax > 0, amax, 1.0))   # amax = m * 2^e, m in [0.5, 1)
    s = e.astype(np.int64) - 10                        # 448 * 2^(e-10) < 2^(e-1) <= amax
    for _ in range(3):                                 # at most two steps are ever needed
        s = np.where(amax > E4M3_MAX * np.ldexp(1.0, s), s + 1, s)
    s = np.clip(s, -127, 127)
    return np.where(amax > 0, s, 0).astype(np.int64)


def quantize_mxfp8(a, block: int = 32):
    """MXFP8 quantisation along the last axis.

    Returns (codes uint8 [..., K], scales uint8 [..., K/32]) with scale byte =
    s + 127 (E8M0) and code = E4M3(x / 2^s).
    """
    a = as_f64(a)
    K = a.shape[-1]
    if K % block:
        raise ValueError("last axis must be a multiple of the block size")
    blk = a.reshape(a.shape[:-1] + (K // block, block))
    amax = np.max(np.abs(blk), axis=-1)
    s = mx_scale_exponent(amax)
    scaled = blk / np.ldexp(1.0, s)[..., None]
    codes = e4m3_encode(scaled).reshape(a.shape)
    return codes, (s + 127).astype(np.uint8)


def dequantize_mxfp8(codes, scales, block: int = 32) -> np.ndarray:
    codes = np.asarray(codes)
    K = codes.shape[-1]
    vals = E4M3_VALUES[codes].reshape(codes.shape[:-1] + (K // block, block))
    s = np.asarray(scales).astype(np.int64) - 127
    return (vals * np.ldexp(1.0, s)[..., None]).reshape(codes.shape)


def _qdq(a):
    return dequantize_mxfp8(*quantize_mxfp8(a))


def layer_forward_mxfp8(x, w_router, bias, w_gate, w_up, w_down, k: int, bm: int = 128, logits=None):
    """Forward with the MXFP8 expert GEMMs.

    Reading of Section 24 Evidence 10 ("two weight caches", 33/32-byte payload)
    and the blog's MXFP8 paragraph: x is quantised once per token along d before
    the dispatch (so the dispatched payload is MXFP8), the forward weight cache
    quantises W_gate/W_up along d and W_down along f, and the SwiGLU output A is
    quantised along f before the second GEMM.  Routing and the combine are as in
    the BF16 layer.
    """
    if logits is None:
        logits = router_logits(x, w_router, bias)
    logits = as_f64(logits)
    T, E = logits.shape
    idx, gates = softmax_topk_gates(logits, k)
    counts = expert_counts(idx, E)
    tile_offsets, row_offsets = tile_layout(counts, bm)
    slot_of_route, route_of_slot = assign_slots(idx, row_offsets)
    n_rows = int(row_offsets[-1])
    xq = _qdq(x)
    Xd = dispatch(xq, slot_of_route, k, n_rows)
    ro = row_offsets.tolist()
    f = np.asarray(w_gate).shape[1]
    d = Xd.shape[1]
    H = np.zeros((n_rows, f))
    U = np.zeros((n_rows, f))
    A = np.zeros((n_rows, f))
    Aq = np.zeros((n_rows, f))
    Y = np.zeros((n_rows, d))
    for e in range(E):
        a, b = ro[e], ro[e + 1]
        if a == b:
            continue
        H[a:b] = Xd[a:b] @ _qdq(w_gate[e]).T
        U[a:b] = Xd[a:b] @ _qdq(w_up[e]).T
        A[a:b] = silu(H[a:b]) * U[a:b]
        Aq[a:b] = _qdq(A[a:b])
        Y[a:b] = Aq[a:b] @ _qdq(w_down[e]).T
    out = combine(Y, gates, slot_of_route, T, k)
    return {
        "logits": logits, "topk_idx": idx, "gates": gates, "counts": counts,
        "offsets": exclusive_scan(counts), "tile_offsets": tile_offsets,
        "row_offsets": row_offsets, "slot_of_route": slot_of_route,
        "route_of_slot": route_of_slot, "Xd": Xd, "H": H, "U": U, "A": A, "Aq": Aq,
        "Y": Y, "out": out, "k": k, "bm": bm,
    }


def layer_backward_mxfp8(fwd, d_out, x, w_router, w_gate, w_up, w_down, lb_coef: float = 0.0):
    """Backward with MXFP8 data-gradient GEMMs and BF16 weight-gradient GEMMs.

    The data-gradient GEMMs quantise their gradient operand along the
    contraction axis (dY along d; dH, dU along f) and use the second weight
    cache (W_down^T quantised along d; W_gate^T, W_up^T quantised along f).
    Weight gradients follow Section 24 Evidence 7 (global dequantisation, then
    BF16 grouped weight-gradient GEMMs): their activation operands are the
    dequantised MXFP8 activations (Xd, A) and their gradient operands the
    unquantised dY, dH, dU.
    """
    T, k = fwd["topk_idx"].shape
    E = fwd["logits"].shape[1]
    n_rows = fwd["Xd"].shape[0]
    d_gates, dY = combine_backward(d_out, fwd["Y"], fwd["gates"], fwd["slot_of_route"], T, k, n_rows)
    ro = fwd["row_offsets"].tolist()
    f, d = np.asarray(w_gate).shape[1:]
    H, U, Xd, Aq = fwd["H"], fwd["U"], fwd["Xd"], fwd["Aq"]
    dH = np.zeros((n_rows, f))
    dU = np.zeros((n_rows, f))
    dXd = np.zeros((n_rows, d))
    dWg = np.zeros((E, f, d))
    dWu = np.zeros((E, f, d))
    dWd = np.zeros((E, d, f))
    for e in range(E):
        a, b = ro[e], ro[e + 1]
        if a == b:
            continue
        dA = _qdq(dY[a:b]) @ _qdq(as_f64(w_down[e]).T).T
        h = H[a:b]
        dH[a:b] = dA * U[a:b] * silu_grad(h)
        dU[a:b] = dA * silu(h)
        dXd[a:b] = (_qdq(dH[a:b]) @ _qdq(as_f64(w_gate[e]).T).T
                    + _qdq(dU[a:b]) @ _qdq(as_f64(w_up[e]).T).T)
        dWd[e] = dY[a:b].T @ Aq[a:b]
        dWg[e] = dH[a:b].T @ Xd[a:b]
        dWu[e] = dU[a:b].T @ Xd[a:b]
    dx = dispatch_backward(dXd, fwd["slot_of_route"], T, k)
    extra = (load_balance_dlogits(fwd["logits"], fwd["topk_idx"], E, lb_coef)
             if lb_coef != 0.0 else None)
    rb = router_backward(d_gates, fwd["gates"], fwd["topk_idx"], E,
                         x if w_router is not None else None, w_router, extra)
    if w_router is not None:
        dx = dx + rb["dx_router"]
    out = {"d_gates": d_gates, "dY": dY, "dH": dH, "dU": dU, "dXd": dXd, "dx": dx,
           "dW_gate": dWg, "dW_up": dWu, "dW_down": dWd, "dlogits": rb["dlogits"]}
    if w_router is not None:
        out["dW_router"] = rb["dW_router"]
    return out
