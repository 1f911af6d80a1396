"""Seeded synthetic inputs for the MoE expert layer.

This module only draws random numbers and stores them; it holds none of the
layer's arithmetic (no routing, no softmax, no GEMM, no quantisation). Both the
oracle-side tests and the GPU-side tests/benchmark take their inputs from here,
so the two sides always see the same bits.

Value recipe (the workloads the pages benchmark use random routing as a systems
reference: "Olmo-core DDP training stack", Section 2, and Section 24 Evidence 1;
operand values must be realistic because GEMM time depends on them: Section 24
Evidence 8 / Table 34):

* x ~ N(0, 1), rounded to bf16 (round-to-nearest-even)
* router weight W_r [E, d], expert weights W_gate/W_up [E, f, d], W_down [E, d, f]
  ~ N(0, 0.02^2) (standard deviation 0.02), rounded to bf16
* router bias [T, E] fp32: N(0, 1) noise for "random routing", a per-expert Zipf
  bias for the skewed workload, or none
* upstream gradient dOut [T, d] ~ N(0, 1), rounded to bf16

Every tensor has its own generator seeded by (seed, tensor tag), so a tensor's
values do not depend on which other tensors were drawn.
"""
from __future__ import annotations

import json
import os
from dataclasses import dataclass, field

import numpy as np

__all__ = [
    "LayerConfig",
    "CONFIGS",
    "bf16_bits_from_f32",
    "f32_from_bf16_bits",
    "make_inputs",
    "zipf_expert_bias",
]

_HERE = os.path.dirname(os.path.abspath(__file__))

# Fixed tags: one independent stream per tensor.
_TAG = {
    "x": 11,
    "w_router": 12,
    "bias": 13,
    "w_gate": 14,
    "w_up": 15,
    "w_down": 16,
    "d_out": 17,
    "zipf_perm": 18,
}


@dataclass(frozen=True)
class LayerConfig:
    """Shape and input recipe of one workload."""

    name: str
    T: int          # tokens
    d: int          # d_model
    E: int          # experts
    k: int          # top-k
    f: int          # d_ff (SwiGLU hidden width per expert)
    prec: str = "bf16"          # "bf16" or "mxfp8"
    routing: str = "normal"     # "normal" (N(0,1) logit noise), "zipf", "none"
    backward: bool = True
    note: str = ""

    @property
    def R(self) -> int:
        return self.T * self.k


CONFIGS: dict[str, LayerConfig] = {
    "tiny_fwd": LayerConfig(
        "tiny_fwd", T=256, d=128, E=8, k=2, f=256, routing="none", backward=False,
        note="tiny forward: routing decided by x.W_r alone; seed 0"),
    "fine_grained": LayerConfig(
        "fine_grained", T=8192, d=2048, E=32, k=4, f=1024, routing="normal",
        note="fine-grained experts, fwd+bwd, near-uniform random routing"),
    "large_pool": LayerConfig(
        "large_pool", T=16384, d=2048, E=128, k=4, f=1024, routing="normal",
        note="128-expert pool, top-4 (47B-total / 3.2B-active style layer)"),
    "skewed": LayerConfig(
        "skewed", T=16384, d=2048, E=64, k=4, f=1408, routing="zipf",
        note="Zipf(s=1.2) per-expert bias; top expert ~15% of routes, >=4 empty"),
    "mxfp8": LayerConfig(
        "mxfp8", T=32768, d=4096, E=64, k=8, f=2048, prec="mxfp8", routing="normal",
        note="MXFP8 forward+backward, random routing"),
    # reduced cases for ncu captures: the same d, f and rows per expert as the
    # full workloads, with few experts so that a capture holds a few GB at most
    "mxfp8_8x4096": LayerConfig(
        "mxfp8_8x4096", T=4096, d=4096, E=8, k=8, f=2048, prec="mxfp8", routing="normal",
        note="8 experts of 4096 rows each (every token routed to all 8), d=4096, f=2048"),
}


def bf16_bits_from_f32(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); return the bits."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32)
    rounding = ((u >> 16) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + rounding) >> 16).astype(np.uint16)


def f32_from_bf16_bits(b: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns to float32."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def _rng(seed: int, tag: str, sub: int = 0) -> np.random.Generator:
    return np.random.default_rng([int(seed), _TAG[tag], int(sub)])


def _normal_bf16(seed: int, tag: str, shape: tuple, std: float) -> np.ndarray:
    """bf16 bits of N(0, std^2) samples; large tensors are drawn slab by slab."""
    out = np.empty(shape, dtype=np.uint16)
    if len(shape) == 3:
        for e in range(shape[0]):
            v = _rng(seed, tag, e + 1).standard_normal(shape[1:], dtype=np.float32)
            if std != 1.0:
                v *= np.float32(std)
            out[e] = bf16_bits_from_f32(v)
        return out
    v = _rng(seed, tag).standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        v *= np.float32(std)
    return bf16_bits_from_f32(v)


def zipf_expert_bias(E: int, seed: int, beta: float, s: float = 1.2, n_empty: int = 4) -> np.ndarray:
    """Per-expert Zipf bias: expert of popularity rank r gets beta * ln(r^-s).

    The rank order is a seeded permutation of the experts.  The n_empty
    lowest-ranked experts get a bias of -30 so that no token selects them.
    """
    perm = _rng(seed, "zipf_perm").permutation(E)      # perm[r-1] = expert of rank r
    bias = np.empty(E, dtype=np.float32)
    for r0, e in enumerate(perm):
        r = r0 + 1
        bias[e] = np.float32(beta * (-s) * np.log(r))
    for r0 in range(E - n_empty, E):
        bias[perm[r0]] = np.float32(-30.0)
    return bias


def _zipf_beta(cfg_name: str) -> float:
    path = os.path.join(os.path.dirname(_HERE), "tests", "golden", "zipf_calibration.json")
    with open(path) as fh:
        return float(json.load(fh)[cfg_name]["beta"])


def make_inputs(cfg: LayerConfig | str | None = None, seed: int = 0, *, T=None, d=None, E=None,
                k=None, f=None, routing=None, zipf_beta=None, with_grad=True) -> dict:
    """Draw every input of one layer call.

    Either pass a config (or its name), or the raw sizes T, d, E, k, f.
    Returns a dict of numpy arrays: bf16 tensors as uint16 bit patterns
    (`x`, `w_router`, `w_gate`, `w_up`, `w_down`, `d_out`) and the fp32
    router bias `bias` ([T, E], or None).
    """
    if isinstance(cfg, str):
        cfg = CONFIGS[cfg]
    if cfg is not None:
        T, d, E, k, f = cfg.T, cfg.d, cfg.E, cfg.k, cfg.f
        routing = cfg.routing if routing is None else routing
    routing = routing or "normal"
    inp = {"T": T, "d": d, "E": E, "k": k, "f": f, "seed": seed, "routing": routing}
    inp["x"] = _normal_bf16(seed, "x", (T, d), 1.0)
    inp["w_router"] = _normal_bf16(seed, "w_router", (E, d), 0.02)
    if routing == "normal":
        inp["bias"] = _rng(seed, "bias").standard_normal((T, E), dtype=np.float32)
    elif routing == "zipf":
        if zipf_beta is None:
            zipf_beta = _zipf_beta(cfg.name if cfg is not None else "skewed")
        row = zipf_expert_bias(E, seed, zipf_beta)
        inp["bias"] = np.ascontiguousarray(np.broadcast_to(row, (T, E)), dtype=np.float32)
        inp["zipf_beta"] = zipf_beta
    elif routing == "none":
        inp["bias"] = None
    else:
        raise ValueError(f"unknown routing recipe {routing!r}")
    inp["w_gate"] = _normal_bf16(seed, "w_gate", (E, f, d), 0.02)
    inp["w_up"] = _normal_bf16(seed, "w_up", (E, f, d), 0.02)
    inp["w_down"] = _normal_bf16(seed, "w_down", (E, d, f), 0.02)
    if with_grad:
        inp["d_out"] = _normal_bf16(seed, "d_out", (T, d), 1.0)
    return inp
