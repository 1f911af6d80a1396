"""Benchmark of the MoE expert layer (forward + backward) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl ours|reference]

One step = moe_layer_fwd + moe_layer_bwd over one batch of synthetic tokens
(router projection, softmax/top-k, counts/offsets/slots, rowwise dispatch,
grouped SwiGLU GEMMs, combine, and the whole backward), inputs resident in HBM.
The default workload is the largest one that fits one GPU: the MXFP8 layer,
T=32768 tokens, d_model=4096, 64 experts, top-8, d_ff=2048, seeded random
routing; its weight caches are rebuilt from the bf16 master weights every step.
`--config fine_grained|large_pool|skewed` runs the bf16 workloads.

Prints ONE JSON line (rank 0).  Multi-GPU (torchrun): every rank runs an
independent replica on its own tokens (the layer has no exchange step), so
scaling is weak and `value` is the total tokens/s of all ranks; the step time
is the maximum over ranks.

`--impl reference` times the CPU oracle (plain C++17 + OpenMP in double, the
correctness reference of this repository) on a bounded sample of the same
workload on the host cores; it is a deliberately slow baseline, not a target.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "moe_layer_tokens_per_s_fwd_bwd"
UNIT = "tokens/s"


# ------------------------------------------------------------------ distributed plumbing
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value: float, world: int) -> float:
    """Maximum of a per-rank float over all ranks (identity on one rank)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(world: int, tokens_per_rank: int, ms_max: float) -> float:
    """Whole-job tokens/s: every rank processed its own tokens within ms_max."""
    return world * tokens_per_rank / (ms_max / 1000.0)


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------ flops / bytes
def gemm_flops(cfg) -> dict:
    """Useful flops of the expert GEMMs per step (no tile padding counted)."""
    R = cfg.T * cfg.k
    return {
        "fwd1": 4.0 * R * cfg.d * cfg.f, "fwd2": 2.0 * R * cfg.d * cfg.f,
        "dgrad2": 2.0 * R * cfg.d * cfg.f, "wgrad2": 2.0 * R * cfg.d * cfg.f,
        "dgrad1": 4.0 * R * cfg.d * cfg.f, "wgrad1": 4.0 * R * cfg.d * cfg.f,
        "router": 2.0 * cfg.T * cfg.d * cfg.E,
    }


# ------------------------------------------------------------------ clocks sampling
class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as fh:
            for line in fh:
                p = [x.strip() for x in line.split(",")]
                if len(p) >= 9 and p[1].replace(".", "").isdigit():
                    rows.append(p)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows]
        mx = max(float(r[2]) for r in rows)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        loaded = [s for s in sm if s > 0.5 * mx] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": mx, "reasons": reasons,
                "samples": len(rows), "power_w_max": max(float(r[3]) for r in rows
                                                          if r[3].replace(".", "").isdigit())}


# ------------------------------------------------------------------ the oracle arm
def oracle_sample(cfg, inp, budget_s: float = 15.0, max_experts: int = 0) -> dict:
    """Time the C++ oracle on a bounded sample of the workload.

    The sample is the routing of all T tokens (router projection, softmax/top-k,
    counts, offsets, slots), then whole experts, one after the other in a seeded
    order, each with every one of its routes: dispatch (MXFP8: tokens quantised),
    forward (MXFP8: weights quantised in both orientations, A quantised), the
    expert's rows of the combine backward, and the backward.  Experts are added
    until `budget_s` has passed (at least one; at most `max_experts` when > 0).
    The full step is extrapolated as routing + (experts with routes) x the mean
    expert time; the combine and dispatch gather-sums over all tokens are O(T k d)
    and are left out."""
    import numpy as np

    from oracle import cpp as O

    mx = cfg.prec == "mxfp8"
    t0 = time.perf_counter()
    logits = O.router_logits(inp["x"], inp["w_router"], inp["bias"])
    idx, gates = O.softmax_topk_gates(logits, cfg.k)
    counts = O.expert_counts(idx, cfg.E)
    _, row_offsets = O.tile_layout(counts, 128)
    sor, ros = O.assign_slots(idx, row_offsets)
    t_route = time.perf_counter() - t0
    order = [int(e) for e in np.random.default_rng(0).permutation(cfg.E) if counts[e] > 0]
    lib = O.lib()
    p = O._ptr
    times, rows_done = [], 0
    t_start = time.perf_counter()
    for e in order:
        a, b = int(row_offsets[e]), int(row_offsets[e]) + int(counts[e])
        routes = ros[a:b]
        tok = routes // cfg.k
        n, d, f = b - a, cfg.d, cfg.f
        t1 = time.perf_counter()
        xe = O.as_f64(inp["x"][tok])
        if mx:
            xe = O._qdq(xe)
        wg, wu, wd = (O.as_f64(inp[nm][e]) for nm in ("w_gate", "w_up", "w_down"))
        H, U, A, Y = (np.empty((n, f)), np.empty((n, f)), np.empty((n, f)), np.empty((n, d)))
        Aq = np.empty((n, f)) if mx else None
        lib.mo_expert_forward(p(xe), n, d, f, p(wg), p(wu), p(wd), int(mx), p(H), p(U), p(A),
                              p(Aq), p(Y))
        dY = gates.reshape(-1)[routes][:, None] * O.as_f64(inp["d_out"][tok])
        dH, dU, dX = np.empty((n, f)), np.empty((n, f)), np.empty((n, d))
        dWg, dWu, dWd = np.empty((f, d)), np.empty((f, d)), np.empty((d, f))
        lib.mo_expert_backward(p(dY), p(xe), p(H), p(U), p(Aq if mx else A), n, d, f, p(wg),
                               p(wu), p(wd), int(mx), p(dH), p(dU), p(dX), p(dWg), p(dWu),
                               p(dWd))
        times.append(time.perf_counter() - t1)
        rows_done += n
        if time.perf_counter() - t_start >= budget_s or (max_experts and len(times) >= max_experts):
            break
    step_s = t_route + len(order) * (sum(times) / len(times))
    return {"value": cfg.T / step_s, "unit": UNIT, "cores": O.threads(), "kind": "oracle",
            "extrapolated": True, "experts_timed": len(times), "seconds": t_route + sum(times),
            "step_s_extrapolated": step_s,
            "sample": (f"'{cfg.name}' workload: routing of all {cfg.T} tokens ({t_route:.1f} s), "
                       f"then {len(times)} of its {len(order)} experts with routes, each with all "
                       f"of its routes ({rows_done} rows in all), dispatch + "
                       f"{'MXFP8 ' if mx else ''}forward + backward "
                       f"({sum(times) / len(times):.2f} s per expert); the step is extrapolated "
                       f"as routing + {len(order)} x the mean expert time; C++ oracle in double, "
                       f"{O.threads()} OpenMP threads")}


def run_reference(args, cfg):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    from synth import make_inputs
    # the whole run stays near two minutes: as many whole-expert samples as fit
    # (at most --steps), each one a step of this arm
    inp = make_inputs(cfg, seed=0)
    res = oracle_sample(cfg, inp, budget_s=90.0, max_experts=max(args.steps, 1))
    v = res["value"]
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
        "steps": res["experts_timed"], "steps_requested": args.steps, "warmup": 0,
        "ms_per_step": 1000.0 * res["step_s_extrapolated"], "extrapolated": True,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_block(cfg),
        "cpu_baseline": {"value": v, "unit": UNIT, "cores": res["cores"], "kind": "oracle",
                         "sample": res["sample"]},
        "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "what": "each step of this arm is one expert of the workload (all of its routes) on the "
                "C++ oracle; ms_per_step is the extrapolated time of a whole layer step",
    }
    print(json.dumps(line), flush=True)
    return 0


def config_block(cfg):
    return {"workload": cfg.name, "T": cfg.T, "d_model": cfg.d, "n_experts": cfg.E, "top_k": cfg.k,
            "d_ff": cfg.f, "precision": cfg.prec, "routing": cfg.routing, "seed": 0,
            "l2": "inputs larger than L2: expert weights alone are 3*E*d*f*2 bytes per step"}


# ------------------------------------------------------------------ our arm
def run_ours(args, cfg):
    import numpy as np
    import torch

    import moe_expert_layer_softmax_gb300 as m
    from synth import make_inputs

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    m.init(local)
    inp = make_inputs(cfg, seed=rank)

    def bf(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

    x, wr, wg, wu, wd, dO = (bf(inp[n]) for n in ("x", "w_router", "w_gate", "w_up", "w_down", "d_out"))
    bias = torch.from_numpy(inp["bias"]).to(dev) if inp["bias"] is not None else None
    mx = cfg.prec == "mxfp8"
    s = m.shape(cfg.T, cfg.d, cfg.E, cfg.k, cfg.f, prec=m.MXFP8 if mx else m.BF16)
    buf = m.allocate(s)
    out = torch.empty(cfg.T, cfg.d, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        if mx:   # the weight caches follow every weight update: rebuilt once per step
            m.build_mx_weights(s, wg, wu, wd, buf.mx_weights)
        m.forward(buf, x, wr, bias, wg, wu, wd, out)
        m.backward(buf, dO, x, wr, wg, wu, wd)

    m.clear_error(buf.ws)
    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    if m.read_error(buf.ws) != 0:
        raise RuntimeError("device error word set during warm-up")

    # ---- timed region: K whole steps
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    ms = e0.elapsed_time(e1) / args.steps
    clk = clocks.stop()
    ms_max = max_over_ranks(ms, world)
    value = job_value(world, cfg.T, ms_max)

    # ---- per-stage times (same kernels, called stage by stage, events on the stream)
    stages = stage_times(m, buf, s, x, wr, bias, wg, wu, wd, dO, out, stream, reps=max(3, args.steps),
                         mx=mx)
    fl = gemm_flops(cfg)
    gemm_ms = sum(stages[k] for k in ("fwd1", "fwd2", "dgrad2", "wgrad2", "dgrad1", "wgrad1"))
    gemm_fl = sum(fl[k] for k in ("fwd1", "fwd2", "dgrad2", "wgrad2", "dgrad1", "wgrad1"))
    peaks = load_peaks()
    dom = max(("fwd1", "fwd2", "dgrad2", "wgrad2", "dgrad1", "wgrad1"), key=lambda k: stages[k])
    # the dominant GEMM's own launch time: CUDA events recorded by the library
    # around each of its launches during another `steps` whole layer steps
    p0 = torch.cuda.Event(enable_timing=True)
    p1 = torch.cuda.Event(enable_timing=True)
    m.profile_start(GEMM_OP[dom])
    p0.record(stream)
    for _ in range(args.steps):
        step()
    p1.record(stream)
    kernel_ms_total, kernel_launches = m.profile_stop()
    torch.cuda.synchronize()
    region_s = p0.elapsed_time(p1) / 1000.0
    kernel_ms = kernel_ms_total / max(kernel_launches, 1)
    achieved = fl[dom] / (kernel_ms / 1000.0) / 1e12
    # the burst peak for a kernel inside a short timed region, the sustained one
    # (power-capped, seconds-long) when the region lasts seconds
    sustained = region_s >= 2.0
    peak = peaks["bf16_tflops_sustained" if sustained else "bf16_tflops"]
    peak_note = (f"{peaks['source']} {'sustained' if sustained else 'burst'} bf16 (the dominant "
                 f"kernel timed inside {args.steps} steps, {region_s:.2f} s)")
    if mx and dom in FP8_OPS:
        # dense fp8 is twice the dense bf16 rate on this part (2.25 -> 4.5 PFLOP/s nominal)
        peak = 2.0 * peak
        peak_note += " x 2 (nominal fp8/bf16 ratio)"
    traffic, traffic_note = gemm_traffic(cfg.name, dom)
    roofline = {"bound": "tensor", "kernel": f"grouped_gemm_kernel ({dom})", "achieved": achieved,
                "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak, "traffic": traffic,
                "traffic_source": traffic_note, "kernel_ms": kernel_ms,
                "kernel_launches_timed": kernel_launches, "peak_source": peak_note,
                "algorithmic": f"{fl[dom] / 1e9:.1f} GFLOP per launch (useful flops, no tile padding)"}

    # ---- per-layer recompute: the backward re-runs dispatch and both expert
    # GEMMs, so the expert activations need not be kept from the forward
    def step_recompute():
        if mx:
            m.build_mx_weights(s, wg, wu, wd, buf.mx_weights)
        m.forward(buf, x, wr, bias, wg, wu, wd, out)
        m.backward(buf, dO, x, wr, wg, wu, wd, recompute=True)

    for _ in range(3):
        step_recompute()
    torch.cuda.synchronize()
    r0 = torch.cuda.Event(enable_timing=True)
    r1 = torch.cuda.Event(enable_timing=True)
    r0.record(stream)
    for _ in range(args.steps):
        step_recompute()
    r1.record(stream)
    torch.cuda.synchronize()
    rc_ms = max_over_ranks(r0.elapsed_time(r1) / args.steps, world)
    rows = m.rows_max(s)
    if mx:   # xd_q, a_q (+ 1/32 scales), H, U, Y
        act_bytes = rows * ((cfg.d + cfg.f) * 33 // 32 + (2 * cfg.f + cfg.d) * 2)
    else:    # Xd, H, U, A, Y in bf16
        act_bytes = rows * (2 * cfg.d + 3 * cfg.f) * 2
    recompute = {"value": job_value(world, cfg.T, rc_ms), "unit": UNIT, "ms_per_step": rc_ms,
                 "activation_bytes_not_kept": int(act_bytes),
                 "what": "backward re-runs dispatch, GEMM1 and GEMM2 from x and the routing "
                         "metadata (per-layer recompute)"}

    # ---- with the load-balancing term: statistics in the forward, coef * LBL's
    # gradient in the backward (dense router backward)
    buf.saved["lb_stats"] = torch.empty(cfg.E + 1, dtype=torch.float32, device=dev)

    def step_lb():
        if mx:
            m.build_mx_weights(s, wg, wu, wd, buf.mx_weights)
        m.forward(buf, x, wr, bias, wg, wu, wd, out)
        m.backward(buf, dO, x, wr, wg, wu, wd, lb_coef=0.01)

    for _ in range(3):
        step_lb()
    torch.cuda.synchronize()
    l0 = torch.cuda.Event(enable_timing=True)
    l1 = torch.cuda.Event(enable_timing=True)
    l0.record(stream)
    for _ in range(args.steps):
        step_lb()
    l1.record(stream)
    torch.cuda.synchronize()
    lb_ms = max_over_ranks(l0.elapsed_time(l1) / args.steps, world)
    lb_line = {"value": job_value(world, cfg.T, lb_ms), "unit": UNIT, "ms_per_step": lb_ms,
               "lbl": float(buf.saved["lb_stats"][0].item()), "coef": 0.01,
               "what": "Switch-style load-balancing scalar in the forward and coef * its "
                       "gradient in the backward (the router backward becomes dense)"}
    buf.saved["lb_stats"] = None

    # ---- two-batch overlap on one GPU: the batch split in halves whose fwd+bwd
    # run on two streams, against the same halves one after the other
    tbo = None
    if not mx and cfg.T % 2 == 0:
        tbo = two_batch_overlap(m, cfg, x, wr, bias, wg, wu, wd, dO, dev, stream, args.steps,
                                world)

    # ---- MXFP8 weight gradient on the natural layout vs dequantise + BF16
    mxw = mx_wgrad_variants(m, dev, stream) if not args.no_extras else None

    # ---- end to end through the public API with host buffers
    e2e = end_to_end(m, buf, cfg, inp, wr, bias, wg, wu, wd, dev, stream, args.steps, world)

    if m.read_error(buf.ws) != 0:
        raise RuntimeError("device error word set during the timed region")

    # the C++ oracle on a bounded sample of the same workload (rank 0 at N = 1)
    cpu = (oracle_sample(cfg, inp) if (rank == 0 and world == 1 and not args.no_cpu_baseline)
           else None)
    # router GEMM, top-k, scan, slots | dispatch, fwd1, fwd2, combine | combine bwd, dgrad2,
    # wgrad2, dgrad1, wgrad1, dispatch bwd, router bwd (2); MXFP8 adds the three weight-cache
    # quantisers (dY is quantised in the combine backward, Xd and A dequantised in the
    # dispatch and the fwd1 epilogue)
    launches_per_step = (16 if wr is not None else 13) + (3 if mx else 0)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": ms_max, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "mxfp8+bf16" if mx else "bf16",
        "data": "synthetic", "config": config_block(cfg),
        "gemm": gemm_summary(cfg, stages, fl, peaks, mx),
        "stage_ms": {k: round(v, 5) for k, v in stages.items()},
        "roofline": roofline, "cpu_baseline": cpu, "clocks": clk, "e2e": e2e,
        "recompute": recompute, "load_balance": lb_line, "two_batch_overlap": tbo,
        "mx_wgrad": mxw,
        "gpu_launches": launches_per_step * args.steps,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


GEMM_OP = {"fwd1": 0, "fwd2": 1, "dgrad2": 2, "dgrad1": 3, "wgrad2": 4, "wgrad1": 5}
GEMMS = ("fwd1", "fwd2", "dgrad2", "wgrad2", "dgrad1", "wgrad1")
FP8_OPS = ("fwd1", "fwd2", "dgrad2", "dgrad1")     # MXFP8 in the MXFP8 layer; weight gradients bf16


def gemm_summary(cfg, stages, fl, peaks, mx):
    """Useful TFLOP/s of the grouped GEMMs per operand type, each against its own
    dense peak: bf16 the measured burst bf16 figure (the stage calls are timed one
    by one), MXFP8 twice that (the nominal fp8/bf16 ratio)."""
    out = {}
    groups = {"mxfp8": [g for g in GEMMS if g in FP8_OPS], "bf16": [g for g in GEMMS if g not in FP8_OPS]} \
        if mx else {"bf16": list(GEMMS)}
    for name, ops in groups.items():
        ms = sum(stages[g] for g in ops)
        flops = sum(fl[g] for g in ops)
        peak = peaks["bf16_tflops"] * (2.0 if name == "mxfp8" else 1.0)
        tf = flops / (ms / 1000.0) / 1e12
        out[name] = {"ops": ops, "ms": ms, "tflops": tf, "peak_tflops": peak, "frac": tf / peak,
                     "per_op_frac": {g: fl[g] / (stages[g] / 1000.0) / 1e12 / peak for g in ops},
                     "peak_source": f"{peaks['source']} burst bf16" + (" x 2 (nominal fp8/bf16 ratio)"
                                                                         if name == "mxfp8" else "")}
    all_ms = sum(stages[g] for g in GEMMS)
    out["all"] = {"ms": all_ms, "tflops": sum(fl[g] for g in GEMMS) / (all_ms / 1000.0) / 1e12}
    return out
GEMM_SOURCES = ("moe_expert_layer_softmax_gb300/csrc/gemm.cu",
                "moe_expert_layer_softmax_gb300/csrc/common.cuh")


def gemm_source_hash(root: str = ROOT) -> str:
    """sha256 of the GEMM sources with comments and whitespace removed (so that
    only a change of the code itself invalidates a recorded ncu capture)."""
    import hashlib
    import re
    h = hashlib.sha256()
    for rel in GEMM_SOURCES:
        with open(os.path.join(root, rel)) as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()


DRAM_RECORD = os.path.join(ROOT, "profiles", "dram_per_launch.json")


def gemm_traffic(workload: str, op: str):
    """DRAM bytes (read + write) of one launch of GEMM `op` on `workload`, from the
    committed record of ncu captures (scaled from a reduced case of the same
    shape when the record says so); None when the GEMM sources changed since."""
    if not os.path.exists(DRAM_RECORD):
        return None, "no ncu DRAM record"
    with open(DRAM_RECORD) as fh:
        recs = json.load(fh).get("records", [])
    rec = next((r for r in recs if r.get("workload") == workload), None)
    if rec is None:
        return None, f"no ncu capture for the '{workload}' workload"
    if rec.get("source_sha256") != gemm_source_hash():
        return None, "GEMM sources changed since the ncu capture"
    ops = rec.get("ops", {})
    if op not in ops:
        return None, f"{op} not in the ncu capture"
    scale = float(rec.get("scale", 1.0))
    note = "dram__bytes_read.sum + dram__bytes_write.sum, " + os.path.relpath(DRAM_RECORD, ROOT)
    if scale != 1.0:
        note += f" (captured on '{rec['captured_on']}', x {scale:g} for the full launch)"
    return int(round((int(ops[op]["read"]) + int(ops[op]["write"])) * scale)), note


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            p = json.load(fh)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained", p["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def stage_times(m, buf, s, x, wr, bias, wg, wu, wd, dO, out, stream, reps=5, mx=False):
    """Average ms of each stage call, events recorded on the launching stream."""
    import torch
    sv, g = buf.saved, buf.grads
    if mx:
        return stage_times_mx(m, buf, s, x, wr, bias, wg, wu, wd, dO, out, stream, reps)
    calls = [
        ("route", lambda: m.route(s, x, wr, bias, sv["logits"], sv["topk_idx"], sv["gates"],
                                  sv["counts"], sv["offsets"], sv["tile_offsets"],
                                  sv["slot_of_route"], sv["route_of_slot"], buf.ws)),
        ("dispatch", lambda: m.dispatch(s, x, sv["slot_of_route"], sv["counts"], sv["tile_offsets"],
                                        sv["xd"])),
        ("fwd1", lambda: m.grouped_gemm(s, m.GEMM_FWD1_SWIGLU, buf.ws, tile_offsets=sv["tile_offsets"],
                                        a0=sv["xd"], w0=wg, w1=wu, out0=sv["h"], out1=sv["u"],
                                        out2=sv["a"])),
        ("fwd2", lambda: m.grouped_gemm(s, m.GEMM_FWD2, buf.ws, tile_offsets=sv["tile_offsets"],
                                        a0=sv["a"], w0=wd, out0=sv["y"])),
        ("combine", lambda: m.combine(s, sv["y"], sv["gates"], sv["slot_of_route"], out)),
        ("combine_bwd", lambda: m.combine_bwd(s, dO, sv["y"], sv["gates"], sv["topk_idx"],
                                              sv["slot_of_route"], sv["counts"], sv["tile_offsets"],
                                              g["dy"], g["d_gates"], g["dlogits"])),
        ("dgrad2", lambda: m.grouped_gemm(s, m.GEMM_DGRAD2_SWIGLU, buf.ws,
                                          tile_offsets=sv["tile_offsets"], a0=g["dy"], w0=wd,
                                          aux0=sv["h"], aux1=sv["u"], out0=g["dh"], out1=g["du"])),
        ("wgrad2", lambda: m.grouped_gemm(s, m.GEMM_WGRAD2, buf.ws, tile_offsets=sv["tile_offsets"],
                                          a0=g["dy"], a1=sv["a"], out0=g["dw_down"])),
        ("dgrad1", lambda: m.grouped_gemm(s, m.GEMM_DGRAD1, buf.ws, tile_offsets=sv["tile_offsets"],
                                          a0=g["dh"], a1=g["du"], w0=wg, w1=wu, out0=g["dxd"])),
        ("wgrad1", lambda: m.grouped_gemm(s, m.GEMM_WGRAD1, buf.ws, tile_offsets=sv["tile_offsets"],
                                          a0=g["dh"], a1=g["du"], aux0=sv["xd"], out0=g["dw_gate"],
                                          out1=g["dw_up"])),
        ("dispatch_bwd", lambda: m.dispatch_bwd(s, g["dxd"], sv["slot_of_route"], sv["topk_idx"],
                                                g["dlogits"], wr, g["dx"])),
        ("router_bwd", lambda: m.router_bwd(s, x, g["dlogits"], sv["route_of_slot"], sv["counts"],
                                            sv["tile_offsets"], g["dw_router"], buf.ws)),
    ]
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(calls) + 1)] for _ in range(reps)]
    for r in range(reps):
        ev[r][0].record(stream)
        for i, (_, fn) in enumerate(calls):
            fn()
            ev[r][i + 1].record(stream)
    torch.cuda.synchronize()
    res = {}
    for i, (name, _) in enumerate(calls):
        res[name] = sum(ev[r][i].elapsed_time(ev[r][i + 1]) for r in range(reps)) / reps
    return res


def stage_times_mx(m, buf, s, x, wr, bias, wg, wu, wd, dO, out, stream, reps):
    """Stage times of the MXFP8 layer (same calls moe_layer_fwd/bwd make)."""
    import torch
    sv, g, w, b = buf.saved, buf.grads, buf.mx_weights, buf.mx
    calls = [
        ("weight_cache", lambda: m.build_mx_weights(s, wg, wu, wd, w)),
        ("route", lambda: m.route(s, x, wr, bias, sv["logits"], sv["topk_idx"], sv["gates"],
                                  sv["counts"], sv["offsets"], sv["tile_offsets"],
                                  sv["slot_of_route"], sv["route_of_slot"], buf.ws)),
        ("dispatch", lambda: m.dispatch(s, x, sv["slot_of_route"], sv["counts"], sv["tile_offsets"],
                                        b["xd_q"], b["xd_s"], xd_dq=b["xd_dq"])),
        ("fwd1", lambda: m.grouped_gemm(s, m.GEMM_FWD1_SWIGLU, buf.ws, tile_offsets=sv["tile_offsets"],
                                        a0=b["xd_q"], sfa0=b["xd_s"], w0=w["gu_q"], sfb0=w["gu_s"],
                                        out0=sv["h"], out1=sv["u"], out2=b["a_q"], osf0=b["a_s"],
                                        out3=b["a_dq"])),
        ("fwd2", lambda: m.grouped_gemm(s, m.GEMM_FWD2, buf.ws, tile_offsets=sv["tile_offsets"],
                                        a0=b["a_q"], sfa0=b["a_s"], w0=w["down_q"], sfb0=w["down_s"],
                                        out0=sv["y"])),
        ("combine", lambda: m.combine(s, sv["y"], sv["gates"], sv["slot_of_route"], out)),
        ("combine_bwd", lambda: m.combine_bwd(s, dO, sv["y"], sv["gates"], sv["topk_idx"],
                                              sv["slot_of_route"], sv["counts"], sv["tile_offsets"],
                                              g["dy"], g["d_gates"], g["dlogits"], dy_q=b["dy_q"],
                                              dy_scales=b["dy_s"])),
        ("dgrad2", lambda: m.grouped_gemm(s, m.GEMM_DGRAD2_SWIGLU, buf.ws,
                                          tile_offsets=sv["tile_offsets"], a0=b["dy_q"], sfa0=b["dy_s"],
                                          w0=w["downT_q"], sfb0=w["downT_s"], aux0=sv["h"],
                                          aux1=sv["u"], out0=g["dh"], out1=g["du"], out2=b["dh_q"],
                                          out3=b["du_q"], osf0=b["dh_s"], osf1=b["du_s"])),
        ("wgrad2", lambda: m.grouped_gemm(s, m.GEMM_WGRAD2, buf.ws, tile_offsets=sv["tile_offsets"],
                                          a0=g["dy"], a1=b["a_dq"], out0=g["dw_down"])),
        ("dgrad1", lambda: m.grouped_gemm(s, m.GEMM_DGRAD1, buf.ws, tile_offsets=sv["tile_offsets"],
                                          a0=b["dh_q"], sfa0=b["dh_s"], a1=b["du_q"], sfa1=b["du_s"],
                                          w0=w["gateT_q"], sfb0=w["gateT_s"], w1=w["upT_q"],
                                          sfb1=w["upT_s"], out0=g["dxd"])),
        ("wgrad1", lambda: m.grouped_gemm(s, m.GEMM_WGRAD1, buf.ws, tile_offsets=sv["tile_offsets"],
                                          a0=g["dh"], a1=g["du"], aux0=b["xd_dq"], out0=g["dw_gate"],
                                          out1=g["dw_up"])),
        ("dispatch_bwd", lambda: m.dispatch_bwd(s, g["dxd"], sv["slot_of_route"], sv["topk_idx"],
                                                g["dlogits"], wr, g["dx"])),
        ("router_bwd", lambda: m.router_bwd(s, x, g["dlogits"], sv["route_of_slot"], sv["counts"],
                                            sv["tile_offsets"], g["dw_router"], buf.ws)),
    ]
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(calls) + 1)] for _ in range(reps)]
    for r in range(reps):
        ev[r][0].record(stream)
        for i, (_, fn) in enumerate(calls):
            fn()
            ev[r][i + 1].record(stream)
    torch.cuda.synchronize()
    return {name: sum(ev[r][i].elapsed_time(ev[r][i + 1]) for r in range(reps)) / reps
            for i, (name, _) in enumerate(calls)}


def two_batch_overlap(m, cfg, x, wr, bias, wg, wu, wd, dO, dev, stream, steps, world):
    """The step's tokens in two halves, each a whole layer fwd+bwd with its own
    buffers: (a) on two streams at once, (b) one after the other on one stream."""
    import torch
    h = cfg.T // 2
    s2 = m.shape(h, cfg.d, cfg.E, cfg.k, cfg.f)
    bufs = [m.allocate(s2) for _ in range(2)]
    outs = [torch.empty(h, cfg.d, dtype=torch.bfloat16, device=dev) for _ in range(2)]
    xs = [x[:h], x[h:]]
    ds = [dO[:h], dO[h:]]
    bs = [bias[:h], bias[h:]] if bias is not None else [None, None]
    streams = [torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)]
    fork = torch.cuda.Event()
    joins = [torch.cuda.Event(), torch.cuda.Event()]

    def half(i, st):
        m.forward(bufs[i], xs[i], wr, bs[i], wg, wu, wd, outs[i], stream=st)
        m.backward(bufs[i], ds[i], xs[i], wr, wg, wu, wd, stream=st)

    def step_overlap():
        fork.record(stream)
        for i in range(2):
            streams[i].wait_event(fork)
            with torch.cuda.stream(streams[i]):
                half(i, streams[i])
            joins[i].record(streams[i])
        for i in range(2):
            stream.wait_event(joins[i])

    def step_serial():
        for i in range(2):
            half(i, stream)

    res = {}
    for name, fn in (("overlapped", step_overlap), ("serial", step_serial)):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        ms = max_over_ranks(e0.elapsed_time(e1) / steps, world)
        res[name] = {"value": job_value(world, cfg.T, ms), "ms_per_step": ms}
    res["unit"] = UNIT
    res["what"] = (f"two halves of {h} tokens per step, each a whole layer fwd+bwd: on two "
                   "streams at once vs one after the other")
    return res


def mx_wgrad_variants(m, dev, stream, sizes=(2048, 4096, 8192), rows=16384, E=8, reps=10):
    """The down-projection weight gradient dW[e] = dY_e^T A_e (K = N = d = f) on
    an MXFP8 activation operand, 16384 rows over 8 experts of 2048 rows: the
    natural-layout kernel (codes dequantised inside the GEMM) against the global
    dequantisation followed by the BF16 grouped GEMM.  L2 is flushed before each
    timed launch."""
    import torch
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    g = torch.Generator(device=dev)
    g.manual_seed(0)
    res = {}
    for K in sizes:
        s = m.shape(rows // 4, K, E, 4, K, prec=m.MXFP8)
        n = m.rows_max(s)
        tiles = rows // E // 128
        to = torch.arange(E + 1, dtype=torch.int32, device=dev) * tiles
        ws = torch.zeros(m.workspace_size(s), dtype=torch.uint8, device=dev)
        dY = torch.zeros(n, K, dtype=torch.bfloat16, device=dev)
        A = torch.zeros(n, K, dtype=torch.bfloat16, device=dev)
        dY[:rows].normal_(generator=g)
        A[:rows].normal_(generator=g)
        Aq = torch.empty(n, K, dtype=torch.uint8, device=dev)
        As = torch.empty(n * K // 32, dtype=torch.uint8, device=dev)
        m.quantize_mxfp8(1, n, K, 1, A, Aq, As, stream=stream)
        del A
        Adq = torch.empty(n, K, dtype=torch.bfloat16, device=dev)
        dW = torch.empty(E, K, K, dtype=torch.float32, device=dev)
        arms = {
            "natural": lambda: m.grouped_gemm(s, m.GEMM_WGRAD2_NATURAL, ws, stream=stream,
                                              tile_offsets=to, a0=dY, a1=Aq, sfb0=As, out0=dW),
            "dq_bf16": lambda: (m.dequantize_mxfp8(n, K, Aq, As, Adq, stream=stream),
                                m.grouped_gemm(s, m.GEMM_WGRAD2, ws, stream=stream,
                                               tile_offsets=to, a0=dY, a1=Adq, out0=dW)),
            "bf16_gemm_alone": lambda: m.grouped_gemm(s, m.GEMM_WGRAD2, ws, stream=stream,
                                                      tile_offsets=to, a0=dY, a1=Adq, out0=dW),
        }
        row = {}
        for name, fn in arms.items():
            for _ in range(3):
                fn()
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(reps)]
            with torch.cuda.stream(stream):
                for e0, e1 in ev:
                    flush.fill_(1)
                    e0.record(stream)
                    fn()
                    e1.record(stream)
            torch.cuda.synchronize()
            ms = sum(e0.elapsed_time(e1) for e0, e1 in ev) / reps
            row[name + "_ms"] = round(ms, 5)
            row[name + "_tflops"] = round(2.0 * rows * K * K / (ms / 1000.0) / 1e12, 1)
        if m.read_error(ws) != 0:
            raise RuntimeError("device error word set in the MXFP8 weight-gradient comparison")
        res[str(K)] = row
        del dY, Aq, As, Adq, dW, ws
    res["what"] = (f"dW_down weight gradient, K = N, {rows} rows over {E} experts: natural "
                   "MXFP8 layout dequantised inside the GEMM vs global dequantisation + BF16 "
                   "grouped GEMM (and that GEMM alone)")
    return res


def end_to_end(m, buf, cfg, inp, wr, bias, wg, wu, wd, dev, stream, steps, world):
    """Same step through the public API, with the step's inputs (x, dOut) copied
    from pinned host memory and its results (out, dx) copied back, every step.

    Uploads run on one copy stream and downloads on another, with two device
    slots for x, dOut, out and dx, so step i+1's upload and step i-1's download
    overlap step i's kernels; every copy is inside the timed region."""
    import numpy as np
    import torch

    def pinned(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).pin_memory()

    hx, hd = pinned(inp["x"]), pinned(inp["d_out"])
    mk = lambda: torch.empty(cfg.T, cfg.d, dtype=torch.bfloat16, device=dev)
    slots = [dict(x=mk(), dO=mk(), out=mk(), dx=mk(),
                  ho=torch.empty(cfg.T, cfg.d, dtype=torch.bfloat16).pin_memory(),
                  hdx=torch.empty(cfg.T, cfg.d, dtype=torch.bfloat16).pin_memory(),
                  up=torch.cuda.Event(), fwd=torch.cuda.Event(), comp=torch.cuda.Event(),
                  down=torch.cuda.Event())
             for _ in range(2)]
    fwd_done = [None]   # event after the latest step's forward
    up_s, down_s = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    mx = buf.mx is not None
    dx_own = buf.grads["dx"]

    # The copies are placed where the GPU is busiest with tensor-core work: step
    # i+1's upload and step i's `out` download wait for step i's forward, so
    # they overlap its backward GEMMs; `dx` goes down after the backward.
    def step(i):
        sl = slots[i % 2]
        with torch.cuda.stream(up_s):
            if i >= 2:
                up_s.wait_event(sl["comp"])           # step i-2 finished reading x, dOut
            if fwd_done[0] is not None:
                up_s.wait_event(fwd_done[0])          # during the previous step's backward
            sl["x"].copy_(hx, non_blocking=True)
            sl["dO"].copy_(hd, non_blocking=True)
            sl["up"].record(up_s)
        stream.wait_event(sl["up"])
        if i >= 2:
            stream.wait_event(sl["down"])             # step i-2's out, dx are on the host
        buf.grads["dx"] = sl["dx"]
        if mx:
            m.build_mx_weights(buf.shape, wg, wu, wd, buf.mx_weights)
        m.forward(buf, sl["x"], wr, bias, wg, wu, wd, sl["out"])
        sl["fwd"].record(stream)
        fwd_done[0] = sl["fwd"]
        with torch.cuda.stream(down_s):
            down_s.wait_event(sl["fwd"])
            sl["ho"].copy_(sl["out"], non_blocking=True)
        m.backward(buf, sl["dO"], sl["x"], wr, wg, wu, wd)
        sl["comp"].record(stream)
        with torch.cuda.stream(down_s):
            down_s.wait_event(sl["comp"])
            sl["hdx"].copy_(sl["dx"], non_blocking=True)
            sl["down"].record(down_s)

    try:
        for i in range(4):
            step(i)
        torch.cuda.synchronize()
        barrier(world)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        up_s.wait_event(e0)
        down_s.wait_event(e0)
        for i in range(steps):
            step(i)
        for sl in slots:
            stream.wait_event(sl["down"])
        e1.record(stream)
        torch.cuda.synchronize()
    finally:
        buf.grads["dx"] = dx_own
    ms = max_over_ranks(e0.elapsed_time(e1) / steps, world)
    nbytes = 2 * cfg.T * cfg.d * 2
    return {"value": job_value(world, cfg.T, ms), "unit": UNIT, "ms_per_step": ms,
            "h2d_bytes_per_step": nbytes, "d2h_bytes_per_step": nbytes,
            "overlap": "uploads and downloads on two copy streams, double-buffered device slots; "
                       "the next step's upload and this step's `out` download overlap the backward"}


def run_profile(args, cfg):
    """Whole layer steps only (weight caches, forward, backward), nothing timed:
    the command that ncu captures."""
    import numpy as np
    import torch

    import moe_expert_layer_softmax_gb300 as m
    from synth import make_inputs

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    m.init(0)
    inp = make_inputs(cfg, seed=0)

    def bf(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

    x, wr, wg, wu, wd, dO = (bf(inp[n]) for n in ("x", "w_router", "w_gate", "w_up", "w_down", "d_out"))
    bias = torch.from_numpy(inp["bias"]).to(dev) if inp["bias"] is not None else None
    mx = cfg.prec == "mxfp8"
    s = m.shape(cfg.T, cfg.d, cfg.E, cfg.k, cfg.f, prec=m.MXFP8 if mx else m.BF16)
    buf = m.allocate(s)
    out = torch.empty(cfg.T, cfg.d, dtype=torch.bfloat16, device=dev)
    m.clear_error(buf.ws)
    for _ in range(args.warmup + args.steps):
        if mx:
            m.build_mx_weights(s, wg, wu, wd, buf.mx_weights)
        m.forward(buf, x, wr, bias, wg, wu, wd, out)
        m.backward(buf, dO, x, wr, wg, wu, wd)
    torch.cuda.synchronize()
    err = m.read_error(buf.ws)
    print(json.dumps({"profile_run": cfg.name, "steps": args.warmup + args.steps, "error_word": err}),
          flush=True)
    return 0 if err == 0 else 1


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", default="mxfp8")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the MXFP8 weight-gradient comparison")
    ap.add_argument("--mx-wgrad-only", action="store_true",
                    help="run only the MXFP8 weight-gradient comparison and print its JSON")
    ap.add_argument("--mx-wgrad-sizes", default="2048,4096,8192")
    ap.add_argument("--mx-wgrad-reps", type=int, default=10)
    ap.add_argument("--profile-run", action="store_true",
                    help="run warmup + steps whole layer steps untimed (the command ncu captures)")
    args = ap.parse_args(argv)
    from synth import CONFIGS
    cfg = CONFIGS[args.config]
    if args.impl == "reference":
        return run_reference(args, cfg)
    if args.mx_wgrad_only:
        return run_mx_wgrad_only(args)
    if args.profile_run:
        return run_profile(args, cfg)
    return run_ours(args, cfg)


def run_mx_wgrad_only(args):
    import torch
    import moe_expert_layer_softmax_gb300 as m
    m.load()
    torch.cuda.set_device(0)
    m.init(0)
    dev = torch.device("cuda", 0)
    stream = torch.cuda.Stream(device=dev)
    sizes = tuple(int(v) for v in args.mx_wgrad_sizes.split(","))
    res = mx_wgrad_variants(m, dev, stream, sizes=sizes, reps=args.mx_wgrad_reps)
    print(json.dumps({"mx_wgrad": res}), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
