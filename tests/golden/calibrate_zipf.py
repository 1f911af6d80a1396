"""Calibrate the Zipf router bias of the skewed workload (writes zipf_calibration.json).

The skewed workload adds a per-expert bias beta * ln(r^-1.2) (r = popularity
rank of the expert) to x . W_r and drives the 4 least popular experts to zero
tokens.  beta is chosen by bisection so that the most popular expert receives
15% of all routes; the routing itself is computed by the oracle only.

Run:  python tests/golden/calibrate_zipf.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

from oracle import cpp as O          # noqa: E402
from synth import CONFIGS, make_inputs, zipf_expert_bias  # noqa: E402

TARGET = 0.15


def top_share(base_logits, E, k, seed, beta):
    logits = base_logits + zipf_expert_bias(E, seed, beta)[None, :].astype(np.float64)
    idx, _ = O.softmax_topk_gates(logits, k)
    counts = O.expert_counts(idx, E)
    return counts.max() / idx.size, int((counts == 0).sum()), counts


def main():
    cfg = CONFIGS["skewed"]
    inp = make_inputs(cfg, seed=0, routing="none", with_grad=False)
    base = O.router_logits(inp["x"], inp["w_router"], None)
    lo, hi = 0.0, 8.0
    for _ in range(40):
        mid = 0.5 * (lo + hi)
        share, _, _ = top_share(base, cfg.E, cfg.k, 0, mid)
        if share < TARGET:
            lo = mid
        else:
            hi = mid
    beta = round(0.5 * (lo + hi), 6)
    share, empty, counts = top_share(base, cfg.E, cfg.k, 0, beta)
    out = {
        "skewed": {
            "beta": beta, "seed": 0, "top_share": round(float(share), 6), "empty_experts": empty,
            "max_count": int(counts.max()), "target_top_share": TARGET,
        }
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "zipf_calibration.json")
    with open(path, "w") as fh:
        json.dump(out, fh, indent=1)
        fh.write("\n")
    print(json.dumps(out))


if __name__ == "__main__":
    main()
