"""Calibrate the synthetic router's Zipf alpha to target maxvio values.

Writes ``load_balancing_topk_gb300/zipf_alpha.json``, the table that
``synth.alpha_for`` reads (inputs, not expected values). It calls only the seeded input
generator and the CPU oracle (``oracle.counts`` / ``oracle.maxvio``): maxvio
is max_e T_e / T_bar - 1 ("月之暗面开源MoonEP：面向MoE训练的专家并行通信库",
section 解决的核心问题). For each workload and target, alpha is bisected at
seed 0 until the realised maxvio is within 0.5% of the target.

Run from the repository root:  python tests/golden/calibrate_alpha.py
"""

import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from load_balancing_topk_gb300 import synth  # noqa: E402

TARGETS = {
    "medium": [0.5],
    "large": [0.5, 1.0, 2.0, 4.0],
    "stress": [10.0],
}


def realised(shape, alpha, seed=0):
    idx, _ = synth.routing(shape, seed=seed, alpha=alpha)
    c = oracle.counts(idx, shape.E)
    return oracle.maxvio(c, shape.R, shape.S, shape.K)


def calibrate(shape, target, lo=0.0, hi=4.0, rel=0.005, iters=40):
    mid = None
    for _ in range(iters):
        mid = 0.5 * (lo + hi)
        m = realised(shape, mid)
        if abs(m - target) <= rel * target:
            return mid, m
        if m < target:
            lo = mid
        else:
            hi = mid
    return mid, realised(shape, mid)


def main():
    table = {}
    for name, targets in TARGETS.items():
        shape = synth.SHAPES[name]
        table[name] = {}
        for tgt in targets:
            a, m = calibrate(shape, tgt)
            table[name][f"{tgt:g}"] = round(a, 6)
            print(f"{name} target {tgt:g}: alpha {a:.6f} -> maxvio {m:.4f}", flush=True)
    out = os.path.join(ROOT, "load_balancing_topk_gb300", "zipf_alpha.json")
    with open(out, "w") as f:
        json.dump(table, f, indent=1, sort_keys=True)
        f.write("\n")


if __name__ == "__main__":
    main()
