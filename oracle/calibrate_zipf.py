"""Pick the Zipf bias strength of the skewed-routing workload with the oracle.

The skewed workload asks for router logits N(0, 1) plus a Zipf(s = 1.2)
per-expert bias strong enough that the busiest expert receives about 8x the
mean load.  This script bisects the bias scale beta on the seed-0 logits,
routing with the CPU oracle, until max/mean load lies in [7.5, 8.5], and
prints the value stored as ``SKEWED_ZIPF_BETA`` in
``activation_paging_gb300/inputs.py``.  It calls only the oracle and the
input generator.

    python -m oracle.calibrate_zipf
"""
from __future__ import annotations

import numpy as np

import oracle
from activation_paging_gb300 import inputs


def load_ratio(beta: float, wl) -> float:
    logits = inputs.router_logits(wl.seed, wl.T, wl.E, wl.zipf_s, beta)
    idx, _ = oracle.route_topk(logits, wl.k)
    counts = oracle.dispatch_plan(idx, wl.E, 0, False)["counts"]
    return float(counts.max()) / (wl.T * wl.k / wl.E)


def calibrate(wl=None, lo: float = 0.0, hi: float = 4.0, target=(7.5, 8.5), steps: int = 40) -> float:
    wl = wl or inputs.WORKLOADS["skewed"]
    for _ in range(steps):
        mid = (lo + hi) / 2
        r = load_ratio(mid, wl)
        if target[0] <= r <= target[1]:
            return mid
        if r < target[0]:
            lo = mid
        else:
            hi = mid
    raise RuntimeError("no beta reached the target load ratio")


if __name__ == "__main__":
    beta = calibrate()
    print(f"SKEWED_ZIPF_BETA = {beta!r}  (max/mean load {load_ratio(beta, inputs.WORKLOADS['skewed']):.3f})")
