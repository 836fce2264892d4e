"""Derives the Zipf offset scale of the imbalanced workload with the oracle's
router and writes tests/golden/zipf_beta.json.

    python tests/golden/make_zipf_beta.py

The workload (T=16384, d=4096, E=128, I=1536, top-8, seed 0) biases router
logits by b_e = -beta * 1.1 * ln(rank_e).  beta is found by bisection so that
the hottest expert receives 8x the mean number of rows (R/E); the script
calls only the oracle's routing and the seeded input generator.
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
from routing_dispatch_grouped_router_gb300 import inputs as gen  # noqa: E402


def hot_ratio(x, wr, shape, s, beta, seed):
    bias = gen.make_zipf_bias(shape, seed, s, beta)
    idx, _, _, flagged, _ = oracle.route_ref(x, wr, bias, shape.k)
    counts = np.bincount(idx.ravel(), minlength=shape.E)
    return counts.max() / (shape.R / shape.E), int(flagged.sum())


def main():
    shape = gen.workload_shape("imbalanced")
    s = gen.WORKLOADS["imbalanced"]["zipf_s"]
    seed = 0
    x = gen.make_x(shape, seed)
    wr = gen.make_router(shape, seed)
    lo, hi = 0.0, 4.0
    target = 8.0
    for _ in range(24):
        mid = 0.5 * (lo + hi)
        r, _ = hot_ratio(x, wr, shape, s, mid, seed)
        if r < target:
            lo = mid
        else:
            hi = mid
    beta = round(0.5 * (lo + hi), 6)
    ratio, flagged = hot_ratio(x, wr, shape, s, beta, seed)
    out = {"workload": "imbalanced", "seed": seed, "zipf_s": s, "beta": beta,
           "hot_over_mean": float(ratio), "near_tie_tokens": flagged,
           "written_by": "tests/golden/make_zipf_beta.py (oracle.route_ref bisection)"}
    with open(os.path.join(HERE, "zipf_beta.json"), "w") as f:
        json.dump(out, f, indent=1)
    print(out)


if __name__ == "__main__":
    main()
