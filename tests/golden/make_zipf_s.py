"""Writes tests/golden/zipf_s.json: the Zipf exponent s of the routing-imbalance
workload (T=16384, d=4096, E=64, k=6) for a hottest-expert load of 1x, 2x and
4x the mean.

The per-expert logit bias is bias_e = -s * ln(rank_e) (rank a seeded
permutation of 1..E).  s is found by bisection on the load of the hottest
expert, as counted from the CPU oracle's routing of the workload's seeded
token rows, until max/mean is within 2 % of the target (s = 0 for 1x).  Only
the oracle computes routing here.

    python tests/golden/make_zipf_s.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from routing_permute_grouped_gb300 import synth  # noqa: E402
from tests.helpers import bits  # noqa: E402


def hot_ratio(L0, bias, k):
    idx, _, _ = oracle.route(L0 + bias[None, :].astype(np.float64), k)
    counts = np.bincount(idx.reshape(-1), minlength=L0.shape[1])
    return counts.max() / counts.mean()


def main():
    out = {}
    for pad in (64, 128):
        for target in (1.0, 2.0, 4.0):
            shape = synth.WORKLOADS[f"imbalance_x{int(target)}_p{pad}"]
            inp = synth.make_inputs(shape, zipf_s=0.0)
            L0 = oracle.router_logits(bits(inp["x"]), bits(inp["Wg"]), None)
            if target == 1.0:
                s = 0.0
            else:
                lo, hi = 0.0, 4.0
                for _ in range(40):
                    mid = 0.5 * (lo + hi)
                    r = hot_ratio(L0, synth.zipf_bias(shape.E, mid, shape.seed).numpy(), shape.k)
                    if abs(r - target) <= 0.02 * target:
                        lo = hi = mid
                        break
                    if r < target:
                        lo = mid
                    else:
                        hi = mid
                s = 0.5 * (lo + hi)
            r = hot_ratio(L0, synth.zipf_bias(shape.E, s, shape.seed).numpy(), shape.k)
            out[shape.name] = s
            out[shape.name + "_hot_over_mean"] = round(float(r), 4)
            print(shape.name, s, r, flush=True)
    with open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "zipf_s.json"), "w") as f:
        json.dump(out, f, indent=1, sort_keys=True)


if __name__ == "__main__":
    main()
