"""Choose the Zipf router-bias strength of the skewed workload.

The skewed workload (T=4096, 128 experts, top-6) biases the router logits by
bias_e = -c * 1.2 * ln(rank_e) (rank_e a seeded permutation of 1..128) and
pins the four lowest-ranked experts at -30 so that some experts get no
tokens.  This script routes the seed-0 tokens with the CPU oracle for a
range of c, bisects for max(count)/mean(count) = 8, and prints the constant
that moe_synth.SKEW_C holds.  It calls only the oracle and the generator.

    python tests/golden/calibrate_skew.py
"""
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__)))))

import moe_synth  # noqa: E402
import oracle  # noqa: E402


def ratio(c, seed=0):
    inp = moe_synth.make_inputs("skew", seed=seed, router_only=True, skew_c=c)
    x = oracle.x_values(inp)
    _, ids, _ = oracle.route(x, inp.w_router, inp.bias, inp.cfg.k)
    counts = np.bincount(ids.reshape(-1), minlength=inp.cfg.E)
    return counts.max() / counts.mean(), int((counts == 0).sum())


def main():
    lo, hi = 0.0, 1.0
    for _ in range(30):
        mid = 0.5 * (lo + hi)
        r, _ = ratio(mid)
        if r < 8.0:
            lo = mid
        else:
            hi = mid
    c = round(0.5 * (lo + hi), 4)
    r, empty = ratio(c)
    print(f"SKEW_C = {c}  (max/mean = {r:.3f}, empty experts = {empty})")


if __name__ == "__main__":
    main()
