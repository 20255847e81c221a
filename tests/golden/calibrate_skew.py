"""Calibrate the skew-sweep bias temperature (``synth.SKEW_TAU``).

The skew sweep draws e_score_correction_bias = -1.1 * tau * ln(rank_e) over a seeded
permutation of the 896 experts, so that expert popularity follows a Zipf law with
exponent 1.1. This script finds tau by bisection: it routes the seed-0 inputs at
T = 4096 with the oracle (FP64 router logits rounded to FP32, oracle sigmoid top-16)
and fits the log-log slope of the sorted expert loads; the target is -1.1 +- 0.05.
It calls only the oracle and the input generators. Run from the repository root:

    python tests/golden/calibrate_skew.py

and copy the printed tau into ``synth.SKEW_TAU``.
"""
import os
import sys
from concurrent.futures import ThreadPoolExecutor

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__)))))

import oracle  # noqa: E402
import synth  # noqa: E402


def load_slope(ids: np.ndarray) -> float:
    loads = np.sort(np.bincount(ids.ravel(), minlength=synth.E))[::-1].astype(np.float64)
    r = np.arange(1, loads.size + 1, dtype=np.float64)
    keep = loads > 0
    return float(np.polyfit(np.log(r[keep]), np.log(loads[keep]), 1)[0])


def main(T: int = 4096, seed: int = 0) -> float:
    x = synth.hidden_rows(T, seed)
    w = synth.router_weight(seed)
    chunks = np.array_split(np.arange(T), os.cpu_count() or 1)
    with ThreadPoolExecutor(len(chunks)) as ex:
        parts = list(ex.map(lambda c: oracle.router_logits(x[c[0]:c[-1] + 1], w)[0], chunks))
    logits = np.concatenate(parts).astype(np.float32)

    def slope(tau):
        ids, _, _ = oracle.topk_route(logits, synth.skew_bias(seed, tau=tau), 16)
        return load_slope(ids)

    lo, hi = 0.0, 2.0
    for _ in range(40):
        mid = 0.5 * (lo + hi)
        if slope(mid) > -1.1:
            lo = mid
        else:
            hi = mid
    tau = round(0.5 * (lo + hi), 4)
    s = slope(tau)
    print(f"tau = {tau}  slope = {s:.4f}")
    assert abs(s + 1.1) <= 0.05, s
    return tau


if __name__ == "__main__":
    main()
