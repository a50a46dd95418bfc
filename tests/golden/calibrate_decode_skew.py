"""Calibrates the decode workload's skew (writes decode_skew.json beside it).

The skewed decode workload shifts the first 16 experts' centroids by alpha
along the unit mean direction of a calibration draw; alpha is chosen by
bisection so that, with the oracle's routing of the T = 256 decode batch, the
16 hot experts receive 40% of all selections (within 0.005).  Calls only the
oracle and the seeded input generators.

    python tests/golden/calibrate_decode_skew.py
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from fine_grained_fp8_bias_b300 import workloads as wl  # noqa: E402
from oracle import oracle as orc  # noqa: E402

TARGET, TOL = 0.40, 0.005


def hot_fraction(alpha: float, T: int) -> float:
    cfg = wl.V3_DECODE.with_(hot_alpha=alpha, T=T)
    u = orc.bf16_bits(wl.tokens(cfg, "cpu"))
    r = orc.route(u, wl.centroids(cfg).numpy(), wl.bias(cfg).numpy(), cfg.K)
    return float((r["idx"] < cfg.hot_experts).mean())


def main():
    orc.build()
    lo, hi = 0.0, 8.0
    f_hi = hot_fraction(hi, 256)
    if f_hi < TARGET:
        raise SystemExit(f"alpha = {hi} reaches only {f_hi:.3f}")
    steps = []
    alpha, f = hi, f_hi
    for _ in range(30):
        alpha = 0.5 * (lo + hi)
        f = hot_fraction(alpha, 256)
        steps.append([round(alpha, 6), round(f, 6)])
        if abs(f - TARGET) <= TOL:
            break
        lo, hi = (alpha, hi) if f < TARGET else (lo, alpha)
    by_T = {str(T): round(hot_fraction(alpha, T), 6) for T in (1, 16, 64, 256)}
    rec = {"hot_alpha": round(alpha, 6), "hot_fraction_T256": round(f, 6), "target": TARGET,
           "tolerance": TOL, "hot_fraction_by_T": by_T, "bisection": steps,
           "how": "oracle routing (orc_route) of the seeded V3 decode batch; bisection of alpha "
                  "in [0, 8]; written by tests/golden/calibrate_decode_skew.py"}
    with open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "decode_skew.json"), "w") as fp:
        json.dump(rec, fp, indent=1)
    print(json.dumps(rec))


if __name__ == "__main__":
    main()
