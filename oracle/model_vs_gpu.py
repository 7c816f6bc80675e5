"""The first page's schedule cost model (Case 2, "Try this") against GPU timings.

Reads the JSON lines that `bench.py --experiments FILE` writes: M x 4096 x 4096 GEMMs with
the 128 x 128 tile and schedules built for 132 units. Prints, per shape, the measured time
of each schedule, the model's makespans at PART = 2 and PART = 8 (EPI = 2), and:
  - whether the hybrid rule's choice was the fastest of the four schedules on the GPU;
  - which PART makes the model pick the measured best.
For each PART it also fits the single free unit of the model, microseconds per
k-iteration plus a launch constant, by least squares. This is a report, not a parity
check: no number here feeds a test.

    python -m oracle.model_vs_gpu FILE      # FILE: the output of bench.py --experiments FILE
"""
from __future__ import annotations

import json
import sys

import numpy as np

from oracle import schedule as S

N = K = 4096
SMS = 132
FOUR = ["data-parallel", "split-K s=2", "split-K s=4", "stream-K"]


def model_rows(m: int, part: float, epi: float = 2.0):
    rows = S.report_rows(m, N, K, SMS, epi, part)[3]
    return {"data-parallel": rows[0][1], "split-K s=2": rows[1][1], "split-K s=4": rows[2][1],
            "stream-K": rows[3][1], "rule": rows[4][1], "rule_label": rows[4][0]}


def fit(points):
    """us = a + b * makespan by least squares; returns (a, b, rms relative error)."""
    x = np.array([p[0] for p in points], dtype=np.float64)
    y = np.array([p[1] for p in points], dtype=np.float64)
    X = np.stack([np.ones_like(x), x], axis=1)
    (a, b), *_ = np.linalg.lstsq(X, y, rcond=None)
    rel = (a + b * x - y) / y
    return float(a), float(b), float(np.sqrt(np.mean(rel ** 2)))


def main(path: str):
    lines = [json.loads(l) for l in open(path) if l.strip()]
    four = [l for l in lines if l["experiment"] == "rule_vs_four"]
    ms = sorted({l["M"] for l in four})
    meas = {(l["M"], l["schedule"]): l["us"] for l in four}
    parts = (2.0, 4.0, 8.0, 16.0)
    print(f"{'M':>5} | measured us: {'DP':>7} {'SK2':>7} {'SK4':>7} {'StrK':>7} {'rule':>7} | rule best? "
          f"| model best at PART=2 / 8 vs measured best")
    agree = {p: 0 for p in parts}
    rule_best = 0
    for m in ms:
        t = {n: meas[(m, n)] for n in FOUR + ["rule"]}
        best = min(FOUR, key=lambda n: t[n])
        ok = t["rule"] <= t[best] * 1.02  # within 2 %: timing noise at a few microseconds
        rule_best += ok
        picks = {}
        for p in parts:
            mr = model_rows(m, p)
            picks[p] = min(FOUR, key=lambda n: mr[n])
            agree[p] += picks[p] == best
        print(f"{m:5d} | {t['data-parallel']:20.1f} {t['split-K s=2']:7.1f} {t['split-K s=4']:7.1f} "
              f"{t['stream-K']:7.1f} {t['rule']:7.1f} | {'yes' if ok else 'no ':>9} | "
              f"{picks[2.0]:>13} / {picks[8.0]:>13} vs {best}")
    print(f"\nrule's choice within 2 % of the measured best: {rule_best}/{len(ms)} shapes")
    for p in parts:
        pts = []
        for m in ms:
            mr = model_rows(m, p)
            for n in FOUR:
                pts.append((mr[n], meas[(m, n)]))
        a, b, rms = fit(pts)
        print(f"PART={p:4.0f}: model picks the measured best on {agree[p]}/{len(ms)} shapes; "
              f"fit us = {a:.2f} + {b * 1e3:.1f} ns x makespan, rms relative error {rms:.1%}")
    sep = [l for l in lines if l["experiment"] == "separate_reduction_m128"]
    if sep:
        _, _, tiles, iters = S.problem_shape(128, N, K)
        print("\nM = 128: Split-K with the reduction as its own launch vs the owner's fixup and Stream-K")
        for l in sep:
            name = l["schedule"]
            s = int(name.split("s=")[1].split()[0]) if "s=" in name else 0
            if "separate reduction" in name:
                mk = {p: S.split_k_separate_makespan(tiles, iters, SMS, s, 2, p) for p in (2, 8)}
            elif "split-K" in name:
                mk = {p: S.split_k_makespan(tiles, iters, SMS, s, 2, p) for p in (2, 8)}
            elif "owner" in name:
                mk = {p: S.makespan(S.build_plan(128, N, K, SMS, S.STREAMK), 2, p) for p in (2, 8)}
            else:
                mk = {2: float("nan"), 8: float("nan")}
            print(f"  {name:36s} {l['us']:7.1f} us  model PART=2 {mk[2]:6.1f}  PART=8 {mk[8]:6.1f}  launches {l['launches']}")


if __name__ == "__main__":
    main(sys.argv[1])
