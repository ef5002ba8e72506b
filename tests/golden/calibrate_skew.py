"""Calibrate the skew workload's router bias with the oracle router.

Writes tests/golden/skew_calibration.json. The chosen strength is copied by
hand into moe_synth.SKEW_KAPPA; tests/test_synth.py checks the two agree.

Target: with T = 2048 tokens of the DiffusionGemma MoE layer (H 2816, E 128,
top-8) and a Zipf(1.2) per-expert offset, the 13 most-loaded experts (10%)
receive 60 +- 5% of the slots and at least three experts receive none.
Usage: python tests/golden/calibrate_skew.py
"""
import dataclasses
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)
import moe_synth as ms  # noqa: E402
import oracle  # noqa: E402


def stats(kappa: float):
    wl = dataclasses.replace(ms.WORKLOADS["skew"], skew_kappa=kappa)
    d = wl.dims
    x = ms.make_x(d, wl.seed, mu=wl.skew_mu)
    wr, sc, pes = ms.make_router(d, wl.seed, kappa=kappa, zipf_s=wl.zipf_s)
    idx = oracle.route(d, x, wr, sc, pes)["idx"]
    cnt = np.bincount(idx.ravel(), minlength=d.E)
    top = np.sort(cnt)[::-1][: round(0.1 * d.E)].sum() / cnt.sum()
    return float(top), int((cnt == 0).sum()), cnt


def main():
    grid = [round(0.00002 * i, 5) for i in range(5, 50)]
    rows = []
    best = None
    for kappa in grid:
        top, empty, _ = stats(kappa)
        rows.append(dict(kappa=kappa, top10pct_share=round(top, 4), empty_experts=empty))
        print(rows[-1], flush=True)
        if empty >= 3 and abs(top - 0.60) <= 0.05:
            if best is None or abs(top - 0.60) < abs(best["top10pct_share"] - 0.60):
                best = rows[-1]
        if top > 0.70:
            break
    assert best is not None, "no kappa on the grid meets the target"
    out = dict(target="top 13 of 128 experts take 60 +- 5% of slots; >= 3 experts empty",
               workload="skew: T=2048, H=2816, E=128, k=8, I=704, g=64, seed 0, mu=1.0, zipf_s=1.2",
               chosen=best, grid=rows)
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "skew_calibration.json")
    with open(path, "w") as fh:
        json.dump(out, fh, indent=1)
    print("chosen", best)


if __name__ == "__main__":
    main()
