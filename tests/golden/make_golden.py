"""Write the stored oracle values for the tiny fp32 workload.

Calls only ``oracle`` (and the shared seeded input generator).  The fixture is a
regression pin for the oracle and for the generator's cross-machine
determinism; the oracle's correctness itself is pinned by the closed-form,
brute-force and invariant tests in ``tests/test_oracle_pins.py``.

Usage:  python tests/golden/make_golden.py
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
from kda_inputs import WORKLOADS, make_prefill  # noqa: E402

OUT = os.path.join(HERE, "tiny_fp32_seed0.txt")


def main():
    wl = WORKLOADS[1]
    d = make_prefill(wl, seed=0)
    o, hT = oracle.forward(d["q"], d["k"], d["v"], d["beta"], d["decay"], d["h0"],
                           use_l2=wl.use_l2)
    rows = []
    # a fixed, spread-out sample of output entries and final-state entries
    for t in (0, 1, 15, 16, 31, 47, 63):
        for h in range(wl.H):
            for j in (0, 7, 19, 31):
                rows.append(("o", 0, t, h, j, o[0, t, h, j]))
    for h in range(wl.H):
        for i in (0, 5, 17, 31):
            for j in (0, 13, 31):
                rows.append(("hT", 0, h, i, j, hT[0, h, i, j]))
    with open(OUT, "w") as f:
        f.write("# Oracle values for the tiny fp32 workload (B=1 T=64 H=2 d=32, seed 0),\n")
        f.write("# written by tests/golden/make_golden.py (calls only the oracle).\n")
        f.write("# o rows: name b t h j value ; hT rows: name b h i j value\n")
        for r in rows:
            f.write(f"{r[0]} {r[1]} {r[2]} {r[3]} {r[4]} {r[5]:.17e}\n")
    print(f"wrote {len(rows)} values to {OUT}")


if __name__ == "__main__":
    main()
