"""The oracle reproduces its stored values for the tiny fp32 workload."""
import os

import numpy as np

from kda_inputs import WORKLOADS, make_prefill

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "tiny_fp32_seed0.txt")


def _read():
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            name, a, b, c, d, val = line.split()
            rows.append((name, int(a), int(b), int(c), int(d), float(val)))
    return rows


def test_tiny_golden(oracle_mod):
    wl = WORKLOADS[1]
    d = make_prefill(wl, seed=0)
    o, hT = oracle_mod.forward(d["q"], d["k"], d["v"], d["beta"], d["decay"], d["h0"],
                               use_l2=wl.use_l2)
    rows = _read()
    assert len(rows) > 50
    for name, a, b, c, e, val in rows:
        got = o[a, b, c, e] if name == "o" else hT[a, b, c, e]
        assert abs(got - val) <= 1e-12 * max(1.0, abs(val)), (name, a, b, c, e, got, val)


def test_generator_is_deterministic():
    wl = WORKLOADS[1]
    d1 = make_prefill(wl, seed=0)
    d2 = make_prefill(wl, seed=0)
    d3 = make_prefill(wl, seed=1)
    for key in ("q", "k", "v", "beta", "decay"):
        assert np.array_equal(d1[key], d2[key])
        assert not np.array_equal(d1[key], d3[key])
    assert d1["h0"] is None
    assert np.all(d1["decay"] <= 0) and np.all((d1["beta"] > 0) & (d1["beta"] < 1))
