"""The seeded input generators shared by the oracle's tests and the GPU tests (no GPU): the
bf16 rounding against torch's own conversion, the named workloads' shapes and recipes, and
the value ranges of every drawn quantity."""
import numpy as np
import pytest

from kda_inputs import WORKLOADS, make_custom, make_gk, make_varlen, round_to_bf16


def test_round_to_bf16_is_round_to_nearest_even():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(5)
    x = np.concatenate([rng.standard_normal(20000).astype(np.float32) * 10.0 ** rng.integers(-6, 6, 20000),
                        np.array([0.0, -0.0, 1.0, -2.5, 3.0e38, -3.0e38, 1e-40], np.float32)])
    want = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    got = round_to_bf16(x)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
    # ties go to the even neighbour: 1 + 2^-8 lies halfway between 1 and 1 + 2^-7
    assert round_to_bf16(np.float32([1 + 2.0 ** -8]))[0] == 1.0
    assert round_to_bf16(np.float32([1 + 3 * 2.0 ** -8]))[0] == 1 + 2.0 ** -6
    assert np.array_equal(round_to_bf16(got), got)   # bf16 values are fixed points


def test_named_workloads():
    w1, w2, w3, w4, w5 = (WORKLOADS[i] for i in range(1, 6))
    assert (w1.dtype, w1.B, w1.T, w1.H, w1.dk, w1.dv, w1.chunk, w1.h0) == ("f32", 1, 64, 2, 32, 32, 16, "zero")
    assert (w2.dtype, w2.B, w2.T, w2.H, w2.dk, w2.chunk, w2.decay) == ("bf16", 2, 2048, 16, 128, 64, "train")
    assert (w3.dtype, w3.B, w3.T, w3.H, w3.dk, w3.dv, w3.decay, w3.h0) == \
        ("bf16", 1, 32768, 32, 128, 128, "long", "normal002")
    assert (w4.kind, w4.B, w4.H, w4.dk, w4.steps) == ("decode", 256, 32, 128, 128)
    assert (w5.kind, w5.nseq, w5.len_range, w5.H, w5.dk, w5.decay) == ("varlen", 16, (256, 4096), 16, 64, "none")
    assert all(w.use_l2 for w in WORKLOADS.values())


@pytest.mark.parametrize("kind", ["small", "train", "long", "strong", "mixed"])
def test_drawn_ranges(kind):
    d = make_custom(2, 256, 3, 32, 16, dtype="bf16", decay=kind, h0="normal002", seed=7)
    assert d["q"].shape == (2, 256, 3, 32) and d["v"].shape == (2, 256, 3, 16)
    for n in ("q", "k", "v"):   # bf16 workloads hold bf16 values
        assert np.array_equal(round_to_bf16(d[n]), d[n])
    assert np.all((d["beta"] > 0) & (d["beta"] < 1))
    assert np.all(d["decay"] <= 0) and np.all(np.isfinite(d["decay"]))
    assert d["h0"].shape == (2, 3, 32, 16) and 0.015 < d["h0"].std() < 0.025
    if kind == "long":   # -softplus(N(-4, 1)): small, strictly negative per-token decays
        assert np.all(d["decay"] < 0) and 0.01 < -d["decay"].mean() < 0.05
    if kind == "strong":
        assert np.all(d["decay"] <= -1.0)


def test_varlen_and_per_channel_recipes():
    d = make_varlen(WORKLOADS[5], seed=0)
    cu = d["cu_seqlens"]
    lengths = np.diff(cu)
    assert cu.dtype == np.int32 and cu[0] == 0 and len(cu) == 17
    assert np.all((lengths >= 256) & (lengths <= 4096))
    assert d["q"].shape == (1, int(cu[-1]), 16, 64) and d.get("decay") is None
    g = make_gk(1, 64, 2, 32, 32, gate_scale=0.3, seed=3)
    assert g["g"].shape == (1, 64, 2, 32) and np.all((g["g"] <= 0) & (g["g"] > -0.3))
