"""Pins for the oracle's gate and beta transforms (ejkernel kernel_delta_attention, kda_decay:
decay = -exp(A_log) softplus(gate + dt_bias), never positive; TileOPs GDNFwdOp / KDAFwdOp:
beta = sigmoid(x), or 2 sigmoid(x) with allow_neg_eigval), each against values fixed by the
mathematics rather than a retyped formula."""
import math

import numpy as np
import pytest


def test_kda_decay_doctest_case(oracle_mod):
    """The page's example: zero gate, A_log and dt_bias of shapes (2, 10, 4), (4,), (4,); the
    decay is non-positive.  With those zeros it is -exp(0) log(1 + e^0) = -ln 2 exactly."""
    d = oracle_mod.gate_decay(np.zeros((2, 10, 4)), np.zeros(4), np.zeros(4))
    assert d.shape == (2, 10, 4)
    assert np.all(d <= 0)
    assert np.all(d == -math.log(2.0))


def test_kda_decay_never_positive_and_monotone(oracle_mod):
    rng = np.random.default_rng(0)
    g = (4 * rng.standard_normal((3, 50, 5))).astype(np.float32)
    a = rng.standard_normal(5).astype(np.float32)
    b = rng.standard_normal(5).astype(np.float32)
    d = oracle_mod.gate_decay(g, a, b)
    assert np.all(d < 0)
    # a larger gate decays more: d is decreasing in the gate
    d2 = oracle_mod.gate_decay(g + 0.5, a, b)
    assert np.all(d2 < d)


def test_kda_decay_special_values(oracle_mod):
    # dt_bias shifts the gate; A_log scales by exp(A_log): A_log = ln 3 triples the decay
    g = np.array([[[0.0, 1.0, -2.0]]], dtype=np.float32)
    base = oracle_mod.gate_decay(g, np.zeros(3), None)
    assert np.allclose(base[0, 0], [-math.log(2.0), -math.log1p(math.e), -math.log1p(math.exp(-2.0))],
                       rtol=1e-15)
    a3 = np.float32(math.log(3.0))                            # ln 3 as stored (float32)
    tripled = oracle_mod.gate_decay(g, np.full(3, a3, np.float32), None)
    assert np.allclose(tripled, base * math.exp(float(a3)), rtol=1e-15)
    assert np.allclose(tripled, 3 * base, rtol=1e-7)
    shifted = oracle_mod.gate_decay(g - 1.0, np.zeros(3), np.ones(3))
    assert np.allclose(shifted, base, rtol=1e-15)
    # asymptotes: softplus(x) -> x for large x, -> e^x for very negative x
    big = oracle_mod.gate_decay(np.full((1, 1, 1), 60.0), np.zeros(1), None)
    assert big[0, 0, 0] == -60.0
    tiny = oracle_mod.gate_decay(np.full((1, 1, 1), -40.0), np.zeros(1), None)
    assert math.isclose(tiny[0, 0, 0], -math.exp(-40.0), rel_tol=1e-12)


def test_kda_decay_per_channel_bias_layout(oracle_mod):
    """[rows, H, K] gates with dt_bias [H, K]: channel c of head h gets bias[h, c].  A bias of
    -gate at one (h, c) gives exactly -exp(A_log[h]) ln 2 there."""
    H, K = 3, 4
    g = np.arange(2 * H * K, dtype=np.float32).reshape(2, H, K) * 0.25
    bias = np.zeros((H, K), np.float32)
    bias[2, 1] = -g[1, 2, 1]
    a = np.array([0.0, 0.5, 1.0], np.float32)
    d = oracle_mod.gate_decay(g, a, bias)
    assert d.shape == (2, H, K)
    assert d[1, 2, 1] == -math.exp(np.float64(np.float32(1.0))) * math.log(2.0)
    assert np.all(d <= 0)


@pytest.mark.parametrize("neg", [False, True])
def test_beta_transform(oracle_mod, neg):
    x = np.array([0.0, 1.5, -1.5, 40.0, -40.0], np.float32)
    b = oracle_mod.beta_transform(x, allow_neg_eigval=neg)
    m = 2.0 if neg else 1.0
    assert b[0] == 0.5 * m                                   # sigmoid(0)
    assert math.isclose(b[1] + b[2], m, rel_tol=1e-15)       # sigmoid(x) + sigmoid(-x) = 1
    assert math.isclose(b[3], m, rel_tol=1e-15) and b[4] < 1e-17 * m
    assert np.all(np.diff(oracle_mod.beta_transform(np.linspace(-5, 5, 11), neg)) > 0)
