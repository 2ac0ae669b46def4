"""Pins for the oracle's per-key-channel decay (TileOPs "Linear Attention Operators",
KDAFwdOp: one log decay per key channel, g [B,T,H,K]; GLARecurrentFwdOp prints the
retention as diag(exp(gk)) applied to the state).  Each check is computed in the test
from mathematics that does not go through the oracle's per-channel code:

* brute force with explicit dk x dk transition matrices, both decay placements;
* every channel sharing one decay gives the scalar oracle (itself pinned elsewhere);
* no decay: both placements give the ungated scalar oracle;
* the decayed read with a shared decay equals the undecayed read with rescaled
  beta and v (an identity of the two transition matrices, via the scalar oracle);
* one-hot keys on a single channel: a closed geometric form per row, which fixes
  both the placement and which channel's decay scales which row;
* beta = 0: pure per-channel exponential decay of the initial state;
* the chunked per-channel form equals the per-channel scan for every chunk size,
  including decays strong enough that a chunk spans e^-100 in some channels;
* packed sequences equal separate calls.
"""
import numpy as np
import pytest

from kda_inputs import make_gk

EXACT = 1e-12


def _l2(x):
    x = np.asarray(x, np.float64)
    return x / np.maximum(np.sqrt(np.sum(x * x, axis=-1, keepdims=True)), 1e-12)


def _rel(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


def _rand(seed, B, T, H, dk, dv, gate, h0=True, f32=True):
    d = make_gk(B, T, H, dk, dv, dtype="f32" if f32 else "bf16", gate_scale=gate,
                h0="normal002" if h0 else "zero", seed=seed)
    if h0:
        d["h0"] = d["h0"] * 50.0   # O(1) initial memory, so that its decay is visible
    return d


# ---------------------------------------------------------------------------
# Brute force.  Transition matrices, written from the two placements:
#   undecayed read: h_t = (D_t - beta_t k k^T) h_{t-1} + beta_t k v^T
#   decayed read:   h_t = (I - beta_t k k^T) D_t h_{t-1} + beta_t k v^T
# h_t is rebuilt from scratch for every t as a product of these matrices.
# ---------------------------------------------------------------------------
def _bruteforce(q, k, v, beta, g, h0, scale, decayed):
    T, dk = k.shape
    kk = _l2(k)
    qq = _l2(q) * scale
    A = []
    for t in range(T):
        D = np.diag(np.exp(g[t].astype(np.float64)))
        P = np.outer(kk[t], kk[t]) * float(beta[t])
        A.append((np.eye(dk) - P) @ D if decayed else D - P)
    o = np.zeros((T, v.shape[1]))
    for t in range(T):
        M = np.eye(dk)
        h = np.zeros_like(h0)
        for s in range(t, -1, -1):           # s = t, t-1, ..., 0: M = A_t ... A_{s+1}
            h = h + M @ (float(beta[s]) * np.outer(kk[s], v[s]))
            M = M @ A[s]
        h = h + M @ h0                       # M = A_t ... A_0
        o[t] = h.T @ qq[t]
    return o, h


@pytest.mark.parametrize("decayed", [False, True])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_bruteforce(oracle_mod, decayed, seed):
    T, dk, dv = 7, 4, 3
    d = _rand(seed, 1, T, 1, dk, dv, gate=1.5)
    scale = 0.7
    ro, rh = _bruteforce(d["q"][0, :, 0], d["k"][0, :, 0], d["v"][0, :, 0],
                         d["beta"][0, :, 0], d["g"][0, :, 0], d["h0"][0, 0].astype(np.float64),
                         scale, decayed)
    for chunk in (None, 1, 3, 4, 8):
        o, h = oracle_mod.forward_gk(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"],
                                     scale=scale, decayed_read=decayed, chunk=chunk)
        assert _rel(o[0, :, 0], ro) < EXACT, chunk
        assert _rel(h[0, 0], rh) < EXACT, chunk


# ---------------------------------------------------------------------------
# All channels share one decay: the per-channel oracle equals the scalar one.
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("chunk", [None, 16, 64])
def test_shared_decay_is_scalar(oracle_mod, chunk):
    B, T, H, dk, dv = 2, 77, 3, 16, 8
    d = _rand(3, B, T, H, dk, dv, gate=0.8)
    dec = d["g"][..., 0].copy()
    g = np.repeat(dec[..., None], dk, axis=-1)
    o1, h1 = oracle_mod.forward(d["q"], d["k"], d["v"], d["beta"], dec, d["h0"], chunk=chunk)
    o2, h2 = oracle_mod.forward_gk(d["q"], d["k"], d["v"], d["beta"], g, d["h0"], chunk=chunk)
    assert _rel(o2, o1) < EXACT and _rel(h2, h1) < EXACT


@pytest.mark.parametrize("decayed", [False, True])
def test_no_decay_is_ungated(oracle_mod, decayed):
    B, T, H, dk, dv = 1, 50, 2, 8, 8
    d = _rand(4, B, T, H, dk, dv, gate=1.0)
    o1, h1 = oracle_mod.forward(d["q"], d["k"], d["v"], d["beta"], None, d["h0"])
    for g in (None, np.zeros_like(d["g"])):
        o2, h2 = oracle_mod.forward_gk(d["q"], d["k"], d["v"], d["beta"], g, d["h0"],
                                       decayed_read=decayed)
        assert _rel(o2, o1) < EXACT and _rel(h2, h1) < EXACT


def test_decayed_read_identity(oracle_mod):
    """With |k| = 1 and one decay a per token, (I - b k k^T) a = a I - (a b) k k^T and
    b k v^T = (a b) k (v / a)^T: the decayed read with (beta, v) is the undecayed read
    with (a beta, v / a).  The right side runs through the scalar oracle."""
    B, T, H, dk, dv = 1, 40, 2, 8, 6
    d = _rand(5, B, T, H, dk, dv, gate=0.6)
    dec = d["g"][..., 0].copy()
    g = np.repeat(dec[..., None], dk, axis=-1)
    a = np.exp(dec.astype(np.float64))
    beta2 = (d["beta"] * a).astype(np.float64)
    v2 = d["v"] / a[..., None]
    # the scalar oracle takes float32 inputs: keep the rescaled ones exact by checking
    # against a float64 brute force when rounding would matter
    o1, h1 = oracle_mod.forward_gk(d["q"], d["k"], d["v"], d["beta"], g, d["h0"],
                                   decayed_read=True)
    ro = np.zeros((T, dv))
    for hh in range(H):
        ro, rh = _bruteforce(d["q"][0, :, hh], d["k"][0, :, hh], v2[0, :, hh], beta2[0, :, hh],
                             np.zeros((T, dk)) + dec[0, :, hh, None], d["h0"][0, hh].astype(np.float64),
                             dk ** -0.5, False)
        assert _rel(o1[0, :, hh], ro) < 1e-11
        assert _rel(h1[0, hh], rh) < 1e-11
    # and the same through the scalar oracle with the float32-rounded rescaling
    o2, h2 = oracle_mod.forward(d["q"], d["k"], v2.astype(np.float32), beta2.astype(np.float32),
                                dec, d["h0"])
    assert _rel(o2, o1) < 1e-5 and _rel(h2, h1) < 1e-5


# ---------------------------------------------------------------------------
# One-hot keys on channel j: rows i != j only decay, h_T[i] = exp(sum_t g_t[i]) h_0[i];
# row j follows x <- c_t x + beta_t v_t with c_t = a_t - beta_t (undecayed read) or
# a_t (1 - beta_t) (decayed read), a_t = exp(g_t[j]).  Closed form:
#   h_T[j] = (prod_t c_t) h_0[j] + sum_t beta_t (prod_{s>t} c_s) v_t.
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("decayed", [False, True])
@pytest.mark.parametrize("j", [0, 5])
def test_onehot_closed_form(oracle_mod, decayed, j):
    T, dk, dv = 30, 8, 5
    d = _rand(6, 1, T, 1, dk, dv, gate=0.5)
    k = np.zeros_like(d["k"])
    k[..., j] = 1.0
    g = d["g"][0, :, 0].astype(np.float64)
    beta = d["beta"][0, :, 0].astype(np.float64)
    v = d["v"][0, :, 0].astype(np.float64)
    h0 = d["h0"][0, 0].astype(np.float64)
    a = np.exp(g[:, j])
    c = a * (1.0 - beta) if decayed else a - beta
    ref = np.exp(g.sum(axis=0))[:, None] * h0
    row = np.prod(c) * h0[j]
    for t in range(T):
        row = row + beta[t] * np.prod(c[t + 1:]) * v[t]
    ref[j] = row
    for chunk in (None, 8, 64):
        _, h = oracle_mod.forward_gk(d["q"], k, d["v"], d["beta"], d["g"], d["h0"],
                                     decayed_read=decayed, chunk=chunk)
        assert _rel(h[0, 0], ref) < EXACT, chunk


@pytest.mark.parametrize("decayed", [False, True])
def test_beta_zero_pure_decay(oracle_mod, decayed):
    T, H, dk, dv = 25, 2, 8, 4
    d = _rand(7, 1, T, H, dk, dv, gate=0.9)
    beta = np.zeros_like(d["beta"])
    G = np.cumsum(d["g"].astype(np.float64), axis=1)     # [1,T,H,dk]
    qq = _l2(d["q"]) * dk ** -0.5
    h0 = d["h0"].astype(np.float64)
    ro = np.einsum("thi,hij->thj", qq[0] * np.exp(G[0]), h0[0])[None]
    rh = np.exp(G[0, -1])[..., None] * h0[0]
    for chunk in (None, 16):
        o, h = oracle_mod.forward_gk(d["q"], d["k"], d["v"], beta, d["g"], d["h0"],
                                     decayed_read=decayed, chunk=chunk)
        assert _rel(o, ro) < EXACT and _rel(h[0], rh) < EXACT


@pytest.mark.parametrize("decayed", [False, True])
@pytest.mark.parametrize("gate", [0.01, 0.3, 2.0, 6.0])
def test_chunked_equals_scan(oracle_mod, decayed, gate):
    """gate 6.0: about -3 per token and channel, a 64-token chunk spans ~e^-190."""
    B, T, H, dk, dv = 1, 131, 2, 16, 8
    d = _rand(8, B, T, H, dk, dv, gate=gate)
    o0, h0 = oracle_mod.forward_gk(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"],
                                   decayed_read=decayed)
    assert np.all(np.isfinite(o0)) and np.all(np.isfinite(h0))
    for chunk in (1, 16, 64):
        o, h = oracle_mod.forward_gk(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"],
                                     decayed_read=decayed, chunk=chunk)
        assert _rel(o, o0) < 1e-11 and _rel(h, h0) < 1e-11, chunk


def test_packed_equals_separate(oracle_mod):
    lengths = [0, 17, 64, 5]
    H, dk, dv = 2, 8, 8
    d = make_gk(1, 0, H, dk, dv, dtype="f32", gate_scale=0.5, h0="normal002", seed=9,
                lengths=lengths)
    cu = d["cu_seqlens"]
    o, h = oracle_mod.forward_gk(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"],
                                 cu_seqlens=cu, decayed_read=True)
    for n, L in enumerate(lengths):
        a, b = int(cu[n]), int(cu[n + 1])
        sl = slice(a, b)
        os_, hs = oracle_mod.forward_gk(d["q"][:, sl], d["k"][:, sl], d["v"][:, sl],
                                        d["beta"][:, sl], d["g"][:, sl], d["h0"][n:n + 1],
                                        decayed_read=True)
        assert np.array_equal(o[:, sl], os_)
        assert np.array_equal(h[n], hs[0])
