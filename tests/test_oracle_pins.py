"""Pins for the fp64 oracle: each test checks it against something other than itself.

The recurrence is the one printed on ejkernel ``kernel_delta_attention._interface``,
``kda()`` ("The core recurrence"); the decay-free single step is TileOPs "Linear
Attention Operators", DeltaNetRecurrentFwdOp.  Every check below is computed in
the test from mathematics that does not go through the oracle's code:

* brute force with explicit dk x dk transition matrices (tiny sizes);
* the decay-free decode identity of DeltaNetRecurrentFwdOp;
* exact retrieval when beta = 1, decay = 0 and |k| = 1;
* a closed form with one-hot keys that fixes where the decay is applied;
* beta = 0: pure exponential decay of the initial state;
* the oracle's chunked WY form equals its recurrent form for every chunk size;
* linearity, permutation, varlen-vs-separate, split-and-chain invariants.
"""
import numpy as np
import pytest

from kda_inputs import make_custom, round_to_bf16

RTOL_EXACT = 1e-12


def _l2(x):
    n = np.sqrt(np.sum(np.asarray(x, np.float64) ** 2, axis=-1, keepdims=True))
    return np.asarray(x, np.float64) / np.maximum(n, 1e-12)


def _rel(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


# ---------------------------------------------------------------------------
# P-1: brute force.  h_t = A_t h_{t-1} + beta_t k_t v_t^T with the explicit
# transition matrix A_t = exp(decay_t) I - beta_t k_t k_t^T, which is the
# printed recurrence rewritten; h_t is formed from scratch for every t as
# (A_t ... A_1) h_0 + sum_s (A_t ... A_{s+1}) beta_s k_s v_s^T.
# ---------------------------------------------------------------------------
def _bruteforce(q, k, v, beta, decay, h0, scale, use_l2):
    T, dk = k.shape
    dv = v.shape[1]
    kk = _l2(k) if use_l2 else k.astype(np.float64)
    qq = (_l2(q) if use_l2 else q.astype(np.float64)) * scale
    A = [np.exp(decay[t]) * np.eye(dk) - beta[t] * np.outer(kk[t], kk[t]) for t in range(T)]

    def prod(lo, hi):  # A_hi ... A_lo  (1-based, inclusive); identity if empty
        M = np.eye(dk)
        for t in range(lo, hi + 1):
            M = A[t - 1] @ M
        return M

    o = np.zeros((T, dv))
    h = None
    for t in range(1, T + 1):
        h = prod(1, t) @ h0
        for s in range(1, t + 1):
            h = h + prod(s + 1, t) @ (beta[s - 1] * np.outer(kk[s - 1], v[s - 1]))
        o[t - 1] = h.T @ qq[t - 1]
    return o, h


@pytest.mark.parametrize("seed", [0, 1, 2])
@pytest.mark.parametrize("use_l2", [True, False])
@pytest.mark.parametrize("dims", [(7, 3, 4), (8, 4, 2), (5, 1, 3)])
def test_bruteforce_tiny(oracle_mod, seed, use_l2, dims):
    T, dk, dv = dims
    rng = np.random.default_rng(100 + seed)
    q = rng.standard_normal((1, T, 1, dk)).astype(np.float32)
    k = rng.standard_normal((1, T, 1, dk)).astype(np.float32)
    v = rng.standard_normal((1, T, 1, dv)).astype(np.float32)
    beta = rng.uniform(0.05, 0.95, (1, T, 1)).astype(np.float32)
    decay = (-0.3 * np.abs(rng.standard_normal((1, T, 1)))).astype(np.float32)
    h0 = rng.standard_normal((1, 1, dk, dv))
    scale = 0.7
    if not use_l2:  # keep the unnormalised recurrence contractive
        k = (k / np.float32(2.0 * np.sqrt(dk))).astype(np.float32)
    o, hT = oracle_mod.forward(q, k, v, beta, decay, h0, scale=scale, use_l2=use_l2)
    ob, hb = _bruteforce(q[0, :, 0], k[0, :, 0], v[0, :, 0], beta[0, :, 0].astype(np.float64),
                         decay[0, :, 0].astype(np.float64), h0[0, 0], scale, use_l2)
    assert _rel(o[0, :, 0], ob) < RTOL_EXACT
    assert _rel(hT[0, 0], hb) < RTOL_EXACT


# ---------------------------------------------------------------------------
# P-2: decay = 0 equals DeltaNetRecurrentFwdOp's step
#   v_new = beta (v - S^T k),  o = S^T q + (q . k) v_new,  S_new = S + k v_new^T
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("seed", [0, 1])
def test_decode_identity_decay_free(oracle_mod, seed):
    rng = np.random.default_rng(200 + seed)
    B, H, dk, dv, T = 2, 3, 16, 8, 5
    q = rng.standard_normal((B, T, H, dk)).astype(np.float32)
    k = rng.standard_normal((B, T, H, dk)).astype(np.float32)
    v = rng.standard_normal((B, T, H, dv)).astype(np.float32)
    beta = rng.uniform(0, 1, (B, T, H)).astype(np.float32)
    S0 = 0.1 * rng.standard_normal((B, H, dk, dv))
    scale = dk ** -0.5
    o, hT = oracle_mod.forward(q, k, v, beta, None, S0, use_l2=True)
    S = S0.copy()
    for t in range(T):
        kk = _l2(k[:, t])
        qq = _l2(q[:, t]) * scale
        vnew = beta[:, t, :, None] * (v[:, t] - np.einsum("bhij,bhi->bhj", S, kk))
        ot = np.einsum("bhij,bhi->bhj", S, qq) + np.sum(qq * kk, -1)[..., None] * vnew
        S = S + kk[..., :, None] * vnew[..., None, :]
        assert _rel(o[:, t], ot) < RTOL_EXACT
    assert _rel(hT, S) < RTOL_EXACT


# ---------------------------------------------------------------------------
# P-3: exact retrieval.  beta = 1, decay = 0, unit keys: the step overwrites the
# memory's answer to k_t with v_t, so reading with q_t = k_t (scale 1) returns v_t.
# ---------------------------------------------------------------------------
def test_exact_retrieval(oracle_mod):
    rng = np.random.default_rng(3)
    B, T, H, dk, dv = 1, 40, 2, 32, 16
    k = rng.standard_normal((B, T, H, dk)).astype(np.float32)
    v = rng.standard_normal((B, T, H, dv)).astype(np.float32)
    beta = np.ones((B, T, H), np.float32)
    h0 = rng.standard_normal((B, H, dk, dv))
    o, _ = oracle_mod.forward(k, k, v, beta, None, h0, scale=1.0, use_l2=True)
    assert np.max(np.abs(o - v)) < 1e-12 * max(1.0, np.max(np.abs(v)))


# ---------------------------------------------------------------------------
# P-4: one-hot keys fix the decay placement.  With k_t = e_{i_t}:
#   row i_t of h becomes (alpha_t - beta_t) h[i_t] + beta_t v_t, other rows alpha_t h.
# (Decaying before the read would instead give alpha_t (1 - beta_t) h[i_t] + beta_t v_t.)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("seed", [0, 1])
def test_one_hot_keys_closed_form(oracle_mod, seed):
    rng = np.random.default_rng(400 + seed)
    dk, dv, T = 6, 3, 9
    idx = rng.integers(0, dk, size=T)
    k = np.zeros((1, T, 1, dk), np.float32)
    k[0, np.arange(T), 0, idx] = 1.0
    q = rng.standard_normal((1, T, 1, dk)).astype(np.float32)
    v = rng.standard_normal((1, T, 1, dv)).astype(np.float32)
    beta = rng.uniform(0.1, 0.9, (1, T, 1)).astype(np.float32)
    decay = (-rng.uniform(0.1, 1.0, (1, T, 1))).astype(np.float32)
    h0 = rng.standard_normal((1, 1, dk, dv))
    o, hT = oracle_mod.forward(q, k, v, beta, decay, h0, scale=1.0, use_l2=True)
    h = h0[0, 0].copy()
    qn = _l2(q[0, :, 0])
    for t in range(T):
        a = np.exp(np.float64(decay[0, t, 0]))
        b = np.float64(beta[0, t, 0])
        i = idx[t]
        row = (a - b) * h[i] + b * v[0, t, 0]
        h = a * h
        h[i] = row
        assert _rel(o[0, t, 0], h.T @ qn[t]) < RTOL_EXACT
    assert _rel(hT[0, 0], h) < RTOL_EXACT


# ---------------------------------------------------------------------------
# P-5: beta = 0 leaves only the decay: h_T = exp(sum decay) h_0 and
#      o_t = exp(sum_{r<=t} decay_r) h_0^T q_t.
# ---------------------------------------------------------------------------
def test_beta_zero_pure_decay(oracle_mod):
    rng = np.random.default_rng(5)
    B, T, H, dk, dv = 2, 30, 2, 8, 8
    q = rng.standard_normal((B, T, H, dk)).astype(np.float32)
    k = rng.standard_normal((B, T, H, dk)).astype(np.float32)
    v = rng.standard_normal((B, T, H, dv)).astype(np.float32)
    beta = np.zeros((B, T, H), np.float32)
    decay = (-0.2 * np.abs(rng.standard_normal((B, T, H)))).astype(np.float32)
    h0 = rng.standard_normal((B, H, dk, dv))
    scale = 0.5
    o, hT = oracle_mod.forward(q, k, v, beta, decay, h0, scale=scale, use_l2=True)
    G = np.cumsum(decay.astype(np.float64), axis=1)            # [B,T,H]
    qn = _l2(q) * scale
    exp_o = np.exp(G)[..., None] * np.einsum("bhij,bthi->bthj", h0, qn)
    exp_h = np.exp(G[:, -1])[..., None, None] * h0
    assert _rel(o, exp_o) < RTOL_EXACT
    assert _rel(hT, exp_h) < RTOL_EXACT


# ---------------------------------------------------------------------------
# P-6: the chunked WY form equals the recurrent scan for every chunk size,
# including chunk sizes that do not divide T and chunk > T.
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("chunk", [1, 2, 3, 4, 8, 16, 37, 64, 100])
def test_chunked_equals_recurrent(oracle_mod, chunk):
    d = make_custom(2, 37, 2, 8, 5, dtype="f32", decay="train", h0="normal002", seed=11)
    d["decay"] = (d["decay"] * 6).astype(np.float32)   # decay ~ -0.3|N|: exercises the exponents
    d["h0"] = (d["h0"] * 50).astype(np.float32)
    o1, h1 = oracle_mod.forward(d["q"], d["k"], d["v"], d["beta"], d["decay"], d["h0"])
    o2, h2 = oracle_mod.forward(d["q"], d["k"], d["v"], d["beta"], d["decay"], d["h0"], chunk=chunk)
    assert _rel(o2, o1) < 1e-10
    assert _rel(h2, h1) < 1e-10


def test_chunked_equals_recurrent_tiny_config(oracle_mod):
    from kda_inputs import WORKLOADS, make_prefill
    wl = WORKLOADS[1]
    d = make_prefill(wl, seed=0)
    o1, h1 = oracle_mod.forward(d["q"], d["k"], d["v"], d["beta"], d["decay"], d["h0"])
    o2, h2 = oracle_mod.forward(d["q"], d["k"], d["v"], d["beta"], d["decay"], d["h0"],
                                chunk=wl.chunk)
    assert _rel(o2, o1) < 1e-10 and _rel(h2, h1) < 1e-10


# ---------------------------------------------------------------------------
# P-7: invariants.
# ---------------------------------------------------------------------------
def test_joint_linearity_in_v_and_h0(oracle_mod):
    """o and h_T are jointly linear in (v, h0) for fixed q, k, beta, decay."""
    d1 = make_custom(1, 20, 2, 8, 6, dtype="bf16", decay="train", h0="normal002", seed=1)
    d2 = make_custom(1, 20, 2, 8, 6, dtype="bf16", decay="train", h0="normal002", seed=2)
    a, b = 0.5, -2.0
    v = a * d1["v"].astype(np.float64) + b * d2["v"].astype(np.float64)
    assert np.array_equal(v.astype(np.float32).astype(np.float64), v)  # exact in f32
    h0 = a * d1["h0"].astype(np.float64) + b * d2["h0"].astype(np.float64)
    args = (d1["q"], d1["k"])
    oa, ha = oracle_mod.forward(*args, d1["v"], d1["beta"], d1["decay"], d1["h0"])
    ob, hb = oracle_mod.forward(*args, d2["v"], d1["beta"], d1["decay"], d2["h0"])
    oc, hc = oracle_mod.forward(*args, v.astype(np.float32), d1["beta"], d1["decay"], h0)
    assert _rel(oc, a * oa + b * ob) < 1e-12
    assert _rel(hc, a * ha + b * hb) < 1e-12


def test_output_linear_in_scale(oracle_mod):
    d = make_custom(1, 25, 2, 8, 8, dtype="f32", decay="train", h0="normal002", seed=4)
    o1, h1 = oracle_mod.forward(d["q"], d["k"], d["v"], d["beta"], d["decay"], d["h0"], scale=0.25)
    o2, h2 = oracle_mod.forward(d["q"], d["k"], d["v"], d["beta"], d["decay"], d["h0"], scale=0.75)
    assert _rel(o2, 3.0 * o1) < 1e-13
    assert _rel(h2, h1) < 1e-15


def test_default_scale_is_inverse_sqrt_dk(oracle_mod):
    d = make_custom(1, 10, 1, 16, 4, dtype="f32", decay="small", seed=6)
    o1, _ = oracle_mod.forward(d["q"], d["k"], d["v"], d["beta"], d["decay"], None)
    o2, _ = oracle_mod.forward(d["q"], d["k"], d["v"], d["beta"], d["decay"], None, scale=0.25)
    assert _rel(o1, o2) < 1e-15


def test_head_and_batch_permutation(oracle_mod):
    d = make_custom(2, 16, 3, 8, 4, dtype="f32", decay="train", h0="normal002", seed=7)
    o, h = oracle_mod.forward(d["q"], d["k"], d["v"], d["beta"], d["decay"], d["h0"])
    pb, ph = [1, 0], [2, 0, 1]
    P = lambda x: x[pb][:, :, ph]  # noqa: E731  permute [B,T,H,...]
    Ps = lambda x: x[pb][:, ph]    # noqa: E731  permute [B,H,...]
    o2, h2 = oracle_mod.forward(P(d["q"]), P(d["k"]), P(d["v"]), P(d["beta"]), P(d["decay"]),
                                Ps(d["h0"]))
    assert np.array_equal(o2, P(o)) and np.array_equal(h2, Ps(h))


def test_head_subset_matches_full(oracle_mod):
    d = make_custom(2, 12, 3, 8, 4, dtype="f32", decay="train", h0="normal002", seed=8)
    o, h = oracle_mod.forward(d["q"], d["k"], d["v"], d["beta"], d["decay"], d["h0"])
    o2, h2 = oracle_mod.forward(d["q"], d["k"], d["v"], d["beta"], d["decay"], d["h0"],
                                heads=[4, 1])
    assert np.array_equal(o2[1, :, 1], o[1, :, 1]) and np.array_equal(o2[0, :, 1], o[0, :, 1])
    assert np.array_equal(h2[1, 1], h[1, 1]) and np.isnan(o2[0, :, 0]).all()


def test_varlen_equals_separate_calls(oracle_mod):
    lengths = [5, 17, 1, 33]
    H, dk, dv = 2, 8, 6
    parts = [make_custom(1, L, H, dk, dv, dtype="f32", decay="train", h0="normal002", seed=20 + i)
             for i, L in enumerate(lengths)]
    cat = lambda key: np.concatenate([p[key] for p in parts], axis=1)  # noqa: E731
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    h0 = np.concatenate([p["h0"] for p in parts], axis=0)
    for chunk in (None, 4):
        o, h = oracle_mod.varlen(cat("q"), cat("k"), cat("v"), cat("beta"), cu, cat("decay"), h0,
                                 chunk=chunk)
        for i, p in enumerate(parts):
            oi, hi = oracle_mod.forward(p["q"], p["k"], p["v"], p["beta"], p["decay"], p["h0"])
            assert _rel(o[:, cu[i]:cu[i + 1]], oi) < 1e-10
            assert _rel(h[i], hi[0]) < 1e-10


def test_decode_steps_equal_prefill(oracle_mod):
    d = make_custom(2, 9, 2, 8, 8, dtype="bf16", decay="small", h0="normal002", seed=9)
    o, h = oracle_mod.forward(d["q"], d["k"], d["v"], d["beta"], d["decay"], d["h0"])
    steps = [{key: d[key][:, t:t + 1] for key in ("q", "k", "v", "beta", "decay")}
             for t in range(9)]
    outs, hd = oracle_mod.decode_steps(steps, d["h0"])
    assert _rel(np.concatenate(outs, axis=1), o) < 1e-13
    assert _rel(hd, h) < 1e-13


@pytest.mark.parametrize("split", [1, 7, 16, 25])
def test_split_and_chain_state(oracle_mod, split):
    d = make_custom(1, 32, 2, 8, 8, dtype="f32", decay="train", h0="normal002", seed=10)
    o, h = oracle_mod.forward(d["q"], d["k"], d["v"], d["beta"], d["decay"], d["h0"])
    a = {key: d[key][:, :split] for key in ("q", "k", "v", "beta", "decay")}
    b = {key: d[key][:, split:] for key in ("q", "k", "v", "beta", "decay")}
    o1, h1 = oracle_mod.forward(a["q"], a["k"], a["v"], a["beta"], a["decay"], d["h0"], chunk=16)
    o2, h2 = oracle_mod.forward(b["q"], b["k"], b["v"], b["beta"], b["decay"], h1)
    assert _rel(np.concatenate([o1, o2], axis=1), o) < 1e-11
    assert _rel(h2, h) < 1e-11


def test_zero_key_row_is_harmless(oracle_mod):
    """A zero key (norm below the 1e-12 floor) writes nothing; only the decay acts."""
    d = make_custom(1, 3, 1, 4, 4, dtype="f32", decay="train", h0="normal002", seed=12)
    d["k"][0, 1] = 0.0
    o, h = oracle_mod.forward(d["q"], d["k"], d["v"], d["beta"], d["decay"], d["h0"])
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(h))
    o01, h01 = oracle_mod.forward(d["q"][:, :1], d["k"][:, :1], d["v"][:, :1], d["beta"][:, :1],
                                  d["decay"][:, :1], d["h0"])
    hmid = np.exp(np.float64(d["decay"][0, 1, 0])) * h01
    o2, _ = oracle_mod.forward(d["q"][:, 1:2], d["k"][:, 1:2], d["v"][:, 1:2], d["beta"][:, 1:2],
                               np.zeros((1, 1, 1), np.float32), hmid)
    assert _rel(o[:, 1], o2[:, 0]) < 1e-12


def test_empty_sequence(oracle_mod):
    d = make_custom(1, 0, 2, 4, 4, dtype="f32", decay="train", h0="normal002", seed=13)
    o, h = oracle_mod.forward(d["q"], d["k"], d["v"], d["beta"], d["decay"], d["h0"])
    assert o.shape == (1, 0, 2, 4)
    assert np.array_equal(h, d["h0"].astype(np.float64))


def test_bf16_rounding_helper():
    x = np.array([1.0, 1.00390625, 1.005859375, -3.14159, 1e-3], np.float32)
    r = round_to_bf16(x)
    assert r[0] == 1.0
    assert r[1] == 1.0                  # exact tie 1 + 2^-8 rounds to even (1.0)
    assert r[2] == np.float32(1.0078125)  # 1 + 1.5*2^-8 rounds up
    assert np.all(np.abs(r - x) <= np.abs(x) * 2.0 ** -8)
    assert np.all((r.view(np.uint32) & 0xFFFF) == 0)
