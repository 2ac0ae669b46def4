"""Pins for the fp64 backward oracle: its forward equals the C oracle's per-channel scan, and
its gradients equal central finite differences of that forward (tiny sizes, every input)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")


def _inputs(seed, B=1, T=5, H=2, dk=3, dv=4):
    rng = np.random.default_rng(seed)
    return dict(q=rng.standard_normal((B, T, H, dk)), k=rng.standard_normal((B, T, H, dk)),
                v=rng.standard_normal((B, T, H, dv)), beta=rng.uniform(0.1, 0.9, (B, T, H)),
                g=-rng.uniform(0, 1.5, (B, T, H, dk)), h0=rng.standard_normal((B, H, dk, dv)))


@pytest.mark.parametrize("decayed", [False, True])
def test_forward_matches_c_oracle(oracle_mod, decayed):
    from oracle import backward as ob
    d = _inputs(1, B=2, T=9, H=2, dk=4, dv=5)
    d32 = {n: np.asarray(x, np.float32) for n, x in d.items()}
    ro, rh = oracle_mod.forward_gk(d32["q"], d32["k"], d32["v"], d32["beta"], d32["g"], d32["h0"],
                                   decayed_read=decayed)
    t = {n: torch.tensor(np.asarray(x, np.float64)) for n, x in d32.items()}
    o, h = ob.forward_torch(t["q"], t["k"], t["v"], t["beta"], t["g"], t["h0"], decayed_read=decayed)
    assert np.max(np.abs(o.numpy() - ro)) < 1e-12 and np.max(np.abs(h.numpy() - rh)) < 1e-12


@pytest.mark.parametrize("use_l2", [True, False])
@pytest.mark.parametrize("decayed", [False, True])
def test_gradients_match_finite_differences(decayed, use_l2):
    from oracle import backward as ob
    d = _inputs(2)
    rng = np.random.default_rng(3)
    do = rng.standard_normal((1, 5, 2, 4))
    dhT = rng.standard_normal((1, 2, 3, 4))
    kw = dict(scale=0.7, use_l2=use_l2, decayed_read=decayed)
    grads = ob.backward(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"], do, dhT, **kw)

    def loss(dd):
        t = {n: torch.tensor(x) for n, x in dd.items()}
        o, h = ob.forward_torch(t["q"], t["k"], t["v"], t["beta"], t["g"], t["h0"], **kw)
        return float((o.numpy() * do).sum() + (h.numpy() * dhT).sum())

    eps = 1e-6
    for name in ("q", "k", "v", "beta", "g", "h0"):
        fd = np.zeros_like(d[name])
        for idx in np.ndindex(d[name].shape):
            p = {n: x.copy() for n, x in d.items()}
            m = {n: x.copy() for n, x in d.items()}
            p[name][idx] += eps
            m[name][idx] -= eps
            fd[idx] = (loss(p) - loss(m)) / (2 * eps)
        err = np.max(np.abs(fd - grads["d" + name])) / max(np.max(np.abs(fd)), 1e-12)
        assert err < 1e-7, (name, err)


@pytest.mark.parametrize("decayed", [False, True])
def test_scalar_decay_gradient_is_the_channel_sum(oracle_mod, decayed):
    """One decay per head (the path's own recurrence, run by the C oracle's scalar scan): the
    gradient of that decay is the sum over key channels of the per-channel dg, checked against
    central differences of the C oracle's forward.  The C oracle rounds its inputs to float32,
    so the step is 1e-3 and the bar 1e-3 (rounding ~6e-5, truncation ~1e-6 relative)."""
    from oracle import backward as ob
    rng = np.random.default_rng(7)
    B, T, H, dk, dv = 1, 6, 2, 4, 3
    q, k = rng.standard_normal((B, T, H, dk)), rng.standard_normal((B, T, H, dk))
    v = rng.standard_normal((B, T, H, dv))
    beta = rng.uniform(0.1, 0.9, (B, T, H))
    dec = -rng.uniform(0.05, 1.0, (B, T, H))
    h0 = rng.standard_normal((B, H, dk, dv))
    do = rng.standard_normal((B, T, H, dv))
    dhT = rng.standard_normal((B, H, dk, dv))
    g = np.repeat(dec[..., None], dk, axis=-1)
    grads = ob.backward(q, k, v, beta, g, h0, do, dhT, use_l2=True, decayed_read=decayed)
    dd = grads["dg"].sum(-1)

    def loss(dc):
        if decayed:   # the decayed read with one decay per head: the per-channel scan, channels equal
            o, h = oracle_mod.forward_gk(q, k, v, beta, np.repeat(dc[..., None], dk, axis=-1), h0,
                                         decayed_read=True)
        else:
            o, h = oracle_mod.forward(q, k, v, beta, dc, h0)
        return float((o * do).sum() + (h * dhT).sum())

    eps = 1e-3   # the C oracle takes float32 inputs
    fd = np.zeros_like(dec)
    for idx in np.ndindex(dec.shape):
        p, m = dec.copy(), dec.copy()
        p[idx] += eps
        m[idx] -= eps
        fd[idx] = (loss(p) - loss(m)) / (2 * eps)
    err = np.max(np.abs(fd - dd)) / np.max(np.abs(fd))
    assert err < 1e-3, err


@pytest.mark.parametrize("decayed", [False, True])
def test_split_sequence_gradients_chain(decayed):
    """A sequence's gradients equal those of its two parts chained through the state at the
    split: the second part starts from that state and hands back its gradient, which the
    first part takes as its final-state gradient (the structure a chunked backward uses)."""
    from oracle import backward as ob
    d = _inputs(7, B=2, T=12, H=2, dk=3, dv=4)
    rng = np.random.default_rng(8)
    do = rng.standard_normal((2, 12, 2, 4))
    dhT = rng.standard_normal((2, 2, 3, 4))
    full = ob.backward(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"], do, dhT, decayed_read=decayed)
    cut = 7
    a = {n: (x[:, :cut] if n != "h0" else x) for n, x in d.items()}
    b = {n: x[:, cut:] for n, x in d.items() if n != "h0"}
    t = {n: torch.tensor(np.asarray(x, np.float64)) for n, x in a.items()}
    _, h_mid = ob.forward_torch(t["q"], t["k"], t["v"], t["beta"], t["g"], t["h0"], decayed_read=decayed)
    second = ob.backward(b["q"], b["k"], b["v"], b["beta"], b["g"], h_mid.numpy(), do[:, cut:], dhT,
                         decayed_read=decayed)
    first = ob.backward(a["q"], a["k"], a["v"], a["beta"], a["g"], a["h0"], do[:, :cut], second["dh0"],
                        decayed_read=decayed)
    for n in ("dq", "dk", "dv", "dbeta", "dg"):
        np.testing.assert_allclose(np.concatenate([first[n], second[n]], axis=1), full[n], rtol=0, atol=1e-10)
    np.testing.assert_allclose(first["dh0"], full["dh0"], rtol=0, atol=1e-10)
