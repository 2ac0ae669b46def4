"""GPU parity of the per-channel backward (kda_gk_recurrent_bwd) against the fp64 autograd
oracle: every gradient (q, k, v, beta, g, initial state), both decay placements, ragged
lengths across the 32-token checkpoints, head dims, both value-slab widths, no decay, no L2
normalisation.  Bar: max|diff| / max|ref| per gradient <= 1e-4 (fp32 inputs), <= 1e-3 (bf16
inputs, the oracle on the same bf16 values; the kernels' arithmetic is fp32 in both)."""
import numpy as np
import pytest

from kda_inputs import make_gk, round_to_bf16
from _util import max_rel, to_dev, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kda():
    import delta_rule_linear_gb300 as m
    from delta_rule_linear_gb300 import build as b
    b.build()
    m.load()
    return m


@pytest.fixture(scope="module")
def dev():
    import torch
    return torch.device("cuda:0")


def _case(kda, dev, B, T, H, dk, dv, dtype, gate, decayed, seed, use_l2=True, scale=None, with_g=True,
          with_dhT=True):
    import torch
    from oracle import backward as ob
    d = make_gk(B, T, H, dk, dv, dtype=dtype, gate_scale=gate, h0="normal002", seed=seed)
    d["h0"] = (d["h0"] * 20).astype(np.float32)
    if not use_l2:
        d["k"] = (d["k"] * (dk ** -0.5)).astype(np.float32)
        if dtype == "bf16":
            d["k"] = round_to_bf16(d["k"])
    rng = np.random.default_rng(seed + 1000)
    do = rng.standard_normal((B, T, H, dv)).astype(np.float32)
    if dtype == "bf16":
        do = round_to_bf16(do)
    dhT = rng.standard_normal((B, H, dk, dv)).astype(np.float32) if with_dhT else None
    g = d["g"] if with_g else None
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    got = kda.gk_recurrent_bwd(*(to_dev(d[n], dev, tdt) for n in ("q", "k", "v")),
                               to_dev(d["beta"], dev, torch.float32),
                               None if g is None else to_dev(g, dev, torch.float32),
                               to_dev(d["h0"], dev, torch.float32), to_dev(do, dev, tdt),
                               None if dhT is None else to_dev(dhT, dev, torch.float32),
                               scale=scale, use_qk_l2norm=use_l2, decayed_read=decayed)
    torch.cuda.synchronize()
    ref = ob.backward(d["q"], d["k"], d["v"], d["beta"], g if g is not None else np.zeros_like(d["q"]),
                      d["h0"], do, dhT, scale=scale, use_l2=use_l2, decayed_read=decayed)
    tol = 1e-4 if dtype == "f32" else 1e-3
    for name in ("dq", "dk", "dv", "dbeta", "dg", "dh0"):
        want = ref[name] if (name != "dg" or g is not None) else np.zeros_like(ref["dg"])
        err = max_rel(to_np(got[name]), want)
        assert err <= tol, f"{name}: {err:.3e}"


@pytest.mark.parametrize("decayed", [False, True])
@pytest.mark.parametrize("gate", [0.05, 0.5, 2.0])
def test_gate_regimes(kda, dev, gate, decayed):
    _case(kda, dev, 2, 70, 2, 64, 64, "f32", gate, decayed, seed=71)


@pytest.mark.parametrize("dims", [(32, 32), (64, 128), (128, 64), (128, 128)])
def test_head_dims(kda, dev, dims):
    _case(kda, dev, 1, 45, 2, dims[0], dims[1], "f32", 0.3, True, seed=72)


def test_bf16_inputs(kda, dev):
    _case(kda, dev, 2, 100, 2, 128, 128, "bf16", 0.3, True, seed=73)


def test_no_decay_no_l2_no_final_gradient(kda, dev):
    _case(kda, dev, 1, 33, 2, 64, 64, "f32", 0.3, False, seed=74, use_l2=False, scale=0.4,
          with_g=False, with_dhT=False)


def test_lengths(kda, dev):
    for T in (1, 31, 32, 33, 64):
        _case(kda, dev, 1, T, 1, 64, 64, "f32", 0.5, True, seed=75 + T)


@pytest.mark.parametrize("dims,H", [((64, 64), 152), ((128, 128), 80)])
def test_wide_slabs(kda, dev, dims, H):
    # enough (sequence, head) pairs that each CTA takes 64 value columns instead of 32
    _case(kda, dev, 1, 37, H, dims[0], dims[1], "f32", 0.3, True, seed=76)


# ------------------------------------------------------------------ one decay per head
def _case_scalar(kda, dev, B, T, H, dk, dv, dtype, decay_kind, decayed, seed, use_decay=True):
    """kda_recurrent_bwd against the fp64 oracle with every channel's decay equal: the
    decay's gradient is the channel sum of the per-channel dg (chain rule)."""
    import torch
    from kda_inputs import make_custom
    from oracle import backward as ob
    d = make_custom(B, T, H, dk, dv, dtype=dtype, decay=decay_kind, h0="normal002", seed=seed)
    d["h0"] = (d["h0"] * 20).astype(np.float32)
    rng = np.random.default_rng(seed + 2000)
    do = rng.standard_normal((B, T, H, dv)).astype(np.float32)
    if dtype == "bf16":
        do = round_to_bf16(do)
    dhT = rng.standard_normal((B, H, dk, dv)).astype(np.float32)
    dec = d["decay"] if use_decay else None
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    got = kda.recurrent_bwd(*(to_dev(d[n], dev, tdt) for n in ("q", "k", "v")),
                            to_dev(d["beta"], dev, torch.float32),
                            None if dec is None else to_dev(dec, dev, torch.float32),
                            to_dev(d["h0"], dev, torch.float32), to_dev(do, dev, tdt),
                            to_dev(dhT, dev, torch.float32), decayed_read=decayed)
    torch.cuda.synchronize()
    g = np.repeat((dec if dec is not None else np.zeros_like(d["beta"]))[..., None], dk, axis=-1)
    ref = ob.backward(d["q"], d["k"], d["v"], d["beta"], g.astype(np.float32), d["h0"], do, dhT,
                      use_l2=True, decayed_read=decayed)
    ref["ddecay"] = ref["dg"].sum(-1) if dec is not None else np.zeros_like(d["beta"])
    tol = 1e-4 if dtype == "f32" else 1e-3
    for name in ("dq", "dk", "dv", "dbeta", "ddecay", "dh0"):
        err = max_rel(to_np(got[name]), ref[name])
        assert err <= tol, f"{name}: {err:.3e}"


@pytest.mark.parametrize("decayed", [False, True])
@pytest.mark.parametrize("decay_kind", ["train", "long", "strong"])
def test_scalar_decay(kda, dev, decay_kind, decayed):
    _case_scalar(kda, dev, 2, 70, 2, 64, 64, "f32", decay_kind, decayed, seed=81)


def test_scalar_decay_bf16_and_shapes(kda, dev):
    _case_scalar(kda, dev, 1, 100, 2, 128, 128, "bf16", "train", True, seed=82)
    _case_scalar(kda, dev, 1, 45, 3, 32, 128, "f32", "train", False, seed=83)
    _case_scalar(kda, dev, 1, 33, 2, 64, 64, "f32", "train", False, seed=84, use_decay=False)
    _case_scalar(kda, dev, 1, 37, 160, 64, 64, "f32", "train", True, seed=85)   # 64-column slabs
