"""GPU parity of the per-channel chunked backward (kda_gk_chunk_bwd) against the fp64 autograd
oracle: every gradient (q, k, v, beta, the per-channel decay g, the initial state) for gate
strengths from weak to strong, both decay placements, ragged lengths across chunks, both
head dims, no decay, no L2 normalisation, and the training shape (B=2, T=2048, H=16, d=128)
on a sample of heads.

Bar (bf16 inputs; the oracle runs on the same bf16 values): max|diff| <= 2e-2 max|ref| per
gradient -- the forward's bar on its output: the chunk maps, the kept states and state
gradients and the recomputed in-chunk states are bf16, every sum fp32."""
import numpy as np
import pytest

from kda_inputs import make_gk, round_to_bf16
from _util import max_rel, to_dev, to_np

pytestmark = pytest.mark.gpu

BAR = 2e-2
NAMES = ("dq", "dk", "dv", "dbeta", "dg", "dh0")


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


def _inputs(B, T, H, D, gate_scale, seed, with_dhT=True):
    d = make_gk(B, T, H, D, D, dtype="bf16", gate_scale=gate_scale, h0="normal002", seed=seed)
    d["h0"] = (d["h0"] * 20).astype(np.float32)
    rng = np.random.default_rng(seed + 5000)
    do = round_to_bf16(rng.standard_normal((B, T, H, D)).astype(np.float32))
    dhT = rng.standard_normal((B, H, D, D)).astype(np.float32) if with_dhT else None
    return d, do, dhT


def _gpu(kda, dev, d, do, dhT, decayed, use_l2=True, use_g=True):
    import torch
    got = kda.gk_chunk_bwd(*(to_dev(d[n], dev, torch.bfloat16) for n in ("q", "k", "v")),
                           to_dev(d["beta"], dev, torch.float32),
                           to_dev(d["g"], dev, torch.float32) if use_g else None,
                           to_dev(d["h0"], dev, torch.float32), to_dev(do, dev, torch.bfloat16),
                           None if dhT is None else to_dev(dhT, dev, torch.float32),
                           use_qk_l2norm=use_l2, decayed_read=decayed)
    torch.cuda.synchronize()
    return {n: to_np(got[n]) for n in NAMES}


def _oracle(d, do, dhT, decayed, use_l2=True, use_g=True, heads=None):
    from oracle import backward as ob
    sel = (lambda x: x) if heads is None else (lambda x: np.ascontiguousarray(x[:, :, heads]))
    selh = (lambda x: x) if heads is None else (lambda x: np.ascontiguousarray(x[:, heads]))
    g = sel(d["g"]) if use_g else np.zeros_like(sel(d["g"]))
    ref = ob.backward(sel(d["q"]), sel(d["k"]), sel(d["v"]), sel(d["beta"]), g, selh(d["h0"]), sel(do),
                      None if dhT is None else selh(dhT), use_l2=use_l2, decayed_read=decayed)
    if not use_g:
        ref["dg"] = np.zeros_like(ref["dg"])   # no decay: the entry point zero-fills dg
    return ref


def _check(got, ref, tag, heads=None):
    for n in NAMES:
        g = got[n]
        if heads is not None:
            g = g[:, heads] if n == "dh0" else g[:, :, heads]
        err = max_rel(g, ref[n])
        assert err <= BAR, f"{tag} {n}: {err:.3e}"


@pytest.mark.parametrize("decayed", [False, True])
@pytest.mark.parametrize("gate_scale", [0.01, 0.3, 2.0])
def test_gate_strengths(kda, dev, gate_scale, decayed):
    d, do, dhT = _inputs(2, 150, 2, 128, gate_scale, seed=191)
    _check(_gpu(kda, dev, d, do, dhT, decayed), _oracle(d, do, dhT, decayed),
           f"gate {gate_scale} decayed={decayed}")


@pytest.mark.parametrize("T", [1, 63, 64, 65, 200])
def test_lengths_d64(kda, dev, T):
    d, do, dhT = _inputs(1, T, 3, 64, 0.1, seed=192 + T)
    _check(_gpu(kda, dev, d, do, dhT, True), _oracle(d, do, dhT, True), f"T={T}")


def test_no_gate_no_l2_no_final_gradient(kda, dev):
    d, do, _ = _inputs(1, 100, 2, 128, 0.1, seed=193, with_dhT=False)
    d["k"] = round_to_bf16((d["k"] * 128 ** -0.5).astype(np.float32))
    got = _gpu(kda, dev, d, do, None, False, use_l2=False, use_g=False)
    _check(got, _oracle(d, do, None, False, use_l2=False, use_g=False), "no gate, no l2")


def test_matches_recurrent_backward(kda, dev):
    """The chunk-parallel walk against the sequential per-channel backward on the GPU, on a
    size the oracle would take long over: both are fp32 sums over the same recurrence."""
    import torch
    d, do, dhT = _inputs(2, 700, 8, 128, 0.05, seed=194)
    got = _gpu(kda, dev, d, do, dhT, True)
    t = {n: to_dev(d[n], dev, torch.bfloat16) for n in ("q", "k", "v")}
    ref = kda.gk_recurrent_bwd(t["q"], t["k"], t["v"], to_dev(d["beta"], dev, torch.float32),
                               to_dev(d["g"], dev, torch.float32), to_dev(d["h0"], dev, torch.float32),
                               to_dev(do, dev, torch.bfloat16), to_dev(dhT, dev, torch.float32),
                               decayed_read=True)
    torch.cuda.synchronize()
    for n in NAMES:
        err = max_rel(got[n], to_np(ref[n]))
        assert err <= BAR, f"vs recurrent {n}: {err:.3e}"


def test_training_shape_head_sample(kda, dev):
    """B=2, T=2048, H=16, d=128 (the training-shape workload, as benched) on the GPU; the
    oracle on three heads of both batch entries over the full T."""
    d, do, dhT = _inputs(2, 2048, 16, 128, 0.01, seed=195)
    got = _gpu(kda, dev, d, do, dhT, True)
    heads = [0, 7, 15]
    _check(got, _oracle(d, do, dhT, True, heads=heads), "training shape", heads=heads)


def test_more_pairs_than_chains(kda, dev):
    """More (sequence, head) pairs than the kept-map forward runs chains at once (a quarter
    of the SMs): the forward walks them in rounds, its ring as deep as every round's chunks."""
    import torch
    pairs = torch.cuda.get_device_properties(dev).multi_processor_count // 4 + 10
    H = 8
    B = (pairs + H - 1) // H
    d, do, dhT = _inputs(B, 130, H, 64, 0.3, seed=196)
    heads = [0, 5]
    got = _gpu(kda, dev, d, do, dhT, True)
    _check(got, _oracle(d, do, dhT, True, heads=heads), f"B={B} H={H}", heads=heads)


def test_no_initial_state_no_final_gradient(kda, dev):
    """initial_state and dfinal_state both absent (zeros): dh0 is still the gradient with
    respect to the zero initial state."""
    import torch
    d, do, _ = _inputs(2, 90, 2, 128, 0.3, seed=197, with_dhT=False)
    got = kda.gk_chunk_bwd(*(to_dev(d[n], dev, torch.bfloat16) for n in ("q", "k", "v")),
                           to_dev(d["beta"], dev, torch.float32), to_dev(d["g"], dev, torch.float32),
                           None, to_dev(do, dev, torch.bfloat16), None, decayed_read=False)
    torch.cuda.synchronize()
    got = {n: to_np(got[n]) for n in NAMES}
    d0 = dict(d, h0=np.zeros_like(d["h0"]))
    _check(got, _oracle(d0, do, None, False), "no h0, no dhT")

