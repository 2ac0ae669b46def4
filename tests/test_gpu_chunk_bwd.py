"""GPU parity of the chunked tensor-core backward (kda_chunk_bwd) against the fp64 autograd
oracle: every gradient (q, k, v, beta, the per-head decay, the initial state), both decay
placements, ragged lengths across chunks, both head dims, no decay, no L2 normalisation,
and the training shape (B=2, T=2048, H=16, d=128) on a sample of heads.

Bar (bf16 inputs; the oracle runs on the same bf16 values): max|diff| <= 2e-2 max|ref| per
gradient -- the forward's bar on its output, since the backward carries the same bf16 chunk
maps and bf16 state operands on the tensor cores (its chunk-local products are tf32 with
fp32 accumulation)."""
import numpy as np
import pytest

from kda_inputs import make_custom, round_to_bf16
from _util import max_rel, to_dev, to_np

pytestmark = pytest.mark.gpu

BAR = 2e-2
NAMES = ("dq", "dk", "dv", "dbeta", "ddecay", "dh0")


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


def _inputs(B, T, H, D, decay, seed, with_dhT=True):
    d = make_custom(B, T, H, D, D, dtype="bf16", decay=decay, h0="normal002", seed=seed)
    d["h0"] = (d["h0"] * 20).astype(np.float32)
    rng = np.random.default_rng(seed + 3000)
    do = round_to_bf16(rng.standard_normal((B, T, H, D)).astype(np.float32))
    dhT = rng.standard_normal((B, H, D, D)).astype(np.float32) if with_dhT else None
    return d, do, dhT


def _gpu(kda, dev, d, do, dhT, decayed, use_l2=True, use_decay=True):
    import torch
    dec = d["decay"] if use_decay else None
    got = kda.chunk_bwd(*(to_dev(d[n], dev, torch.bfloat16) for n in ("q", "k", "v")),
                        to_dev(d["beta"], dev, torch.float32),
                        None if dec is None else to_dev(dec, dev, torch.float32),
                        to_dev(d["h0"], dev, torch.float32), to_dev(do, dev, torch.bfloat16),
                        None if dhT is None else to_dev(dhT, dev, torch.float32),
                        use_qk_l2norm=use_l2, decayed_read=decayed)
    torch.cuda.synchronize()
    return {n: to_np(got[n]) for n in NAMES}


def _oracle(d, do, dhT, decayed, use_l2=True, use_decay=True, heads=None):
    from oracle import backward as ob
    sel = (lambda x: x) if heads is None else (lambda x: np.ascontiguousarray(x[:, :, heads]))
    selh = (lambda x: x) if heads is None else (lambda x: np.ascontiguousarray(x[:, heads]))
    D = d["q"].shape[-1]
    dec = d["decay"] if use_decay else np.zeros_like(d["beta"])
    g = np.repeat(sel(dec)[..., None], D, axis=-1).astype(np.float32)
    ref = ob.backward(sel(d["q"]), sel(d["k"]), sel(d["v"]), sel(d["beta"]), g, selh(d["h0"]), sel(do),
                      None if dhT is None else selh(dhT), use_l2=use_l2, decayed_read=decayed)
    ref["ddecay"] = ref["dg"].sum(-1) if use_decay else np.zeros_like(sel(d["beta"]))
    return ref


def _check(got, ref, tag, heads=None):
    for n in NAMES:
        g = got[n]
        if heads is not None:
            g = g[:, heads] if n == "dh0" else g[:, :, heads]
        err = max_rel(g, ref[n])
        assert err <= BAR, f"{tag} {n}: {err:.3e}"


@pytest.mark.parametrize("decayed", [False, True])
@pytest.mark.parametrize("decay", ["train", "long", "strong"])
def test_decay_regimes(kda, dev, decay, decayed):
    d, do, dhT = _inputs(2, 150, 2, 128, decay, seed=91)
    _check(_gpu(kda, dev, d, do, dhT, decayed), _oracle(d, do, dhT, decayed), f"{decay} decayed={decayed}")


@pytest.mark.parametrize("T", [1, 63, 64, 65, 200])
def test_lengths_d64(kda, dev, T):
    d, do, dhT = _inputs(1, T, 3, 64, "train", seed=92 + T)
    _check(_gpu(kda, dev, d, do, dhT, False), _oracle(d, do, dhT, False), f"T={T}")


def test_no_decay_no_l2_no_final_gradient(kda, dev):
    d, do, dhT = _inputs(1, 100, 2, 128, "train", seed=93, with_dhT=False)
    d["k"] = round_to_bf16((d["k"] * 128 ** -0.5).astype(np.float32))
    got = _gpu(kda, dev, d, do, None, False, use_l2=False, use_decay=False)
    _check(got, _oracle(d, do, None, False, use_l2=False, use_decay=False), "no decay, no l2")


def test_training_shape_head_sample(kda, dev):
    """B=2, T=2048, H=16, d=128 (the training-shape workload, as benched) on the GPU; the
    oracle on three heads of both batch entries over the full T."""
    d, do, dhT = _inputs(2, 2048, 16, 128, "train", seed=94)
    got = _gpu(kda, dev, d, do, dhT, False)
    heads = [0, 7, 15]
    _check(got, _oracle(d, do, dhT, False, heads=heads), "training shape", heads=heads)


def test_more_pairs_than_chains(kda, dev):
    """More (sequence, head) pairs than the kept-map forward runs chains at once (a quarter
    of the SMs): the forward walks them in rounds, its ring as deep as every round's chunks."""
    import torch
    pairs = torch.cuda.get_device_properties(dev).multi_processor_count // 4 + 10
    H = 8
    B = (pairs + H - 1) // H
    d, do, dhT = _inputs(B, 130, H, 64, "train", seed=95)
    heads = [0, 5]
    got = _gpu(kda, dev, d, do, dhT, False)
    _check(got, _oracle(d, do, dhT, False, heads=heads), f"B={B} H={H}", heads=heads)

