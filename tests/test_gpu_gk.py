"""GPU parity of the per-key-channel decay paths (TileOPs KDAFwdOp: g [B,T,H,K]) through
the C ABI, against the fp64 oracle on the same seeded inputs.  Same bars as the scalar
paths: fp32 max|diff|/max|ref| <= 1e-4; bf16 max|do| <= 2e-2 max|o| and final_state
Frobenius-relative <= 1e-2.  Gate regimes: g = -scale * U[0,1) with the scales of the
kda-neuron-kernels README's warning table (0.01, 0.3, 2.0) and a stronger 6.0.
"""
import numpy as np
import pytest

from kda_inputs import make_gk, make_gk_decode_step
from _util import assert_parity, to_dev, to_np

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


def _dev_inputs(d, dev, dtype):
    import torch
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    t = {n: to_dev(d[n], dev, tdt) for n in ("q", "k", "v")}
    for n in ("beta", "g", "h0"):
        t[n] = to_dev(d.get(n), dev, torch.float32)
    if "cu_seqlens" in d:
        t["cu_seqlens"] = to_dev(d["cu_seqlens"], dev, torch.int32)
    return t


def _run(kda, d, dev, dtype, decayed, use_g=True, **kw):
    import torch
    t = _dev_inputs(d, dev, dtype)
    o, h = kda.gk_recurrent_fwd(t["q"], t["k"], t["v"], t["beta"], t["g"] if use_g else None,
                                t["h0"], cu_seqlens=t.get("cu_seqlens"), decayed_read=decayed,
                                **kw)
    torch.cuda.synchronize()
    return to_np(o), to_np(h)


@pytest.mark.parametrize("decayed", [False, True])
@pytest.mark.parametrize("gate", [0.01, 0.3, 2.0, 6.0])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_recurrent_gate_regimes(kda, oracle_mod, dev, dtype, gate, decayed):
    d = make_gk(2, 203, 3, 128, 128, dtype=dtype, gate_scale=gate, h0="normal002", seed=11)
    o, h = _run(kda, d, dev, dtype, decayed)
    ro, rh = oracle_mod.forward_gk(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"],
                                   decayed_read=decayed)
    assert_parity(dtype, o, ro, h, rh, tag=f"gk gate={gate} decayed={decayed}")


@pytest.mark.parametrize("dims", [(32, 32), (64, 64), (32, 128), (128, 64), (64, 32)])
@pytest.mark.parametrize("decayed", [False, True])
def test_recurrent_head_dims(kda, oracle_mod, dev, dims, decayed):
    dk, dv = dims
    d = make_gk(1, 77, 4, dk, dv, dtype="f32", gate_scale=0.3, h0="normal002", seed=12)
    o, h = _run(kda, d, dev, "f32", decayed)
    ro, rh = oracle_mod.forward_gk(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"],
                                   decayed_read=decayed)
    assert_parity("f32", o, ro, h, rh, tag=f"gk dims={dims}")


def test_recurrent_no_gate_no_l2_custom_scale(kda, oracle_mod, dev):
    d = make_gk(2, 50, 2, 64, 64, dtype="f32", gate_scale=0.3, seed=13)
    d["k"] = (d["k"] * 0.125).astype(np.float32)      # keep beta |k|^2 below 2 without l2
    o, h = _run(kda, d, dev, "f32", True, use_g=False, use_qk_l2norm=False, scale=0.3)
    ro, rh = oracle_mod.forward_gk(d["q"], d["k"], d["v"], d["beta"], None, d["h0"],
                                   use_l2=False, scale=0.3)
    assert_parity("f32", o, ro, h, rh, tag="gk no gate")


def test_shared_gate_matches_scalar_path(kda, dev):
    """Every channel carrying one decay and the undecayed read: the per-channel kernel and
    the scalar recurrent kernel compute the same recurrence."""
    import torch
    d = make_gk(2, 90, 4, 128, 128, dtype="f32", gate_scale=0.5, h0="normal002", seed=14)
    dec = np.ascontiguousarray(d["g"][..., 0])
    d["g"] = np.ascontiguousarray(np.repeat(dec[..., None], 128, axis=-1))
    t = _dev_inputs(d, dev, "f32")
    o1, h1 = kda.gk_recurrent_fwd(t["q"], t["k"], t["v"], t["beta"], t["g"], t["h0"])
    o2, h2 = kda.recurrent_fwd(t["q"], t["k"], t["v"], t["beta"],
                               torch.from_numpy(dec).to(dev), t["h0"])
    torch.cuda.synchronize()
    assert torch.allclose(o1, o2, rtol=1e-5, atol=1e-6)
    assert torch.allclose(h1, h2, rtol=1e-5, atol=1e-6)


@pytest.mark.parametrize("decayed", [False, True])
def test_varlen(kda, oracle_mod, dev, decayed):
    import torch
    lengths = [0, 1, 63, 64, 65, 200, 7]
    d = make_gk(1, 0, 4, 128, 128, dtype="bf16", gate_scale=0.3, h0="normal002", seed=15,
                lengths=lengths)
    o, h = _run(kda, d, dev, "bf16", decayed, cu_seqlens_cpu=torch.from_numpy(d["cu_seqlens"]))
    ro, rh = oracle_mod.forward_gk(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"],
                                   cu_seqlens=d["cu_seqlens"], decayed_read=decayed)
    assert_parity("bf16", o, ro, h, rh, tag="gk varlen")


def test_zero_length_and_state_aliasing(kda, dev):
    import torch
    d = make_gk(2, 0, 2, 64, 64, dtype="f32", gate_scale=0.3, h0="normal002", seed=16)
    t = _dev_inputs(d, dev, "f32")
    h = t["h0"].clone()
    kda.gk_recurrent_fwd(t["q"], t["k"], t["v"], t["beta"], t["g"], h, final_state=h)
    _, h2 = kda.gk_recurrent_fwd(t["q"], t["k"], t["v"], t["beta"], t["g"], t["h0"])
    torch.cuda.synchronize()
    assert torch.equal(h, t["h0"]) and torch.equal(h2, t["h0"])
    # T > 0 with the final state written over the initial one
    d = make_gk(2, 40, 2, 64, 64, dtype="f32", gate_scale=0.3, h0="normal002", seed=17)
    t = _dev_inputs(d, dev, "f32")
    o_ref, h_ref = kda.gk_recurrent_fwd(t["q"], t["k"], t["v"], t["beta"], t["g"], t["h0"])
    h = t["h0"].clone()
    o, _ = kda.gk_recurrent_fwd(t["q"], t["k"], t["v"], t["beta"], t["g"], h, final_state=h)
    torch.cuda.synchronize()
    assert torch.equal(o, o_ref) and torch.equal(h, h_ref)


@pytest.mark.parametrize("decayed", [False, True])
@pytest.mark.parametrize("dtype,dims", [("bf16", (128, 128)), ("f32", (64, 64)),
                                        ("bf16", (64, 128)), ("f32", (32, 32))])
def test_decode_steps(kda, oracle_mod, dev, dtype, dims, decayed):
    """Eight single-token steps with the state carried in place, against the oracle's
    fp64 state carried over the same steps."""
    import torch
    dk, dv = dims
    B, H, steps = 6, 4, 8
    rng = np.random.Generator(np.random.PCG64(18))
    h0 = (0.3 * rng.standard_normal((B, H, dk, dv))).astype(np.float32)
    state = torch.from_numpy(h0).to(dev)
    ref = h0.astype(np.float64)
    for s in range(steps):
        st = make_gk_decode_step(B, H, dk, dv, s, dtype=dtype, gate_scale=2.0, seed=19)
        t = _dev_inputs(st, dev, dtype)
        o = kda.gk_decode_step(t["q"], t["k"], t["v"], t["beta"], t["g"], state,
                               decayed_read=decayed)
        ro, ref = oracle_mod.forward_gk(st["q"], st["k"], st["v"], st["beta"], st["g"], ref,
                                        decayed_read=decayed)
        torch.cuda.synchronize()
        assert_parity(dtype, to_np(o), ro, tag=f"decode step {s}")
    assert_parity(dtype, to_np(o), ro, to_np(state), ref, tag="decode final")


def test_decode_equals_prefill(kda, dev):
    """T single-token decode steps from a state = one T-token recurrent prefill."""
    import torch
    d = make_gk(3, 12, 2, 128, 128, dtype="f32", gate_scale=0.3, h0="normal002", seed=20)
    t = _dev_inputs(d, dev, "f32")
    o_ref, h_ref = kda.gk_recurrent_fwd(t["q"], t["k"], t["v"], t["beta"], t["g"], t["h0"],
                                        decayed_read=True)
    state = t["h0"].clone()
    outs = []
    for s in range(12):
        sl = slice(s, s + 1)
        outs.append(kda.gk_decode_step(t["q"][:, sl].contiguous(), t["k"][:, sl].contiguous(),
                                       t["v"][:, sl].contiguous(), t["beta"][:, sl].contiguous(),
                                       t["g"][:, sl].contiguous(), state, decayed_read=True))
    torch.cuda.synchronize()
    o = torch.cat(outs, dim=1)
    assert torch.allclose(o, o_ref, rtol=1e-5, atol=1e-6)
    assert torch.allclose(state, h_ref, rtol=1e-5, atol=1e-6)


def test_decode_full_size_head_sample(kda, oracle_mod, dev):
    """B=256 sequences x H=32 heads x 128 x 128 (the batched-decode shape), one step with
    per-channel gates; every head of eight batch entries (256 pairs) against the oracle."""
    import torch
    B, H, D = 256, 32, 128
    rng = np.random.Generator(np.random.PCG64(21))
    h0 = (0.02 * rng.standard_normal((B, H, D, D), dtype=np.float32)).astype(np.float32)
    st = make_gk_decode_step(B, H, D, D, 0, dtype="bf16", gate_scale=0.3, seed=22)
    t = _dev_inputs(st, dev, "bf16")
    state = torch.from_numpy(h0).to(dev)
    o = kda.gk_decode_step(t["q"], t["k"], t["v"], t["beta"], t["g"], state)
    torch.cuda.synchronize()
    batches = np.sort(rng.choice(B, size=8, replace=False))
    heads = (batches[:, None] * H + np.arange(H)[None, :]).reshape(-1)
    ro, rh = oracle_mod.forward_gk(st["q"], st["k"], st["v"], st["beta"], st["g"], h0,
                                   heads=heads)
    on, hn = to_np(o), to_np(state)
    b, h = heads // H, heads % H
    assert_parity("bf16", on[b, 0, h], ro[b, 0, h], hn[b, h], rh[b, h], tag="decode sample")


# ------------------------------------------------------------------ chunked (tensor cores)
def _run_chunk(kda, d, dev, dtype, decayed, chunk=64, **kw):
    import torch
    t = _dev_inputs(d, dev, dtype)
    o, h = kda.gk_chunk_fwd(t["q"], t["k"], t["v"], t["beta"], t["g"], t["h0"],
                            cu_seqlens=t.get("cu_seqlens"), decayed_read=decayed, chunk_size=chunk,
                            check_device=True, **kw)
    torch.cuda.synchronize()
    return to_np(o), to_np(h)


@pytest.mark.parametrize("decayed", [False, True])
@pytest.mark.parametrize("gate", [0.01, 0.3, 2.0, 6.0, 12.0])
@pytest.mark.parametrize("D", [128, 64])
def test_chunk_gate_regimes(kda, oracle_mod, dev, D, gate, decayed):
    """gate 12: about -6 per token, so most 16-token sub-blocks span more than e^60 in
    some channel and take the exact CUDA-core diagonal."""
    d = make_gk(2, 203, 3, D, D, dtype="bf16", gate_scale=gate, h0="normal002", seed=31)
    o, h = _run_chunk(kda, d, dev, "bf16", decayed)
    ro, rh = oracle_mod.forward_gk(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"],
                                   decayed_read=decayed)
    assert_parity("bf16", o, ro, h, rh, tag=f"gk chunk D={D} gate={gate} decayed={decayed}")


@pytest.mark.parametrize("T", [1, 16, 63, 64, 65, 130])
def test_chunk_lengths(kda, oracle_mod, dev, T):
    d = make_gk(2, T, 2, 128, 128, dtype="bf16", gate_scale=0.3, h0="normal002", seed=32)
    o, h = _run_chunk(kda, d, dev, "bf16", True)
    ro, rh = oracle_mod.forward_gk(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"],
                                   decayed_read=True)
    assert_parity("bf16", o, ro, h, rh, tag=f"gk chunk T={T}")


def test_chunk_several_rounds(kda, oracle_mod, dev):
    """More (sequence, head) pairs than chains (several rounds), 20 chunks per pair (more
    than the ring of E_c slots)."""
    d = make_gk(2, 1250, 48, 64, 64, dtype="bf16", gate_scale=0.3, h0="normal002", seed=33)
    o, h = _run_chunk(kda, d, dev, "bf16", False)
    ro, rh = oracle_mod.forward_gk(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"])
    assert_parity("bf16", o, ro, h, rh, tag="gk chunk several rounds")


@pytest.mark.parametrize("decayed", [False, True])
def test_chunk_varlen(kda, oracle_mod, dev, decayed):
    import torch
    lengths = [0, 1, 63, 64, 65, 200, 7]
    d = make_gk(1, 0, 4, 128, 128, dtype="bf16", gate_scale=2.0, h0="normal002", seed=34,
                lengths=lengths)
    o, h = _run_chunk(kda, d, dev, "bf16", decayed,
                      cu_seqlens_cpu=torch.from_numpy(d["cu_seqlens"]))
    ro, rh = oracle_mod.forward_gk(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"],
                                   cu_seqlens=d["cu_seqlens"], decayed_read=decayed)
    assert_parity("bf16", o, ro, h, rh, tag="gk chunk varlen")


def test_chunk_other_shapes_use_the_scan(kda, oracle_mod, dev):
    """fp32, or a chunk size other than 64: the per-channel token-by-token kernel."""
    d = make_gk(1, 70, 2, 64, 32, dtype="f32", gate_scale=0.3, h0="normal002", seed=35)
    o, h = _run_chunk(kda, d, dev, "f32", True, chunk=32)
    ro, rh = oracle_mod.forward_gk(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"],
                                   decayed_read=True)
    assert_parity("f32", o, ro, h, rh, tag="gk chunk fp32")


def test_chunk_training_shape(kda, oracle_mod, dev):
    """B=2, T=2048, H=16, d=128 (the training-shape workload) with g = -0.3 U[0,1)."""
    d = make_gk(2, 2048, 16, 128, 128, dtype="bf16", gate_scale=0.3, seed=36)
    o, h = _run_chunk(kda, d, dev, "bf16", True)
    ro, rh = oracle_mod.forward_gk(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"],
                                   decayed_read=True)
    assert_parity("bf16", o, ro, h, rh, tag="gk chunk training shape")


@pytest.mark.parametrize("packed", [False, True])
def test_chunk_without_gate(kda, oracle_mod, dev, packed):
    """g = None on the tensor-core shapes (bf16, d = 128, chunk 64), equal-length and packed:
    no decay, against the oracle with no gate."""
    import torch
    kw = dict(lengths=[70, 1, 200]) if packed else {}
    d = make_gk(2, 130, 2, 128, 128, dtype="bf16", gate_scale=0.1, h0="normal002", seed=39, **kw)
    t = _dev_inputs(d, dev, "bf16")
    extra = dict(cu_seqlens_cpu=torch.from_numpy(d["cu_seqlens"])) if packed else {}
    o, h = kda.gk_chunk_fwd(t["q"], t["k"], t["v"], t["beta"], None, t["h0"],
                            cu_seqlens=t.get("cu_seqlens"), check_device=True, **extra)
    torch.cuda.synchronize()
    ro, rh = oracle_mod.forward_gk(d["q"], d["k"], d["v"], d["beta"], None, d["h0"],
                                   cu_seqlens=d.get("cu_seqlens"))
    assert_parity("bf16", to_np(o), ro, to_np(h), rh, tag=f"gk chunk without gate packed={packed}")


def test_chunk_matches_recurrent_kernel(kda, dev):
    """The chunked and token-by-token per-channel kernels agree (bf16 rounding of E_c)."""
    import torch
    d = make_gk(1, 300, 8, 128, 128, dtype="bf16", gate_scale=1.0, h0="normal002", seed=37)
    t = _dev_inputs(d, dev, "bf16")
    o1, h1 = kda.gk_chunk_fwd(t["q"], t["k"], t["v"], t["beta"], t["g"], t["h0"], check_device=True)
    o2, h2 = kda.gk_recurrent_fwd(t["q"], t["k"], t["v"], t["beta"], t["g"], t["h0"])
    torch.cuda.synchronize()
    assert_parity("bf16", to_np(o1), to_np(o2), to_np(h1), to_np(h2), tag="chunk vs scan")


def test_chunk_full_size(kda, oracle_mod, dev):
    """The per-channel long-sequence prefill as timed: B=1, T=32768, H=32, d=128, one
    cooperative launch, g = -0.01 U[0,1), decayed read, carried-in state; every head against
    the oracle over the full T."""
    d = make_gk(1, 32768, 32, 128, 128, dtype="bf16", gate_scale=0.01, h0="normal002", seed=38)
    o, h = _run_chunk(kda, d, dev, "bf16", True)
    ro, rh = oracle_mod.forward_gk(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"],
                                   decayed_read=True)
    for hh in range(32):
        assert_parity("bf16", o[:, :, hh], ro[:, :, hh], h[:, hh], rh[:, hh],
                      tag=f"gk chunk full size head {hh}")
