"""GPU parity: every path through the C ABI against the fp64 oracle.

Inputs come from the shared seeded generator; the oracle runs on the same
(bf16-rounded where the workload is bf16) values.  Bars:
fp32: max|diff|/max|ref| <= 1e-4 on o and final_state;
bf16: max|do| <= 2e-2 max|o| and final_state Frobenius-relative <= 1e-2.
"""
import numpy as np
import pytest

from kda_inputs import WORKLOADS, make_custom, make_decode_state, make_decode_step, make_prefill, \
    make_varlen
from _util import assert_parity, inputs_to_dev, max_rel, frob_rel, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kda():
    """The binding, with every prefill call checking the device error word afterwards
    (a kernel whose bounded wait ran out makes the call raise)."""
    import functools
    import types

    import delta_rule_linear_gb300 as m
    from delta_rule_linear_gb300 import build as b
    b.build()
    m.load()
    return types.SimpleNamespace(
        chunk_fwd=functools.partial(m.chunk_fwd, check_device=True),
        varlen_fwd=functools.partial(m.varlen_fwd, check_device=True),
        recurrent_fwd=m.recurrent_fwd, decode_step=m.decode_step)


@pytest.fixture(scope="module")
def dev():
    import torch
    return torch.device("cuda:0")


def _run_chunk(kda, d, dev, dtype, chunk, use_l2=True, scale=None, recurrent=False):
    import torch
    t = inputs_to_dev(d, dev, dtype)
    if recurrent:
        o, h = kda.recurrent_fwd(t["q"], t["k"], t["v"], t["beta"], t["decay"], t["h0"],
                                 scale=scale, use_qk_l2norm=use_l2)
    else:
        o, h = kda.chunk_fwd(t["q"], t["k"], t["v"], t["beta"], t["decay"], t["h0"], scale=scale,
                             chunk_size=chunk, use_qk_l2norm=use_l2)
    torch.cuda.synchronize()
    return to_np(o), to_np(h)


# ---------------------------------------------------------------- the five workloads
@pytest.mark.parametrize("recurrent", [False, True])
def test_tiny_fp32_workload(kda, oracle_mod, dev, recurrent):
    wl = WORKLOADS[1]
    d = make_prefill(wl, seed=0)
    o, h = _run_chunk(kda, d, dev, "f32", wl.chunk, recurrent=recurrent)
    ro, rh = oracle_mod.forward(d["q"], d["k"], d["v"], d["beta"], d["decay"], d["h0"])
    assert_parity("f32", o, ro, h, rh, tag="tiny")


def test_training_shape_workload(kda, oracle_mod, dev):
    wl = WORKLOADS[2]
    d = make_prefill(wl, seed=0)
    o, h = _run_chunk(kda, d, dev, "bf16", wl.chunk)
    ro, rh = oracle_mod.forward(d["q"], d["k"], d["v"], d["beta"], d["decay"], d["h0"])
    assert_parity("bf16", o, ro, h, rh, tag="train")


def _select_heads(d, heads, H):
    """Gather (b, h) pairs into a batch of single-head problems [n, T, 1, D]."""
    out = {}
    for n in ("q", "k", "v", "beta", "decay"):
        x = d.get(n)
        out[n] = None if x is None else np.ascontiguousarray(
            np.stack([x[bh // H, :, bh % H] for bh in heads])[:, :, None])
    h0 = d.get("h0")
    out["h0"] = None if h0 is None else np.ascontiguousarray(
        np.stack([h0[bh // H, bh % H] for bh in heads])[:, None])
    return out


def test_long_sequence_workload(kda, oracle_mod, dev):
    """Full T=32768, H=32 on the GPU, every head checked against the oracle over the full
    length (the oracle runs its heads on all host threads)."""
    wl = WORKLOADS[3]
    d = make_prefill(wl, seed=0)
    o, h = _run_chunk(kda, d, dev, "bf16", wl.chunk)
    ro, rh = oracle_mod.forward(d["q"], d["k"], d["v"], d["beta"], d["decay"], d["h0"])
    for bh in range(wl.B * wl.H):
        b, hh = divmod(bh, wl.H)
        assert_parity("bf16", o[b, :, hh], ro[b, :, hh], h[b, hh], rh[b, hh], tag=f"long head {bh}")


def test_batched_decode_workload_head_sample(kda, oracle_mod, dev):
    """128 decode steps over B=256, H=32 on the GPU; the oracle follows every head of eight
    batch entries spread over the batch (256 (b, h) pairs, each through all 128 steps)."""
    import torch
    wl = WORKLOADS[4]
    S0 = make_decode_state(wl, seed=0)
    state = torch.from_numpy(S0).to(dev)
    batches = sorted(np.random.default_rng(1).choice(wl.B, size=8, replace=False).tolist())
    heads = [b * wl.H + hh for b in batches for hh in range(wl.H)]
    steps, outs = [], []
    for s in range(wl.steps):
        st = make_decode_step(wl, s, seed=0)
        t = inputs_to_dev(st, dev, "bf16")
        o = kda.decode_step(t["q"], t["k"], t["v"], t["beta"], t["decay"], state)
        outs.append(to_np(o))
        steps.append(_select_heads(st, heads, wl.H))
    torch.cuda.synchronize()
    h0 = np.stack([S0[bh // wl.H, bh % wl.H] for bh in heads])[:, None]
    routs, rh = oracle_mod.decode_steps(steps, h0)
    hs = to_np(state)
    for i, bh in enumerate(heads):
        b, hh = divmod(bh, wl.H)
        go = np.stack([x[b, 0, hh] for x in outs])
        ro = np.stack([x[i, 0, 0] for x in routs])
        assert_parity("bf16", go, ro, hs[b, hh], rh[i, 0], tag=f"decode head {bh}")
    assert np.all(np.isfinite(hs))


def test_varlen_workload(kda, oracle_mod, dev):
    import torch
    wl = WORKLOADS[5]
    d = make_varlen(wl, seed=0)
    t = inputs_to_dev(d, dev, "bf16")
    o, h = kda.varlen_fwd(t["q"], t["k"], t["v"], t["beta"], t["cu_seqlens"], t["decay"], t["h0"],
                          cu_seqlens_cpu=torch.from_numpy(d["cu_seqlens"]), chunk_size=wl.chunk)
    torch.cuda.synchronize()
    ro, rh = oracle_mod.varlen(d["q"], d["k"], d["v"], d["beta"], d["cu_seqlens"], d["decay"],
                               d["h0"])
    assert_parity("bf16", to_np(o), ro, to_np(h), rh, tag="varlen")


# ---------------------------------------------------------------- shapes and edge cases
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("chunk", [16, 32, 64])
@pytest.mark.parametrize("T", [1, 15, 64, 65, 200])
def test_chunk_lengths(kda, oracle_mod, dev, dtype, chunk, T):
    d = make_custom(2, T, 3, 64, 64, dtype=dtype, decay="train", h0="normal002", seed=T + chunk)
    o, h = _run_chunk(kda, d, dev, dtype, chunk)
    ro, rh = oracle_mod.forward(d["q"], d["k"], d["v"], d["beta"], d["decay"], d["h0"])
    assert_parity(dtype, o, ro, h, rh, tag=f"T={T} C={chunk}")


@pytest.mark.parametrize("dims", [(32, 32), (32, 128), (128, 32), (64, 128), (128, 64), (128, 128)])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_head_dims(kda, oracle_mod, dev, dims, dtype):
    dk, dv = dims
    d = make_custom(1, 150, 2, dk, dv, dtype=dtype, decay="long", h0="normal002", seed=dk + dv)
    for recurrent in (False, True):
        o, h = _run_chunk(kda, d, dev, dtype, 64, recurrent=recurrent)
        ro, rh = oracle_mod.forward(d["q"], d["k"], d["v"], d["beta"], d["decay"], d["h0"])
        assert_parity(dtype, o, ro, h, rh, tag=f"dk={dk} dv={dv} rec={recurrent}")


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("decay", ["strong", "mixed"])
def test_strong_decay(kda, oracle_mod, dev, D, decay):
    """Chunks whose log-decay sum falls far below -80, where any factorisation of the decay
    ratios exp(G_a - G_b) into per-token exponentials would overflow fp32; "mixed"
    alternates such chunks with weakly decaying ones along the sequence."""
    d = make_custom(2, 300, 2, D, D, dtype="bf16", decay=decay, h0="normal002", seed=D + len(decay))
    o, h = _run_chunk(kda, d, dev, "bf16", 64)
    ro, rh = oracle_mod.forward(d["q"], d["k"], d["v"], d["beta"], d["decay"], d["h0"])
    assert_parity("bf16", o, ro, h, rh, tag=f"D={D} decay={decay}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_no_decay_no_state_no_l2_custom_scale(kda, oracle_mod, dev, dtype):
    d = make_custom(2, 100, 2, 64, 64, dtype=dtype, decay="none", h0="zero", seed=3,
                    qkv_scale=1.0 / 8.0)   # small raw keys keep the unnormalised run contractive
    for use_l2, scale in ((False, 0.3), (True, 0.5), (True, None)):
        o, h = _run_chunk(kda, d, dev, dtype, 32, use_l2=use_l2, scale=scale)
        ro, rh = oracle_mod.forward(d["q"], d["k"], d["v"], d["beta"], None, None, scale=scale,
                                    use_l2=use_l2)
        assert_parity(dtype, o, ro, h, rh, tag=f"l2={use_l2} scale={scale}")


def test_zero_length_and_aliasing(kda, oracle_mod, dev):
    import torch
    d = make_custom(2, 0, 2, 64, 64, dtype="bf16", decay="train", h0="normal002", seed=4)
    t = inputs_to_dev(d, dev, "bf16")
    o, h = kda.chunk_fwd(t["q"], t["k"], t["v"], t["beta"], t["decay"], t["h0"], chunk_size=64)
    torch.cuda.synchronize()
    assert np.array_equal(to_np(h), d["h0"].astype(np.float64))
    # final_state aliasing initial_state: the state is read before it is overwritten
    d = make_custom(2, 77, 2, 64, 64, dtype="bf16", decay="train", h0="normal002", seed=5)
    t = inputs_to_dev(d, dev, "bf16")
    st = t["h0"].clone()
    kda.chunk_fwd(t["q"], t["k"], t["v"], t["beta"], t["decay"], st, chunk_size=64, final_state=st)
    torch.cuda.synchronize()
    ro, rh = oracle_mod.forward(d["q"], d["k"], d["v"], d["beta"], d["decay"], d["h0"])
    assert frob_rel(to_np(st), rh) <= 1e-2


def test_split_and_chain_state(kda, oracle_mod, dev):
    """Two calls chained through final_state equal one call (split mid-chunk)."""
    import torch
    d = make_custom(1, 300, 2, 128, 128, dtype="bf16", decay="train", h0="normal002", seed=6)
    t = inputs_to_dev(d, dev, "bf16")
    cut = 137
    part = lambda x, a, b: None if x is None else x[:, a:b].contiguous()  # noqa: E731
    o1, h1 = kda.chunk_fwd(*(part(t[n], 0, cut) for n in ("q", "k", "v", "beta", "decay")), t["h0"])
    o2, h2 = kda.chunk_fwd(*(part(t[n], cut, 300) for n in ("q", "k", "v", "beta", "decay")), h1)
    torch.cuda.synchronize()
    ro, rh = oracle_mod.forward(d["q"], d["k"], d["v"], d["beta"], d["decay"], d["h0"])
    o = np.concatenate([to_np(o1), to_np(o2)], axis=1)
    assert_parity("bf16", o, ro, to_np(h2), rh, tag="split")


def test_decode_equals_prefill(kda, dev):
    """T single-token decode steps give the prefill's outputs and state."""
    import torch
    d = make_custom(3, 12, 2, 128, 128, dtype="bf16", decay="small", h0="normal002", seed=7)
    t = inputs_to_dev(d, dev, "bf16")
    o, h = kda.chunk_fwd(t["q"], t["k"], t["v"], t["beta"], t["decay"], t["h0"])
    st = t["h0"].clone()
    outs = []
    for i in range(12):
        sl = lambda x: x[:, i:i + 1].contiguous()  # noqa: E731
        outs.append(kda.decode_step(sl(t["q"]), sl(t["k"]), sl(t["v"]), sl(t["beta"]),
                                    sl(t["decay"]), st))
    torch.cuda.synchronize()
    od = torch.cat(outs, dim=1)
    # the decode path is fp32 throughout; the bf16 prefill runs its products on bf16
    # operands, so the two agree to the bf16 bar
    assert max_rel(to_np(od), to_np(o)) <= 2e-2
    assert frob_rel(to_np(st), to_np(h)) <= 1e-2


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dims", [(32, 32), (64, 64), (128, 128), (128, 64)])
def test_decode_shapes(kda, oracle_mod, dev, dtype, dims):
    import torch
    dk, dv = dims
    d = make_custom(5, 1, 3, dk, dv, dtype=dtype, decay="small", h0="normal002", seed=dk)
    t = inputs_to_dev(d, dev, dtype)
    st = t["h0"].clone()
    o = kda.decode_step(t["q"], t["k"], t["v"], t["beta"], t["decay"], st)
    torch.cuda.synchronize()
    ro, rh = oracle_mod.forward(d["q"], d["k"], d["v"], d["beta"], d["decay"], d["h0"])
    assert_parity(dtype, to_np(o), ro, to_np(st), rh, tag="decode")


def test_varlen_edge_lengths(kda, oracle_mod, dev):
    """Empty sequences, length-1 sequences, exact chunk multiples, and a decay."""
    import torch
    from kda_inputs import Workload
    wl = Workload("edge", "varlen", "bf16", 1, 0, 2, 128, 128, 64, True, "train", "normal002",
                  nseq=7)
    d = make_varlen(wl, seed=3, lengths=[0, 1, 64, 65, 0, 130, 7])
    t = inputs_to_dev(d, dev, "bf16")
    for host in (True, False):
        o, h = kda.varlen_fwd(t["q"], t["k"], t["v"], t["beta"], t["cu_seqlens"], t["decay"],
                              t["h0"], cu_seqlens_cpu=torch.from_numpy(d["cu_seqlens"]) if host
                              else None)
        torch.cuda.synchronize()
        ro, rh = oracle_mod.varlen(d["q"], d["k"], d["v"], d["beta"], d["cu_seqlens"], d["decay"],
                                   d["h0"])
        assert_parity("bf16", to_np(o), ro, to_np(h), rh, tag=f"varlen edge host={host}")


@pytest.mark.parametrize("extra", [0, 1])
def test_chain_rounds(kda, oracle_mod, dev, extra):
    """B*H at a quarter of the SM count (the most chains there are): one chain per
    (sequence, head), a single round; one pair more: fewer chains than pairs, two rounds.
    T = 1100 (18 chunks) wraps every chain's ring of E_c slots.  Both against the oracle."""
    import torch
    quarter = torch.cuda.get_device_properties(dev).multi_processor_count // 4
    nsh = quarter + extra
    H = next(h for h in (19, 17, 13, 11, 7, 5, 3, 2, 1) if nsh % h == 0)
    d = make_custom(nsh // H, 1100, H, 64, 64, dtype="bf16", decay="train", h0="normal002",
                    seed=nsh)
    o, h = _run_chunk(kda, d, dev, "bf16", 64)
    ro, rh = oracle_mod.forward(d["q"], d["k"], d["v"], d["beta"], d["decay"], d["h0"])
    assert_parity("bf16", o, ro, h, rh, tag=f"B*H={nsh}")


def test_varlen_several_rounds(kda, oracle_mod, dev):
    """More (sequence, head) pairs than chains (several rounds, sequences taken longest
    first), with ragged and empty sequences and some longer than the ring of E_c slots."""
    import torch
    from kda_inputs import Workload
    quarter = torch.cuda.get_device_properties(dev).multi_processor_count // 4
    lengths = [5, 130, 0, 64, 1900, 1, 63, 128, 77, 0, 190, 33, 1100, 512, 513, 2]
    H = -(-2 * quarter // len(lengths))   # at least twice as many pairs as chains
    wl = Workload("many", "varlen", "bf16", 1, 0, H, 64, 64, 64, True, "long", "normal002",
                  nseq=len(lengths))
    d = make_varlen(wl, seed=5, lengths=lengths)
    t = inputs_to_dev(d, dev, "bf16")
    for host in (True, False):
        o, h = kda.varlen_fwd(t["q"], t["k"], t["v"], t["beta"], t["cu_seqlens"], t["decay"], t["h0"],
                              cu_seqlens_cpu=torch.from_numpy(d["cu_seqlens"]) if host else None,
                              chunk_size=64)
        torch.cuda.synchronize()
        ro, rh = oracle_mod.varlen(d["q"], d["k"], d["v"], d["beta"], d["cu_seqlens"], d["decay"],
                                   d["h0"])
        assert_parity("bf16", to_np(o), ro, to_np(h), rh, tag=f"varlen many pairs host={host}")
