"""GPU parity of the kernel options (kda_options): the decayed-read placement of the
per-head decay, the in-kernel gate (ejkernel kda_decay: -exp(A_log) softplus(gate + dt_bias);
TileOPs use_gate_in_kernel) and the beta transforms (use_beta_sigmoid_in_kernel,
allow_neg_eigval), on every path, against the fp64 oracle.  The oracle takes the transformed
decay / beta (its own fp64 transforms, rounded to float32 as kernel inputs are) and, for the
decayed read with one decay per head, its per-channel form with every channel equal."""
import numpy as np
import pytest

from kda_inputs import make_custom, make_gate_params, make_gk
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


def _t(x, dev, dtype=None):
    import torch
    if x is None:
        return None
    return to_dev(x, dev, dtype or torch.float32)


def _oracle(oracle_mod, d, decay, beta, decayed, **kw):
    """fp64 reference with the transformed decay and beta (float32 as a kernel would see them)."""
    dk = d["q"].shape[-1]
    beta = np.ascontiguousarray(beta, dtype=np.float32)
    if decayed:
        g = None if decay is None else np.ascontiguousarray(
            np.repeat(np.asarray(decay, np.float32)[..., None], dk, axis=-1))
        return oracle_mod.forward_gk(d["q"], d["k"], d["v"], beta, g, d.get("h0"), decayed_read=True, **kw)
    return oracle_mod.forward(d["q"], d["k"], d["v"], beta,
                              None if decay is None else np.asarray(decay, np.float32), d.get("h0"), **kw)


PATHS = [  # (dtype, dk, dv, chunk, T): tensor cores, CUDA-core chunks, odd shapes
    ("bf16", 128, 128, 64, 150),
    ("bf16", 64, 64, 64, 150),
    ("f32", 32, 32, 16, 70),
    ("f32", 64, 128, 32, 70),
]


@pytest.mark.parametrize("path", PATHS, ids=lambda p: f"{p[0]}-{p[1]}x{p[2]}-c{p[3]}")
@pytest.mark.parametrize("mode", ["decayed", "gate", "beta", "all"])
def test_chunk_options(kda, oracle_mod, dev, path, mode):
    import torch
    dtype, dk, dv, chunk, T = path
    B, H = 2, 3
    d = make_custom(B, T, H, dk, dv, dtype=dtype, decay="train", h0="normal002", seed=41)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    gate, A_log, dt_bias = make_gate_params((B, T, H), H, seed=41)
    decayed = mode in ("decayed", "all")
    use_gate = mode in ("gate", "all")
    use_beta = mode in ("beta", "all")
    raw_beta = (2.0 * d["beta"] - 1.0).astype(np.float32) * 3 if use_beta else d["beta"]
    dec_in = gate if use_gate else d["decay"]
    dec_ref = oracle_mod.gate_decay(gate, A_log, dt_bias) if use_gate else d["decay"]
    beta_ref = oracle_mod.beta_transform(raw_beta, allow_neg_eigval=(mode == "all")) if use_beta else raw_beta
    o, h = kda.chunk_fwd(_t(d["q"], dev, tdt), _t(d["k"], dev, tdt), _t(d["v"], dev, tdt),
                         _t(raw_beta, dev), _t(dec_in, dev), _t(d["h0"], dev), chunk_size=chunk,
                         check_device=True, decayed_read=decayed,
                         A_log=_t(A_log, dev) if use_gate else None,
                         dt_bias=_t(dt_bias, dev) if use_gate else None,
                         beta_sigmoid=use_beta, allow_neg_eigval=(mode == "all"))
    torch.cuda.synchronize()
    ro, rh = _oracle(oracle_mod, d, dec_ref, beta_ref, decayed)
    assert_parity(dtype, to_np(o), ro, to_np(h), rh, tag=f"chunk {path} {mode}")


@pytest.mark.parametrize("mode", ["decayed", "all"])
def test_recurrent_decode_varlen_options(kda, oracle_mod, dev, mode):
    import torch
    B, T, H, D = 2, 40, 4, 128
    d = make_custom(B, T, H, D, D, dtype="bf16", decay="train", h0="normal002", seed=42)
    gate, A_log, dt_bias = make_gate_params((B, T, H), H, seed=42)
    use = mode == "all"
    raw_beta = ((2.0 * d["beta"] - 1.0) * 3).astype(np.float32) if use else d["beta"]
    dec_in = gate if use else d["decay"]
    dec_ref = oracle_mod.gate_decay(gate, A_log, dt_bias) if use else d["decay"]
    beta_ref = oracle_mod.beta_transform(raw_beta) if use else raw_beta
    kw = dict(decayed_read=True, A_log=_t(A_log, dev) if use else None,
              dt_bias=_t(dt_bias, dev) if use else None, beta_sigmoid=use)
    q, k, v = (_t(d[n], dev, torch.bfloat16) for n in ("q", "k", "v"))
    o, h = kda.recurrent_fwd(q, k, v, _t(raw_beta, dev), _t(dec_in, dev), _t(d["h0"], dev), **kw)
    ro, rh = _oracle(oracle_mod, d, dec_ref, beta_ref, True)
    assert_parity("bf16", to_np(o), ro, to_np(h), rh, tag=f"recurrent {mode}")
    # decode: T single-token steps from h0
    state = _t(d["h0"], dev).clone()
    outs = []
    for t in range(T):
        sl = slice(t, t + 1)
        outs.append(kda.decode_step(q[:, sl].contiguous(), k[:, sl].contiguous(), v[:, sl].contiguous(),
                                    _t(np.ascontiguousarray(raw_beta[:, sl]), dev),
                                    _t(np.ascontiguousarray(dec_in[:, sl]), dev), state, **kw))
    torch.cuda.synchronize()
    assert_parity("bf16", to_np(torch.cat(outs, 1)), ro, to_np(state), rh, tag=f"decode {mode}")
    # packed: the two sequences back to back
    cu = np.array([0, T, 2 * T], np.int32)
    pk = {n: np.ascontiguousarray(d[n].reshape((1, B * T) + d[n].shape[2:])) for n in ("q", "k", "v")}
    o2, h2 = kda.varlen_fwd(*(_t(pk[n], dev, torch.bfloat16) for n in ("q", "k", "v")),
                            _t(np.ascontiguousarray(raw_beta.reshape(1, B * T, H)), dev),
                            _t(cu, dev, torch.int32),
                            _t(np.ascontiguousarray(dec_in.reshape(1, B * T, H)), dev), _t(d["h0"], dev),
                            cu_seqlens_cpu=torch.from_numpy(cu), check_device=True, **kw)
    torch.cuda.synchronize()
    assert_parity("bf16", to_np(o2).reshape(B, T, H, D), ro, to_np(h2), rh, tag=f"varlen {mode}")


@pytest.mark.parametrize("chunked", [True, False])
@pytest.mark.parametrize("D", [128, 64])
def test_gk_gate_and_beta(kda, oracle_mod, dev, chunked, D):
    """Per-channel gate in the kernel: g holds the raw gate, dt_bias [H, dk]."""
    import torch
    B, T, H = 2, 130, 3
    d = make_gk(B, T, H, D, D, dtype="bf16", gate_scale=0.3, h0="normal002", seed=43)
    gate, A_log, dt_bias = make_gate_params((B, T, H, D), H, K=D, seed=43)
    raw_beta = ((2.0 * d["beta"] - 1.0) * 3).astype(np.float32)
    g_ref = oracle_mod.gate_decay(gate, A_log, dt_bias).astype(np.float32)
    beta_ref = oracle_mod.beta_transform(raw_beta, allow_neg_eigval=True).astype(np.float32)
    q, k, v = (_t(d[n], dev, torch.bfloat16) for n in ("q", "k", "v"))
    kw = dict(decayed_read=True, A_log=_t(A_log, dev), dt_bias=_t(dt_bias, dev), beta_sigmoid=True,
              allow_neg_eigval=True)
    if chunked:
        o, h = kda.gk_chunk_fwd(q, k, v, _t(raw_beta, dev), _t(gate, dev), _t(d["h0"], dev),
                                check_device=True, **kw)
    else:
        o, h = kda.gk_recurrent_fwd(q, k, v, _t(raw_beta, dev), _t(gate, dev), _t(d["h0"], dev), **kw)
    torch.cuda.synchronize()
    ro, rh = oracle_mod.forward_gk(d["q"], d["k"], d["v"], beta_ref, g_ref, d["h0"], decayed_read=True)
    assert_parity("bf16", to_np(o), ro, to_np(h), rh, tag=f"gk gate chunked={chunked} D={D}")
    if not chunked:   # one decode step from the final state, with the same options
        state = h.clone()
        st = make_gk(B, 1, H, D, D, dtype="bf16", gate_scale=0.3, seed=44)
        g1, _, _ = make_gate_params((B, 1, H, D), H, K=D, seed=44)
        b1 = ((2.0 * st["beta"] - 1.0) * 3).astype(np.float32)
        o1 = kda.gk_decode_step(*(_t(st[n], dev, torch.bfloat16) for n in ("q", "k", "v")), _t(b1, dev),
                                _t(g1, dev), state, **kw)
        torch.cuda.synchronize()
        r1, rs = oracle_mod.forward_gk(st["q"], st["k"], st["v"],
                                       oracle_mod.beta_transform(b1, True).astype(np.float32),
                                       oracle_mod.gate_decay(g1, A_log, dt_bias).astype(np.float32),
                                       to_np(h), decayed_read=True)
        assert_parity("bf16", to_np(o1), r1, to_np(state), rs, tag="gk decode gate")


@pytest.mark.parametrize("K", [1, 128])
def test_gate_decay_op(kda, oracle_mod, dev, K):
    H = 4
    shape = (3, 17, H) if K == 1 else (3, 17, H, K)
    gate, A_log, dt_bias = make_gate_params(shape, H, K=K, seed=45)
    gate = gate * 5   # the softplus tails as well
    out = kda.gate_decay(_t(gate, dev), _t(A_log, dev), _t(dt_bias, dev))
    ref = oracle_mod.gate_decay(gate, A_log, dt_bias)
    got = to_np(out)
    assert np.all(got <= 0)
    assert np.max(np.abs(got - ref) / np.maximum(np.abs(ref), 1e-30)) < 1e-5
    z = kda.gate_decay(_t(np.zeros((2, 10, H), np.float32), dev), _t(np.zeros(H, np.float32), dev))
    assert np.allclose(to_np(z), -np.log(2.0), rtol=1e-6)


def test_gated_long_prefill(kda, oracle_mod, dev):
    """The long-sequence workload with the prologues in the kernel, as timed (B=1, T=32768,
    H=32, d=128, raw gate with A_log and dt_bias, beta from logits, decayed read, carried-in
    state); every head against the oracle over the full T."""
    import torch
    from kda_inputs import WORKLOADS, make_prefill
    wl = WORKLOADS[3]
    d = make_prefill(wl, seed=3)
    gate, A_log, dt_bias = make_gate_params((wl.B, wl.T, wl.H), wl.H, seed=3)
    raw_beta = ((2.0 * d["beta"] - 1.0) * 3).astype(np.float32)
    q, k, v = (_t(d[n], dev, torch.bfloat16) for n in ("q", "k", "v"))
    o, h = kda.chunk_fwd(q, k, v, _t(raw_beta, dev), _t(gate, dev), _t(d["h0"], dev),
                         chunk_size=wl.chunk, check_device=True, decayed_read=True,
                         A_log=_t(A_log, dev), dt_bias=_t(dt_bias, dev), beta_sigmoid=True)
    torch.cuda.synchronize()
    heads = np.arange(wl.H)
    sub = {n: np.ascontiguousarray(d[n][:, :, heads]) for n in ("q", "k", "v")}
    sub["h0"] = np.ascontiguousarray(d["h0"][:, heads])
    dec_ref = oracle_mod.gate_decay(np.ascontiguousarray(gate[:, :, heads]), np.ascontiguousarray(A_log[heads]),
                                    np.ascontiguousarray(dt_bias[heads]))
    beta_ref = oracle_mod.beta_transform(np.ascontiguousarray(raw_beta[:, :, heads]))
    ro, rh = _oracle(oracle_mod, sub, dec_ref, beta_ref, True)
    on, hn = to_np(o), to_np(h)
    for hh in heads:
        assert_parity("bf16", on[:, :, hh], ro[:, :, hh], hn[:, hh], rh[:, hh],
                      tag=f"gated long prefill head {hh}")
