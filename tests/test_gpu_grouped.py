"""GPU parity of grouped value heads (TileOPs GDNFwdOp / KDAFwdOp: q and k have H heads; v, beta,
the decay or g, the output and the state have HV = m H heads).  Reading taken: value head hv
uses q/k head hv // m (consecutive value heads share a q/k head).  The oracle runs the plain
recurrence with q and k repeated m times along the head axis."""
import numpy as np
import pytest

from kda_inputs import make_custom, make_gate_params, make_gk
from _util import assert_parity, to_dev, to_np

pytestmark = pytest.mark.gpu
M = 3   # value heads per q/k head


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


def _split(d, m=M):
    """q, k keep every m-th head (H = HV / m); the oracle sees them repeated m times."""
    qk = {n: np.ascontiguousarray(d[n][:, :, ::m]) for n in ("q", "k")}
    rep = {n: np.ascontiguousarray(np.repeat(qk[n], m, axis=2)) for n in ("q", "k")}
    return qk, rep


def _dev(x, dev, dtype=None):
    import torch
    return None if x is None else to_dev(x, dev, dtype or torch.float32)


@pytest.mark.parametrize("path", [("bf16", 128, 128, 64), ("bf16", 64, 64, 64), ("f32", 32, 32, 16),
                                  ("f32", 64, 128, 32)], ids=lambda p: f"{p[0]}-{p[1]}x{p[2]}-c{p[3]}")
def test_chunk(kda, oracle_mod, dev, path):
    import torch
    dtype, dk, dv, chunk = path
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    d = make_custom(2, 150, 2 * M, dk, dv, dtype=dtype, decay="train", h0="normal002", seed=51)
    qk, rep = _split(d)
    o, h = kda.chunk_fwd(_dev(qk["q"], dev, tdt), _dev(qk["k"], dev, tdt), _dev(d["v"], dev, tdt),
                         _dev(d["beta"], dev), _dev(d["decay"], dev), _dev(d["h0"], dev),
                         chunk_size=chunk, check_device=True)
    torch.cuda.synchronize()
    assert o.shape == d["v"].shape and h.shape == d["h0"].shape
    ro, rh = oracle_mod.forward(rep["q"], rep["k"], d["v"], d["beta"], d["decay"], d["h0"])
    assert_parity(dtype, to_np(o), ro, to_np(h), rh, tag=f"grouped chunk {path}")


def test_recurrent_decode_varlen_and_gate(kda, oracle_mod, dev):
    import torch
    B, T, HV, D = 2, 40, 2 * M, 128
    d = make_custom(B, T, HV, D, D, dtype="bf16", decay="train", h0="normal002", seed=52)
    qk, rep = _split(d)
    gate, A_log, dt_bias = make_gate_params((B, T, HV), HV, seed=52)
    dec_ref = oracle_mod.gate_decay(gate, A_log, dt_bias).astype(np.float32)
    kw = dict(A_log=_dev(A_log, dev), dt_bias=_dev(dt_bias, dev))
    q, k, v = (_dev(x, dev, torch.bfloat16) for x in (qk["q"], qk["k"], d["v"]))
    beta, g, h0 = _dev(d["beta"], dev), _dev(gate, dev), _dev(d["h0"], dev)
    ro, rh = oracle_mod.forward(rep["q"], rep["k"], d["v"], d["beta"], dec_ref, d["h0"])
    o, h = kda.recurrent_fwd(q, k, v, beta, g, h0, **kw)
    torch.cuda.synchronize()
    assert_parity("bf16", to_np(o), ro, to_np(h), rh, tag="grouped recurrent")
    state = h0.clone()
    outs = [kda.decode_step(q[:, t:t + 1].contiguous(), k[:, t:t + 1].contiguous(),
                            v[:, t:t + 1].contiguous(), beta[:, t:t + 1].contiguous(),
                            g[:, t:t + 1].contiguous(), state, **kw) for t in range(T)]
    torch.cuda.synchronize()
    assert_parity("bf16", to_np(torch.cat(outs, 1)), ro, to_np(state), rh, tag="grouped decode")
    cu = np.array([0, T, 2 * T], np.int32)
    flat = lambda x: x.reshape((1, B * T) + tuple(x.shape[2:])).contiguous()  # noqa: E731
    o2, h2 = kda.varlen_fwd(flat(q), flat(k), flat(v), flat(beta), _dev(cu, dev, torch.int32), flat(g), h0,
                            cu_seqlens_cpu=torch.from_numpy(cu), check_device=True, **kw)
    torch.cuda.synchronize()
    assert_parity("bf16", to_np(o2).reshape(B, T, HV, D), ro, to_np(h2), rh, tag="grouped varlen")


@pytest.mark.parametrize("which", ["chunk", "recurrent", "decode"])
def test_per_channel(kda, oracle_mod, dev, which):
    import torch
    B, T, HV, D = 2, 70 if which != "decode" else 1, 2 * M, 128
    d = make_gk(B, T, HV, D, D, dtype="bf16", gate_scale=0.5, h0="normal002", seed=53)
    qk, rep = _split(d)
    q, k, v = (_dev(x, dev, torch.bfloat16) for x in (qk["q"], qk["k"], d["v"]))
    beta, g, h0 = _dev(d["beta"], dev), _dev(d["g"], dev), _dev(d["h0"], dev)
    if which == "chunk":
        o, h = kda.gk_chunk_fwd(q, k, v, beta, g, h0, decayed_read=True, check_device=True)
    elif which == "recurrent":
        o, h = kda.gk_recurrent_fwd(q, k, v, beta, g, h0, decayed_read=True)
    else:
        h = h0.clone()
        o = kda.gk_decode_step(q, k, v, beta, g, h, decayed_read=True)
    torch.cuda.synchronize()
    ro, rh = oracle_mod.forward_gk(rep["q"], rep["k"], d["v"], d["beta"], d["g"], d["h0"],
                                   decayed_read=True)
    assert_parity("bf16", to_np(o), ro, to_np(h), rh, tag=f"grouped per-channel {which}")
