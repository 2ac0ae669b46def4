"""GPU parity with value-major states (TileOPs GDNFwdOp / KDAFwdOp state_v_first: [N, HV, V, K]
instead of key-major [N, HV, K, V]) on every path: the same recurrence, the initial and final
states (and the decode state) transposed per head.  Against the fp64 oracle, which takes and
returns key-major states."""
import numpy as np
import pytest

from kda_inputs import make_custom, make_gk
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


def _T(x):   # key-major <-> value-major, per head
    return np.ascontiguousarray(np.swapaxes(x, -1, -2))


def _dev(x, dev, dtype=None):
    import torch
    return None if x is None else to_dev(x, dev, dtype or torch.float32)


@pytest.mark.parametrize("path", [("bf16", 128, 128, 64), ("bf16", 64, 64, 64), ("f32", 64, 128, 32),
                                  ("f32", 32, 32, 16), ("f32", 128, 64, 64)],
                         ids=lambda p: f"{p[0]}-{p[1]}x{p[2]}-c{p[3]}")
@pytest.mark.parametrize("recurrent", [False, True])
def test_prefill(kda, oracle_mod, dev, path, recurrent):
    import torch
    dtype, dk, dv, chunk = path
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    d = make_custom(2, 130, 3, dk, dv, dtype=dtype, decay="train", h0="normal002", seed=61)
    d["h0"] = (d["h0"] * 20).astype(np.float32)
    args = [_dev(d[n], dev, tdt) for n in ("q", "k", "v")] + [_dev(d["beta"], dev), _dev(d["decay"], dev),
                                                            _dev(_T(d["h0"]), dev)]
    if recurrent:
        o, h = kda.recurrent_fwd(*args, state_v_first=True)
    else:
        o, h = kda.chunk_fwd(*args, chunk_size=chunk, check_device=True, state_v_first=True)
    torch.cuda.synchronize()
    assert h.shape == (2, 3, dv, dk)
    ro, rh = oracle_mod.forward(d["q"], d["k"], d["v"], d["beta"], d["decay"], d["h0"])
    assert_parity(dtype, to_np(o), ro, _T(to_np(h)), rh, tag=f"v-first {path} recurrent={recurrent}")


@pytest.mark.parametrize("dtype,dims", [("bf16", (128, 128)), ("f32", (64, 32)), ("f32", (32, 128))])
def test_decode_in_place(kda, oracle_mod, dev, dtype, dims):
    import torch
    dk, dv = dims
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    d = make_custom(5, 3, 4, dk, dv, dtype=dtype, decay="train", h0="normal002", seed=62)
    d["h0"] = (d["h0"] * 20).astype(np.float32)
    state = _dev(_T(d["h0"]), dev)
    outs = []
    for t in range(3):
        sl = slice(t, t + 1)
        outs.append(kda.decode_step(*(_dev(np.ascontiguousarray(d[n][:, sl]), dev, tdt) for n in ("q", "k", "v")),
                                    _dev(np.ascontiguousarray(d["beta"][:, sl]), dev),
                                    _dev(np.ascontiguousarray(d["decay"][:, sl]), dev), state,
                                    state_v_first=True))
    torch.cuda.synchronize()
    ro, rh = oracle_mod.forward(d["q"], d["k"], d["v"], d["beta"], d["decay"], d["h0"])
    assert_parity(dtype, to_np(torch.cat(outs, 1)), ro, _T(to_np(state)), rh, tag=f"v-first decode {dims}")


def test_varlen_and_per_channel(kda, oracle_mod, dev):
    import torch
    lengths = [0, 70, 5, 129]
    d = make_gk(1, 0, 2, 128, 128, dtype="bf16", gate_scale=0.5, h0="normal002", seed=63, lengths=lengths)
    d["h0"] = (d["h0"] * 20).astype(np.float32)
    cu = torch.from_numpy(d["cu_seqlens"])
    q, k, v = (_dev(d[n], dev, torch.bfloat16) for n in ("q", "k", "v"))
    beta, g, h0v = _dev(d["beta"], dev), _dev(d["g"], dev), _dev(_T(d["h0"]), dev)
    cud = cu.to(dev)
    for chunked in (True, False):
        f = kda.gk_chunk_fwd if chunked else kda.gk_recurrent_fwd
        kw = dict(check_device=True) if chunked else {}
        o, h = f(q, k, v, beta, g, h0v, cu_seqlens=cud, cu_seqlens_cpu=cu, decayed_read=True,
                 state_v_first=True, **kw)
        torch.cuda.synchronize()
        ro, rh = oracle_mod.forward_gk(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"],
                                       cu_seqlens=d["cu_seqlens"], decayed_read=True)
        assert_parity("bf16", to_np(o), ro, _T(to_np(h)), rh, tag=f"v-first per-channel chunked={chunked}")
    # scalar-decay packed prefill with value-major states (g's first channel as the decay)
    dec = np.ascontiguousarray(d["g"][..., 0])
    o, h = kda.varlen_fwd(q, k, v, beta, cud, _dev(dec, dev), h0v, cu_seqlens_cpu=cu, check_device=True,
                          state_v_first=True)
    torch.cuda.synchronize()
    ro, rh = oracle_mod.varlen(d["q"], d["k"], d["v"], d["beta"], d["cu_seqlens"], dec, d["h0"])
    assert_parity("bf16", to_np(o), ro, _T(to_np(h)), rh, tag="v-first varlen")
    # per-channel decode, in place
    st = make_gk(4, 1, 2, 128, 128, dtype="bf16", gate_scale=0.5, h0="normal002", seed=64)
    st["h0"] = (st["h0"] * 20).astype(np.float32)
    state = _dev(_T(st["h0"]), dev)
    o = kda.gk_decode_step(*(_dev(st[n], dev, torch.bfloat16) for n in ("q", "k", "v")), _dev(st["beta"], dev),
                           _dev(st["g"], dev), state, decayed_read=True, state_v_first=True)
    torch.cuda.synchronize()
    ro, rh = oracle_mod.forward_gk(st["q"], st["k"], st["v"], st["beta"], st["g"], st["h0"], decayed_read=True)
    assert_parity("bf16", to_np(o), ro, _T(to_np(state)), rh, tag="v-first per-channel decode")
