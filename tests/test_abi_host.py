"""Host-side checks of the C ABI: the library loads, exports every declared symbol,
answers workspace queries, and rejects bad arguments before touching the device.

None of these calls reaches a CUDA launch (argument errors return first), so they
run without a GPU.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kda.h")


@pytest.fixture(scope="module")
def lib():
    from delta_rule_linear_gb300 import build as b
    b.build()
    from delta_rule_linear_gb300 import _lib
    return _lib.load()


def _declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"\b(kda_[a-z_]+)\s*\(", src)
    return sorted(set(names))


def test_header_declares_expected_entry_points():
    names = _declared_functions()
    for n in ("kda_chunk_fwd", "kda_decode_step", "kda_varlen_fwd", "kda_chunk_fwd_workspace",
              "kda_varlen_fwd_workspace", "kda_query_device_error", "kda_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    from delta_rule_linear_gb300 import _lib
    names = _declared_functions()
    assert set(_lib.EXPORTS) == set(names), (set(_lib.EXPORTS) ^ set(names))
    for n in names:
        assert hasattr(lib, n), f"libkda.so does not export {n}"


def test_status_strings(lib):
    for code in range(10):
        s = lib.kda_status_string(code)
        assert s and isinstance(s, bytes)
    assert lib.kda_status_string(0) == b"ok"
    assert lib.kda_status_string(1234) == b"unknown status"


def test_workspace_queries(lib):
    assert lib.kda_chunk_fwd_workspace(2, 2048, 16, 128, 128, 64, 1) >= 256
    assert lib.kda_chunk_fwd_workspace(1, 64, 2, 32, 32, 16, 0) >= 256
    assert lib.kda_chunk_fwd_workspace(1, 64, 2, 48, 32, 16, 0) == 0      # unsupported dk
    assert lib.kda_chunk_fwd_workspace(1, 64, 2, 32, 32, 24, 0) == 0      # unsupported chunk
    assert lib.kda_chunk_fwd_workspace(-1, 64, 2, 32, 32, 16, 0) == 0
    assert lib.kda_chunk_fwd_workspace(1, 64, 2, 32, 32, 16, 7) == 0      # bad dtype
    assert lib.kda_varlen_fwd_workspace(16, 34816, 16, 64, 64, 64, 1) >= 256
    assert lib.kda_varlen_fwd_workspace(16, 34816, 0, 64, 64, 64, 1) == 0


def _fake(addr=0x1000):
    return ctypes.c_void_p(addr)


def _chunk(lib, **kw):
    a = dict(q=_fake(), k=_fake(), v=_fake(), beta=_fake(), decay=None, h0=None, o=_fake(),
             hT=None, B=1, T=64, H=2, dk=32, dv=32, dt=0, scale=0.0, chunk=16, l2=1,
             ws=_fake(), ws_bytes=256, stream=None)
    a.update(kw)
    return lib.kda_chunk_fwd(a["q"], a["k"], a["v"], a["beta"], a["decay"], a["h0"], a["o"],
                             a["hT"], a["B"], a["T"], a["H"], a["dk"], a["dv"], a["dt"],
                             a["scale"], a["chunk"], a["l2"], a["ws"], a["ws_bytes"], a["stream"])


def test_chunk_fwd_rejects_bad_arguments(lib):
    assert _chunk(lib, q=None) == 1                 # KDA_ERR_NULL
    assert _chunk(lib, beta=None) == 1
    assert _chunk(lib, B=-1) == 2                   # KDA_ERR_SHAPE
    assert _chunk(lib, H=0) == 2
    assert _chunk(lib, dt=5) == 3                   # KDA_ERR_DTYPE
    assert _chunk(lib, dk=48) == 4                  # KDA_ERR_UNSUPPORTED
    assert _chunk(lib, dv=256) == 4
    assert _chunk(lib, chunk=128) == 4
    assert _chunk(lib, q=_fake(0x1008)) == 5        # KDA_ERR_ALIGN
    assert _chunk(lib, beta=_fake(0x1002)) == 5
    assert _chunk(lib, ws=None) == 6                # KDA_ERR_WORKSPACE
    assert _chunk(lib, ws_bytes=8) == 6
    assert _chunk(lib, ws=_fake(0x1004)) == 5


def test_decode_rejects_bad_arguments(lib):
    def call(**kw):
        a = dict(q=_fake(), k=_fake(), v=_fake(), beta=_fake(), decay=None, state=_fake(),
                 o=_fake(), B=4, H=2, dk=64, dv=64, dt=1, scale=0.0, l2=1, stream=None)
        a.update(kw)
        return lib.kda_decode_step(a["q"], a["k"], a["v"], a["beta"], a["decay"], a["state"],
                                   a["o"], a["B"], a["H"], a["dk"], a["dv"], a["dt"], a["scale"],
                                   a["l2"], a["stream"])
    assert call(state=None) == 1
    assert call(k=None) == 1
    assert call(B=-2) == 2
    assert call(dk=96) == 4
    assert call(state=_fake(0x1010 + 4)) == 5
    assert call(B=0) == 0                           # nothing to do, no launch


def test_varlen_rejects_bad_cu_seqlens(lib):
    def call(host, N=3, total=10, **kw):
        hs = (ctypes.c_int * len(host))(*host)
        a = dict(q=_fake(), k=_fake(), v=_fake(), beta=_fake(), decay=None, cu=_fake(),
                 h0=None, o=_fake(), hT=None, H=2, dk=64, dv=64, dt=1, chunk=64, l2=1,
                 ws=_fake(), ws_bytes=256)
        a.update(kw)
        return lib.kda_varlen_fwd(a["q"], a["k"], a["v"], a["beta"], a["decay"], a["cu"],
                                  ctypes.cast(hs, ctypes.c_void_p), N, total, a["H"], a["dk"],
                                  a["dv"], a["h0"], a["o"], a["hT"], a["dt"], 0.0, a["chunk"],
                                  a["l2"], a["ws"], a["ws_bytes"], None)
    assert call([0, 4, 3, 10]) == 9                 # not monotone
    assert call([1, 4, 6, 10]) == 9                 # does not start at 0
    assert call([0, 4, 6, 9]) == 9                  # does not end at total_T
    assert call([0, 4, 6, 10], cu=None) == 1
    assert call([0, 4, 6, 10], chunk=48) == 4


def test_query_device_error_null_reads_the_builtin_array(lib):
    """ws == NULL reads the no-alloc entry point's built-in array on the current device:
    nothing recorded there (KDA_OK) with a GPU; KDA_ERR_CUDA without one (no crash)."""
    import torch
    assert lib.kda_query_device_error(None, None) == (0 if torch.cuda.is_available() else 7)


def test_python_binding_refuses_host_tensors():
    import torch
    import delta_rule_linear_gb300 as kda
    x = torch.zeros(1, 4, 1, 32)
    b = torch.zeros(1, 4, 1)
    h = torch.zeros(1, 1, 32, 32)
    with pytest.raises(ValueError):
        kda.chunk_fwd(x, x, x, b, chunk_size=16)
    for call in (lambda: kda.recurrent_fwd(x, x, x, b),
                 lambda: kda.decode_step(x[:, :1], x[:, :1], x[:, :1], b[:, :1], None, h),
                 lambda: kda.gk_recurrent_fwd(x, x, x, b, x),
                 lambda: kda.recurrent_bwd(x, x, x, b, b, h, x),
                 lambda: kda.gk_recurrent_bwd(x, x, x, b, x, h, x)):
        with pytest.raises(ValueError):
            call()


def test_diag_wait_timeout_argument_errors(lib):
    """The probe's argument checks return before any CUDA call (a dummy aligned address
    is never dereferenced)."""
    fake = ctypes.c_void_p(0x10000)
    assert lib.kda_diag_wait_timeout(None, 4096, 1000, None) == 1        # KDA_ERR_NULL
    assert lib.kda_diag_wait_timeout(fake, 100, 1000, None) == 6         # KDA_ERR_WORKSPACE
    assert lib.kda_diag_wait_timeout(ctypes.c_void_p(0x10004), 4096, 1000, None) == 5   # ALIGN
    assert lib.kda_diag_wait_timeout(fake, 4096, 0, None) == 2           # KDA_ERR_SHAPE
    assert lib.kda_diag_wait_timeout(fake, 4096, 2_000_001, None) == 2


def test_gk_entry_points_reject_bad_arguments(lib):
    """Per-key-channel decay: the same checks, plus g's 16-byte alignment."""
    def rec(**kw):
        a = dict(q=_fake(), k=_fake(), v=_fake(), beta=_fake(), g=_fake(), h0=None, o=_fake(),
                 hT=None, B=1, T=64, H=2, dk=64, dv=64, dt=1, l2=1, opt=None)
        a.update(kw)
        return lib.kda_gk_recurrent_fwd(a["q"], a["k"], a["v"], a["beta"], a["g"], a["h0"],
                                        a["o"], a["hT"], a["B"], a["T"], a["H"], a["dk"],
                                        a["dv"], a["dt"], 0.0, a["l2"], a["opt"], None)
    assert rec(q=None) == 1
    assert rec(T=-1) == 2
    assert rec(dt=9) == 3
    assert rec(dk=80) == 4
    assert rec(g=_fake(0x1004)) == 5
    assert rec(B=0) == 0                            # nothing to do, no launch

    def dec(**kw):
        a = dict(q=_fake(), k=_fake(), v=_fake(), beta=_fake(), g=None, state=_fake(),
                 o=_fake(), B=4, H=2, dk=128, dv=128, dt=1, l2=1, opt=None)
        a.update(kw)
        return lib.kda_gk_decode_step(a["q"], a["k"], a["v"], a["beta"], a["g"], a["state"],
                                      a["o"], a["B"], a["H"], a["dk"], a["dv"], a["dt"], 0.0,
                                      a["l2"], a["opt"], None)
    assert dec(state=None) == 1
    assert dec(g=_fake(0x1008)) == 5
    assert dec(dv=16) == 4
    assert dec(B=0) == 0

    def var(host, N=3, total=10, **kw):
        hs = (ctypes.c_int * len(host))(*host)
        a = dict(q=_fake(), k=_fake(), v=_fake(), beta=_fake(), g=_fake(), cu=_fake(),
                 h0=None, o=_fake(), hT=None, H=2, dk=64, dv=64, dt=1)
        a.update(kw)
        return lib.kda_gk_varlen_recurrent_fwd(a["q"], a["k"], a["v"], a["beta"], a["g"],
                                               a["cu"], ctypes.cast(hs, ctypes.c_void_p), N,
                                               total, a["H"], a["dk"], a["dv"], a["h0"], a["o"],
                                               a["hT"], a["dt"], 0.0, 1, None, None)
    assert var([0, 4, 3, 10]) == 9
    assert var([0, 4, 6, 9]) == 9
    assert var([0, 4, 6, 10], cu=None) == 1
    assert var([0, 4, 6, 10], g=_fake(0x100c)) == 5


def test_gk_chunk_entry_points_reject_bad_arguments(lib):
    def call(**kw):
        a = dict(q=_fake(), k=_fake(), v=_fake(), beta=_fake(), g=_fake(), h0=None, o=_fake(),
                 hT=None, B=1, T=64, H=2, dk=128, dv=128, dt=1, chunk=64, ws=_fake(), ws_bytes=1 << 30)
        a.update(kw)
        return lib.kda_gk_chunk_fwd(a["q"], a["k"], a["v"], a["beta"], a["g"], a["h0"], a["o"],
                                    a["hT"], a["B"], a["T"], a["H"], a["dk"], a["dv"], a["dt"], 0.0,
                                    a["chunk"], 1, None, a["ws"], a["ws_bytes"], None)
    assert call(k=None) == 1
    assert call(H=-1) == 2
    assert call(dt=4) == 3
    assert call(chunk=48) == 4
    assert call(g=_fake(0x1004)) == 5
    assert call(ws=None) == 6
    assert call(ws_bytes=300) == 6
    hs = (ctypes.c_int * 3)(0, 5, 4)
    assert lib.kda_gk_varlen_fwd(_fake(), _fake(), _fake(), _fake(), _fake(), _fake(),
                                 ctypes.cast(hs, ctypes.c_void_p), 2, 4, 2, 64, 64, None, _fake(),
                                 None, 1, 0.0, 64, 1, None, _fake(), 1 << 30, None) == 9



def _opts(**kw):
    import ctypes as ct
    from delta_rule_linear_gb300 import _lib
    o = _lib.KdaOptions(kw.get("decayed_read", 0), kw.get("A_log"), kw.get("dt_bias"),
                        kw.get("beta_sigmoid", 0), kw.get("allow_neg_eigval", 0))
    return ct.pointer(o)


def test_options_are_checked(lib):
    """kda_options: dt_bias needs A_log, A_log needs the decay (gate) array, 4-byte alignment."""
    def chunk(opt, decay=_fake()):
        return lib.kda_chunk_fwd_ex(_fake(), _fake(), _fake(), _fake(), decay, None, _fake(), None,
                                    1, 64, 2, 64, 64, 1, 0.0, 64, 1, opt, _fake(), 1 << 30, None)
    assert chunk(_opts(dt_bias=0x2000)) == 1
    assert chunk(_opts(A_log=0x2000), decay=None) == 1
    assert chunk(_opts(A_log=0x2002)) == 5
    assert chunk(_opts(A_log=0x2000, dt_bias=0x2001)) == 5

    def dec(opt, B=4):
        return lib.kda_decode_step_ex(_fake(), _fake(), _fake(), _fake(), _fake(), _fake(), _fake(),
                                      B, 2, 64, 64, 1, 0.0, 1, opt, None)
    assert dec(_opts(dt_bias=0x2000)) == 1
    assert dec(_opts(dt_bias=0x2000), B=0) == 1    # checked before the empty-batch return
    assert dec(_opts(decayed_read=1), B=0) == 0
    assert lib.kda_gk_decode_step(_fake(), _fake(), _fake(), _fake(), None, _fake(), _fake(), 4, 2,
                                  64, 64, 1, 0.0, 1, _opts(A_log=0x2000), None) == 1


def test_gate_decay_argument_errors(lib):
    assert lib.kda_gate_decay(_fake(), _fake(), None, _fake(), -1, 2, 1, None) == 2
    assert lib.kda_gate_decay(_fake(), _fake(), None, _fake(), 10, 0, 1, None) == 2
    assert lib.kda_gate_decay(None, _fake(), None, _fake(), 10, 2, 1, None) == 1
    assert lib.kda_gate_decay(_fake(), None, None, _fake(), 10, 2, 1, None) == 1
    assert lib.kda_gate_decay(_fake(0x1002), _fake(), None, _fake(), 10, 2, 1, None) == 5
    assert lib.kda_gate_decay(_fake(), _fake(), None, _fake(), 0, 2, 1, None) == 0


def test_grouped_heads_option_checked(lib):
    """v_heads_per_qk_head < 0 is a shape error; the workspace check uses the value heads."""
    import ctypes as ct
    from delta_rule_linear_gb300 import _lib

    def chunk(m, ws_bytes):
        o = _lib.KdaOptions(0, None, None, 0, 0, m)
        return lib.kda_chunk_fwd_ex(_fake(), _fake(), _fake(), _fake(), None, None, _fake(), None,
                                    1, 640, 2, 128, 128, 1, 0.0, 64, 1, ct.pointer(o), _fake(),
                                    ws_bytes, None)
    assert chunk(-2, 1 << 30) == 2
    need2 = lib.kda_chunk_fwd_workspace(1, 640, 2, 128, 128, 64, 1)
    need6 = lib.kda_chunk_fwd_workspace(1, 640, 6, 128, 128, 64, 1)
    assert need6 > need2
    assert chunk(3, need2) == 6          # three value heads per q/k head need the HV-sized workspace


def test_backward_entry_points_reject_bad_arguments(lib):
    """kda_gk_recurrent_bwd and kda_recurrent_bwd: workspace sizes, and every argument error
    returned before anything is enqueued."""
    assert lib.kda_gk_recurrent_bwd_workspace(2, 2048, 16, 128, 128) > 256
    assert lib.kda_recurrent_bwd_workspace(2, 2048, 16, 128, 128) == \
        lib.kda_gk_recurrent_bwd_workspace(2, 2048, 16, 128, 128)
    assert lib.kda_recurrent_bwd_workspace(1, 64, 2, 48, 64) == 0      # unsupported dk
    assert lib.kda_recurrent_bwd_workspace(1, 64, 0, 64, 64) == 0
    need = lib.kda_recurrent_bwd_workspace(1, 64, 2, 64, 64)

    def call(fn, **kw):
        a = dict(q=_fake(), k=_fake(), v=_fake(), beta=_fake(), dec=None, h0=None, do=_fake(),
                 dhT=None, dq=_fake(), dk_=_fake(), dv_=_fake(), db=_fake(), dd=None, dh0=None,
                 B=1, T=64, H=2, dk=64, dv=64, dt=1, l2=1, dr=0, ws=_fake(), wsb=need)
        a.update(kw)
        return fn(a["q"], a["k"], a["v"], a["beta"], a["dec"], a["h0"], a["do"], a["dhT"], a["dq"],
                  a["dk_"], a["dv_"], a["db"], a["dd"], a["dh0"], a["B"], a["T"], a["H"], a["dk"],
                  a["dv"], a["dt"], 0.0, a["l2"], a["dr"], a["ws"], a["wsb"], None)

    for fn in (lib.kda_gk_recurrent_bwd, lib.kda_recurrent_bwd):
        assert call(fn, q=None) == 1
        assert call(fn, dq=None) == 1
        assert call(fn, T=-1) == 2
        assert call(fn, dt=9) == 3
        assert call(fn, dk=80) == 4
        assert call(fn, dd=_fake(0x1002)) == 5
        assert call(fn, dh0=_fake(0x1004)) == 5
        assert call(fn, ws=None) == 6
        assert call(fn, wsb=need - 1) == 6
        assert call(fn, ws=_fake(0x1008)) == 5
        assert call(fn, B=0) == 0                   # nothing to do, no launch
    assert call(lib.kda_gk_recurrent_bwd, dec=_fake(0x1004)) == 5   # g: 16-byte aligned
    assert call(lib.kda_recurrent_bwd, dec=_fake(0x1002)) == 5      # decay: 4-byte aligned


def test_chunk_bwd_rejects_bad_arguments(lib):
    """kda_chunk_bwd (the chunked backward on the tensor cores): workspace sizes, and every
    argument error returned before anything is enqueued."""
    need = lib.kda_chunk_bwd_workspace(1, 64, 2, 64, 64)
    assert need > 256
    assert lib.kda_chunk_bwd_workspace(2, 2048, 16, 128, 128) > lib.kda_chunk_bwd_workspace(1, 64, 2, 128, 128)
    assert lib.kda_chunk_bwd_workspace(1, 64, 2, 64, 128) == 0      # dk != dv
    assert lib.kda_chunk_bwd_workspace(1, 64, 2, 96, 96) == 0       # head dim not 64 / 128
    assert lib.kda_chunk_bwd_workspace(1, 64, 0, 64, 64) == 0
    assert lib.kda_chunk_bwd_workspace(-1, 64, 2, 64, 64) == 0
    assert lib.kda_chunk_bwd_workspace(0, 64, 2, 64, 64) == 256     # header only

    def call(**kw):
        a = dict(q=_fake(), k=_fake(), v=_fake(), beta=_fake(), dec=None, h0=None, do=_fake(),
                 dhT=None, dq=_fake(), dk_=_fake(), dv_=_fake(), db=_fake(), dd=None, dh0=None,
                 B=1, T=64, H=2, dk=64, dv=64, dt=1, l2=1, dr=0, ws=_fake(), wsb=need)
        a.update(kw)
        return lib.kda_chunk_bwd(a["q"], a["k"], a["v"], a["beta"], a["dec"], a["h0"], a["do"], a["dhT"],
                                 a["dq"], a["dk_"], a["dv_"], a["db"], a["dd"], a["dh0"], a["B"], a["T"],
                                 a["H"], a["dk"], a["dv"], a["dt"], 0.0, a["l2"], a["dr"], a["ws"], a["wsb"],
                                 None)

    assert call(q=None) == 1
    assert call(do=None) == 1
    assert call(dq=None) == 1
    assert call(dv_=None) == 1
    assert call(T=-1) == 2
    assert call(dt=9) == 3
    assert call(dt=0) == 4                      # fp32 inputs: not on this path
    assert call(dk=96, dv=96) == 4
    assert call(dk=64, dv=128) == 4
    assert call(dd=_fake(0x1002)) == 5          # ddecay: 4-byte aligned
    assert call(dh0=_fake(0x1004)) == 5         # dh0: 16-byte aligned
    assert call(ws=None) == 6
    assert call(wsb=need - 1) == 6
    assert call(ws=_fake(0x1008)) == 5
    assert call(B=0) == 0                       # nothing to do, no launch


def test_gk_chunk_bwd_rejects_bad_arguments(lib):
    """kda_gk_chunk_bwd (the per-channel chunked backward): workspace sizes, and every argument
    error returned before anything is enqueued."""
    need = lib.kda_gk_chunk_bwd_workspace(1, 64, 2, 64, 64)
    assert need > 256
    assert lib.kda_gk_chunk_bwd_workspace(2, 2048, 16, 128, 128) > lib.kda_gk_chunk_bwd_workspace(1, 64, 2, 128, 128)
    assert lib.kda_gk_chunk_bwd_workspace(1, 64, 2, 64, 128) == 0      # dk != dv
    assert lib.kda_gk_chunk_bwd_workspace(1, 64, 2, 96, 96) == 0       # head dim not 64 / 128
    assert lib.kda_gk_chunk_bwd_workspace(1, 64, 0, 64, 64) == 0
    assert lib.kda_gk_chunk_bwd_workspace(0, 64, 2, 64, 64) == 256     # header only

    def call(**kw):
        a = dict(q=_fake(), k=_fake(), v=_fake(), beta=_fake(), g=_fake(), h0=None, do=_fake(),
                 dhT=None, dq=_fake(), dk_=_fake(), dv_=_fake(), db=_fake(), dg=_fake(), dh0=None,
                 B=1, T=64, H=2, dk=64, dv=64, dt=1, l2=1, dr=0, ws=_fake(), wsb=need)
        a.update(kw)
        return lib.kda_gk_chunk_bwd(a["q"], a["k"], a["v"], a["beta"], a["g"], a["h0"], a["do"], a["dhT"],
                                    a["dq"], a["dk_"], a["dv_"], a["db"], a["dg"], a["dh0"], a["B"], a["T"],
                                    a["H"], a["dk"], a["dv"], a["dt"], 0.0, a["l2"], a["dr"], a["ws"], a["wsb"],
                                    None)

    assert call(q=None) == 1
    assert call(do=None) == 1
    assert call(dk_=None) == 1
    assert call(db=None) == 1
    assert call(T=-1) == 2
    assert call(dt=9) == 3
    assert call(dt=0) == 4                      # fp32 inputs: not on this path
    assert call(dk=96, dv=96) == 4
    assert call(dk=64, dv=128) == 4
    assert call(g=_fake(0x1004)) == 5           # g: 16-byte aligned
    assert call(dg=_fake(0x1002)) == 5          # dg: 4-byte aligned
    assert call(dh0=_fake(0x1004)) == 5         # dh0: 16-byte aligned
    assert call(ws=None) == 6
    assert call(wsb=need - 1) == 6
    assert call(ws=_fake(0x1008)) == 5
    assert call(B=0) == 0                       # nothing to do, no launch
