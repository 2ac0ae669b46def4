"""CPU fp64 oracle for the delta-rule linear-attention forward -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The GPU library never links, imports or
calls it, and it shares no code with the GPU path.

It restates page 1 (ejkernel ``kernels._xla.kernel_delta_attention._interface``,
``kda()``, "The core recurrence") as a per-token double-precision scan, plus the
chunked WY form derived from that recurrence (``kda()`` "Algorithm Modes":
chunked = parallel inside a chunk, sequential across chunks), plus the packed
variable-length layout of TileOPs "Linear Attention Operators", DeltaNetFwdOp
(``cu_seqlens``, one state per sequence), plus the per-key-channel decay of
KDAFwdOp on the same page (``forward_gk``: g [.., dk], either decay placement).
The arithmetic lives in ``kda_oracle.c``; this module only builds it with gcc
and marshals numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libkda_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``kda_oracle.c`` into ``oracle/_build/libkda_oracle.so`` (gcc, -O2, no fast-math)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
           "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I = ctypes.c_int
            D = ctypes.c_double
            lib.kda_oracle_forward.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I,
                                               D, I, I, I, P, I, I]
            lib.kda_oracle_forward.restype = I
            lib.kda_oracle_varlen.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I,
                                              D, I, I, I, P, I, I]
            lib.kda_oracle_varlen.restype = I
            lib.kda_oracle_gk.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, I,
                                          D, I, I, I, I, P, I, I]
            lib.kda_oracle_gk.restype = I
            L = ctypes.c_long
            lib.kda_oracle_gate_decay.argtypes = [P, P, P, P, L, I, I]
            lib.kda_oracle_gate_decay.restype = None
            lib.kda_oracle_beta.argtypes = [P, P, L, I]
            lib.kda_oracle_beta.restype = None
            lib.kda_oracle_threads.argtypes = []
            lib.kda_oracle_threads.restype = I
            _lib = lib
    return _lib


def threads_available() -> int:
    """Host threads the oracle uses by default (online CPU count)."""
    return int(_load().kda_oracle_threads())


def _f32(x):
    if x is None:
        return None
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    return a


def _f64(x):
    if x is None:
        return None
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def forward(q, k, v, beta, decay=None, h0=None, *, scale=None, use_l2=True,
            chunk=None, heads=None, threads=0, return_threads=False):
    """fp64 forward of an equal-length batch.

    q, k: [B,T,H,dk]; v: [B,T,H,dv]; beta, decay: [B,T,H]; h0: [B,H,dk,dv] or None.
    ``chunk=None`` runs the recurrent scan; an integer runs the chunked WY form.
    ``heads`` restricts the computation to the listed flat indices b*H+h
    (the outputs of the other heads are NaN).  Returns (o [B,T,H,dv], hT [B,H,dk,dv]).
    """
    q, k, v, beta, decay = _f32(q), _f32(k), _f32(v), _f32(beta), _f32(decay)
    h0 = _f64(h0)
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    assert k.shape == q.shape and v.shape[:3] == q.shape[:3]
    assert beta.shape == (B, T, H)
    assert decay is None or decay.shape == (B, T, H)
    assert h0 is None or h0.shape == (B, H, dk, dv)
    o = np.full((B, T, H, dv), np.nan, dtype=np.float64)
    hT = np.full((B, H, dk, dv), np.nan, dtype=np.float64)
    bh = None if heads is None else np.ascontiguousarray(np.asarray(heads, dtype=np.int32))
    rc = _load().kda_oracle_forward(
        _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(decay), _ptr(h0), _ptr(o), _ptr(hT),
        B, T, H, dk, dv, float(scale) if scale else 0.0, int(bool(use_l2)),
        0 if chunk is None else 1, int(chunk or 0),
        _ptr(bh), 0 if bh is None else int(bh.size), int(threads))
    if rc < 0:
        raise ValueError(f"oracle rejected the arguments (code {rc})")
    return (o, hT, rc) if return_threads else (o, hT)


def varlen(q, k, v, beta, cu_seqlens, decay=None, h0=None, *, scale=None, use_l2=True,
           chunk=None, pairs=None, threads=0, return_threads=False):
    """fp64 forward of a packed variable-length batch.

    q, k: [1,total,H,dk]; v: [1,total,H,dv]; beta, decay: [1,total,H];
    cu_seqlens: [N+1] int prefix offsets; h0: [N,H,dk,dv] or None.
    ``pairs`` restricts to flat indices n*H+h.  Returns (o [1,total,H,dv], hT [N,H,dk,dv]).
    """
    q, k, v, beta, decay = _f32(q), _f32(k), _f32(v), _f32(beta), _f32(decay)
    h0 = _f64(h0)
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    _, total, H, dk = q.shape
    dv = v.shape[-1]
    N = int(cu.size) - 1
    assert int(cu[-1]) == total and int(cu[0]) == 0
    o = np.full((1, total, H, dv), np.nan, dtype=np.float64)
    hT = np.full((N, H, dk, dv), np.nan, dtype=np.float64)
    nh = None if pairs is None else np.ascontiguousarray(np.asarray(pairs, dtype=np.int32))
    rc = _load().kda_oracle_varlen(
        _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(decay), _ptr(h0), _ptr(o), _ptr(hT),
        _ptr(cu), N, H, dk, dv, float(scale) if scale else 0.0, int(bool(use_l2)),
        0 if chunk is None else 1, int(chunk or 0),
        _ptr(nh), 0 if nh is None else int(nh.size), int(threads))
    if rc < 0:
        raise ValueError(f"oracle rejected the arguments (code {rc})")
    return (o, hT, rc) if return_threads else (o, hT)


def decode_steps(steps, h0, *, scale=None, use_l2=True, heads=None, threads=0):
    """Repeated single-token steps carried in fp64 (P1 "Algorithm Modes": single-step).

    ``steps`` is a sequence of dicts with q, k [B,1,H,dk], v [B,1,H,dv], beta and
    decay [B,1,H].  The state stays float64 between steps.  Returns the list of
    per-step outputs and the final state.
    """
    h = _f64(h0)
    outs = []
    for st in steps:
        o, h_new = forward(st["q"], st["k"], st["v"], st["beta"], st.get("decay"), h,
                           scale=scale, use_l2=use_l2, heads=heads, threads=threads)
        if heads is not None:
            keep = np.isnan(h_new)
            h_new[keep] = h[keep]
        h = h_new
        outs.append(o)
    return outs, h


def forward_gk(q, k, v, beta, g=None, h0=None, *, cu_seqlens=None, scale=None, use_l2=True,
               decayed_read=False, chunk=None, heads=None, threads=0):
    """fp64 forward with one log decay per key channel (TileOPs KDAFwdOp).

    Equal length: q, k, g [B,T,H,dk]; v [B,T,H,dv]; beta [B,T,H]; h0 [B,H,dk,dv].
    Packed (``cu_seqlens`` [N+1] given): the token arrays have B == 1 and h0 is
    [N,H,dk,dv].  ``decayed_read`` selects where the delta term reads the memory
    (False: h_{t-1} as in kda()'s printed recurrence; True: diag(exp g_t) h_{t-1},
    the gated delta rule).  ``chunk=None`` runs the recurrent scan, an integer
    the chunked form.  ``heads`` restricts to flat indices n*H+h (others NaN).
    Returns (o, hT).
    """
    q, k, v, beta, g = _f32(q), _f32(k), _f32(v), _f32(beta), _f32(g)
    h0 = _f64(h0)
    Bq, T, H, dk = q.shape
    dv = v.shape[-1]
    assert k.shape == q.shape and v.shape[:3] == q.shape[:3]
    assert beta.shape == (Bq, T, H)
    assert g is None or g.shape == q.shape
    cu = None
    if cu_seqlens is not None:
        cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
        assert Bq == 1 and int(cu[0]) == 0 and int(cu[-1]) == T
        N = int(cu.size) - 1
    else:
        N = Bq
    assert h0 is None or h0.shape == (N, H, dk, dv)
    o = np.full((Bq, T, H, dv), np.nan, dtype=np.float64)
    hT = np.full((N, H, dk, dv), np.nan, dtype=np.float64)
    lst = None if heads is None else np.ascontiguousarray(np.asarray(heads, dtype=np.int32))
    rc = _load().kda_oracle_gk(
        _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g), _ptr(h0), _ptr(o), _ptr(hT), _ptr(cu),
        N, T, H, dk, dv, float(scale) if scale else 0.0, int(bool(use_l2)),
        int(bool(decayed_read)), 0 if chunk is None else 1, int(chunk or 0),
        _ptr(lst), 0 if lst is None else int(lst.size), int(threads))
    if rc < 0:
        raise ValueError(f"oracle rejected the arguments (code {rc})")
    return o, hT


def gate_decay(gate, A_log, dt_bias=None):
    """fp64 kda_decay (ejkernel kernel_delta_attention, kda_decay): -exp(A_log) softplus(gate +
    dt_bias).  gate [..., H] (one decay per head; A_log, dt_bias [H]) or [..., H, K] (one per key
    channel; A_log [H], dt_bias [H, K]).  Returns float64 with gate's shape."""
    gate = _f32(gate)
    A_log = _f32(A_log)
    H = A_log.shape[0]
    if gate.shape[-1] == H and (dt_bias is None or np.asarray(dt_bias).ndim == 1):
        K = 1
    else:
        K = gate.shape[-1]
        assert gate.shape[-2] == H
    dt_bias = _f32(dt_bias)
    assert dt_bias is None or dt_bias.size == H * K
    out = np.empty(gate.shape, dtype=np.float64)
    rows = gate.size // (H * K)
    _load().kda_oracle_gate_decay(_ptr(gate), _ptr(A_log), _ptr(dt_bias), _ptr(out), rows, H, K)
    return out


def beta_transform(x, allow_neg_eigval=False):
    """fp64 beta from logits (TileOPs GDNFwdOp / KDAFwdOp use_beta_sigmoid_in_kernel):
    sigmoid(x), or 2 sigmoid(x) with allow_neg_eigval."""
    x = _f32(x)
    out = np.empty(x.shape, dtype=np.float64)
    _load().kda_oracle_beta(_ptr(x), _ptr(out), x.size, int(bool(allow_neg_eigval)))
    return out
