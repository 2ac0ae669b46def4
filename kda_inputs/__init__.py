"""Seeded synthetic inputs for the delta-rule linear-attention forward.

This module is the one thing the CPU oracle and the GPU path share: it draws the
inputs and nothing else (none of the method's arithmetic lives here).  Every
array is numpy float32 whose values are exactly representable in the declared
compute dtype: bf16 workloads are rounded to bf16 (round-to-nearest-even) here,
so the GPU copy (a bf16 tensor) and the oracle copy (widened to float64) hold
identical numbers.

Draws use numpy's PCG64 generator, which gives the same stream on x86_64 and
aarch64.  Order inside one workload: sequence lengths (varlen only), q, k, v,
beta logits, decay normals, initial state.  Decode draws the initial state from
the base seed and each step's token from the seed pair (seed, step + 1).

The five workloads follow the shapes and distributions of the five benchmark
configurations:

  1 tiny      fp32, B=1 T=64 H=2 d=32, chunk 16, zero state, l2 on,
              q,k,v ~ N(0,1), beta = sigmoid(N(0,1)), decay = -0.01|N(0,1)|
  2 train     bf16, B=2 T=2048 H=16 d=128, chunk 64, zero state, l2 on,
              decay = -0.05|N(0,1)|
  3 long      bf16, B=1 T=32768 H=32 d=128, chunk 64, state ~ N(0, 0.02^2),
              decay = -softplus(N(-4,1)), l2 on
  4 decode    bf16, B=256 H=32 d=128, 128 single-token steps, state ~ N(0,0.02^2),
              decay = -0.01|N(0,1)| per step, l2 on
  5 varlen    bf16, 16 sequences of length U[256, 4096], H=16 d=64, chunk 64,
              decay None, zero state per sequence, l2 on

Per-key-channel decay (TileOPs KDAFwdOp, g [B,T,H,K]) draws, after q, k, v and the
beta logits, g = -gate_scale * U[0,1) per token and key channel: the gate regimes of
the kda-neuron-kernels README ("Functional warning": scales 0.01, 0.3, 2.0; its
examples draw -rand * 0.01).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

__all__ = ["Workload", "WORKLOADS", "round_to_bf16", "make_prefill", "make_varlen",
           "make_decode_state", "make_decode_step", "make_custom", "make_gk",
           "make_gk_decode_step", "make_gate_params"]


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str            # "prefill" | "decode" | "varlen"
    dtype: str           # "f32" | "bf16"   (q, k, v, o; beta/decay/state are fp32)
    B: int
    T: int
    H: int
    dk: int
    dv: int
    chunk: int
    use_l2: bool
    decay: str           # "small" | "train" | "long" | "none"
    h0: str              # "zero" | "normal002"
    steps: int = 1       # decode steps
    nseq: int = 0        # varlen sequences
    len_range: tuple = field(default=(0, 0))


WORKLOADS = {
    1: Workload("tiny fp32 prefill B=1 T=64 H=2 d=32", "prefill", "f32", 1, 64, 2, 32, 32, 16,
                True, "small", "zero"),
    2: Workload("training-shape prefill B=2 T=2048 H=16 d=128", "prefill", "bf16", 2, 2048, 16,
                128, 128, 64, True, "train", "zero"),
    3: Workload("long-sequence prefill B=1 T=32768 H=32 d=128 carried state", "prefill", "bf16",
                1, 32768, 32, 128, 128, 64, True, "long", "normal002"),
    4: Workload("batched decode B=256 H=32 d=128 x128 steps", "decode", "bf16", 256, 1, 32, 128,
                128, 64, True, "small", "normal002", steps=128),
    5: Workload("ungated packed varlen 16 seqs U[256,4096] H=16 d=64", "varlen", "bf16", 1, 0, 16,
                64, 64, 64, True, "none", "zero", nseq=16, len_range=(256, 4096)),
}


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """float32 -> float32 holding the nearest bf16 value (ties to even)."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) & 0xFFFF0000
    return b.astype(np.uint32).view(np.float32)


def _cast(x: np.ndarray, dtype: str) -> np.ndarray:
    x = x.astype(np.float32, copy=False)
    return round_to_bf16(x) if dtype == "bf16" else x


def _sigmoid(x):
    return (1.0 / (1.0 + np.exp(-x.astype(np.float64)))).astype(np.float32)


def _decay(rng, shape, kind):
    if kind == "none":
        return None
    z = rng.standard_normal(shape, dtype=np.float32)
    if kind == "small":
        return (-0.01 * np.abs(z)).astype(np.float32)
    if kind == "train":
        return (-0.05 * np.abs(z)).astype(np.float32)
    if kind == "long":
        x = z.astype(np.float64) - 4.0
        return (-np.logaddexp(0.0, x)).astype(np.float32)  # -softplus(N(-4, 1))
    if kind == "strong":   # about -1.8 per token: a 64-token chunk spans far more than e^-80
        return (-(1.0 + np.abs(z))).astype(np.float32)
    if kind == "mixed":    # along T, 64-token blocks alternate between "train" and "strong"
        t = np.arange(shape[1]).reshape((1, -1) + (1,) * (len(shape) - 2))
        strong = (t // 64) % 2 == 1
        return np.where(strong, -(1.0 + np.abs(z)), -0.05 * np.abs(z)).astype(np.float32)
    raise ValueError(kind)


def _h0(rng, shape, kind):
    if kind == "zero":
        return None
    if kind == "normal002":
        return (0.02 * rng.standard_normal(shape, dtype=np.float32)).astype(np.float32)
    raise ValueError(kind)


def make_custom(B, T, H, dk, dv, *, dtype="bf16", decay="small", h0="zero", seed=0,
                qkv_scale=1.0):
    """Equal-length inputs of any shape, same recipe as the named workloads."""
    rng = np.random.Generator(np.random.PCG64(seed))
    q = _cast(qkv_scale * rng.standard_normal((B, T, H, dk), dtype=np.float32), dtype)
    k = _cast(qkv_scale * rng.standard_normal((B, T, H, dk), dtype=np.float32), dtype)
    v = _cast(qkv_scale * rng.standard_normal((B, T, H, dv), dtype=np.float32), dtype)
    beta = _sigmoid(rng.standard_normal((B, T, H), dtype=np.float32))
    dec = _decay(rng, (B, T, H), decay)
    st = _h0(rng, (B, H, dk, dv), h0)
    return dict(q=q, k=k, v=v, beta=beta, decay=dec, h0=st)


def make_prefill(wl: Workload, seed: int = 0):
    assert wl.kind == "prefill"
    return make_custom(wl.B, wl.T, wl.H, wl.dk, wl.dv, dtype=wl.dtype, decay=wl.decay,
                       h0=wl.h0, seed=seed)


def make_varlen(wl: Workload, seed: int = 0, lengths=None):
    """Packed inputs: token arrays [1, total, H, D], cu_seqlens int32 [N+1]."""
    rng = np.random.Generator(np.random.PCG64(seed))
    if lengths is None:
        lo, hi = wl.len_range
        lengths = rng.integers(lo, hi + 1, size=wl.nseq)
    lengths = np.asarray(lengths, dtype=np.int64)
    cu = np.zeros(len(lengths) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lengths)
    total = int(cu[-1])
    H, dk, dv = wl.H, wl.dk, wl.dv
    q = _cast(rng.standard_normal((1, total, H, dk), dtype=np.float32), wl.dtype)
    k = _cast(rng.standard_normal((1, total, H, dk), dtype=np.float32), wl.dtype)
    v = _cast(rng.standard_normal((1, total, H, dv), dtype=np.float32), wl.dtype)
    beta = _sigmoid(rng.standard_normal((1, total, H), dtype=np.float32))
    dec = _decay(rng, (1, total, H), wl.decay)
    st = _h0(rng, (len(lengths), H, dk, dv), wl.h0)
    return dict(q=q, k=k, v=v, beta=beta, decay=dec, h0=st, cu_seqlens=cu)


def make_decode_state(wl: Workload, seed: int = 0):
    rng = np.random.Generator(np.random.PCG64(seed))
    st = _h0(rng, (wl.B, wl.H, wl.dk, wl.dv), wl.h0)
    if st is None:
        st = np.zeros((wl.B, wl.H, wl.dk, wl.dv), dtype=np.float32)
    return st


def make_decode_step(wl: Workload, step: int, seed: int = 0):
    """One token per sequence: q, k [B,1,H,dk], v [B,1,H,dv], beta/decay [B,1,H]."""
    rng = np.random.Generator(np.random.PCG64([seed, step + 1]))
    B, H = wl.B, wl.H
    q = _cast(rng.standard_normal((B, 1, H, wl.dk), dtype=np.float32), wl.dtype)
    k = _cast(rng.standard_normal((B, 1, H, wl.dk), dtype=np.float32), wl.dtype)
    v = _cast(rng.standard_normal((B, 1, H, wl.dv), dtype=np.float32), wl.dtype)
    beta = _sigmoid(rng.standard_normal((B, 1, H), dtype=np.float32))
    dec = _decay(rng, (B, 1, H), wl.decay)
    return dict(q=q, k=k, v=v, beta=beta, decay=dec)


def make_gk(B, T, H, dk, dv, *, dtype="bf16", gate_scale=0.01, h0="zero", seed=0,
            lengths=None):
    """Inputs with one log decay per key channel: g [B,T,H,dk] = -gate_scale * U[0,1).

    With ``lengths`` the batch is packed: token arrays [1, total, H, .] and
    ``cu_seqlens`` int32 [N+1]; the state then has N rows.  Without it, B sequences
    of T tokens.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    out = {}
    if lengths is not None:
        lengths = np.asarray(lengths, dtype=np.int64)
        cu = np.zeros(len(lengths) + 1, dtype=np.int32)
        cu[1:] = np.cumsum(lengths)
        out["cu_seqlens"] = cu
        B, T, nstate = 1, int(cu[-1]), len(lengths)
    else:
        nstate = B
    q = _cast(rng.standard_normal((B, T, H, dk), dtype=np.float32), dtype)
    k = _cast(rng.standard_normal((B, T, H, dk), dtype=np.float32), dtype)
    v = _cast(rng.standard_normal((B, T, H, dv), dtype=np.float32), dtype)
    beta = _sigmoid(rng.standard_normal((B, T, H), dtype=np.float32))
    g = (-gate_scale * rng.random((B, T, H, dk), dtype=np.float32)).astype(np.float32)
    st = _h0(rng, (nstate, H, dk, dv), h0)
    out.update(q=q, k=k, v=v, beta=beta, g=g, h0=st)
    return out


def make_gk_decode_step(B, H, dk, dv, step, *, dtype="bf16", gate_scale=0.01, seed=0):
    """One token per sequence with per-channel decay: q, k, g [B,1,H,dk], v [B,1,H,dv]."""
    rng = np.random.Generator(np.random.PCG64([seed, step + 1]))
    q = _cast(rng.standard_normal((B, 1, H, dk), dtype=np.float32), dtype)
    k = _cast(rng.standard_normal((B, 1, H, dk), dtype=np.float32), dtype)
    v = _cast(rng.standard_normal((B, 1, H, dv), dtype=np.float32), dtype)
    beta = _sigmoid(rng.standard_normal((B, 1, H), dtype=np.float32))
    g = (-gate_scale * rng.random((B, 1, H, dk), dtype=np.float32)).astype(np.float32)
    return dict(q=q, k=k, v=v, beta=beta, g=g)


def make_gate_params(shape, H, K=1, seed=0):
    """Raw gates for the in-kernel decay (ejkernel kda_decay; TileOPs use_gate_in_kernel), drawn
    the usual state-space way: gate ~ N(0, 1) with the given shape (trailing dims [H] or [H, K]),
    A = exp(A_log) ~ U[1, 16), and dt_bias the inverse softplus of dt = exp(U[ln 1e-3, ln 1e-1)),
    [H] or [H, K].  Returns float32 (gate, A_log, dt_bias)."""
    rng = np.random.Generator(np.random.PCG64([seed, 99]))
    gate = rng.standard_normal(shape, dtype=np.float32)
    A_log = np.log(rng.uniform(1.0, 16.0, size=H)).astype(np.float32)
    dt = np.exp(rng.uniform(np.log(1e-3), np.log(1e-1), size=(H,) if K == 1 else (H, K)))
    dt_bias = np.log(np.expm1(dt)).astype(np.float32)
    return gate, A_log, dt_bias
