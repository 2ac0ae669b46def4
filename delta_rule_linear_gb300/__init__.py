"""Delta-rule linear attention with per-token decay on GB300 (sm_103a).

Forward of the recurrence on ejkernel ``kernels._xla.kernel_delta_attention._interface``
(``kda()``, "The core recurrence"):

    h_t = exp(decay_t) h_{t-1} + k_t (beta_t (v_t - h_{t-1}^T k_t))^T,   o_t = h_t^T (scale q_t)

served by a C-ABI CUDA library (``libkda.so``, declared in ``include/kda.h``):
chunked prefill, recurrent prefill, single-token decode and packed varlen prefill;
and the per-key-channel decay of TileOPs KDAFwdOp (g [B,T,H,dk], ``gk_*``); gradients of
both recurrences (``recurrent_bwd``, ``gk_recurrent_bwd``; by chunks on the tensor cores,
``chunk_bwd``, ``gk_chunk_bwd``).
This package is the thin binding; all compute runs in the library's kernels.
"""
from ._lib import (KdaError, chunk_bwd, chunk_fwd, chunk_fwd_noalloc, decode_step, diag_wait_timeout,  # noqa: F401
                   gate_decay, gk_chunk_bwd, gk_chunk_fwd, gk_decode_step, gk_recurrent_bwd, gk_recurrent_fwd, load,
                   query_device_error, recurrent_bwd, recurrent_fwd, varlen_fwd)

__all__ = ["kda", "chunk_fwd", "chunk_fwd_noalloc", "recurrent_fwd", "recurrent_bwd", "chunk_bwd", "decode_step",
           "varlen_fwd", "gk_chunk_fwd", "gk_recurrent_fwd", "gk_recurrent_bwd", "gk_chunk_bwd", "gk_decode_step",
           "gate_decay",
           "query_device_error",
           "diag_wait_timeout", "load", "KdaError"]


def kda(query, key, value, beta, decay=None, *, softmax_scale=None, chunk_size=64,
        initial_state=None, use_qk_l2norm=True, use_chunked=True):
    """Functional form with the argument names of ejkernel ``kda()`` ("Parameters").

    query, key [B,T,H,dk]; value [B,T,H,dv] (bf16 or fp32, CUDA); beta, decay [B,T,H] fp32;
    initial_state [B,H,dk,dv] fp32.  Returns (output [B,T,H,dv], final_state [B,H,dk,dv]).
    ``use_chunked=False`` runs the token-by-token kernel (the recurrent mode).
    """
    if use_chunked:
        return chunk_fwd(query, key, value, beta, decay, initial_state, scale=softmax_scale,
                         chunk_size=chunk_size, use_qk_l2norm=use_qk_l2norm)
    return recurrent_fwd(query, key, value, beta, decay, initial_state, scale=softmax_scale,
                         use_qk_l2norm=use_qk_l2norm)
