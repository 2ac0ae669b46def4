"""ctypes binding of libkda.so (include/kda.h).  Argument marshalling only.

Every compute step runs in the library's CUDA kernels; PyTorch is used here for
device memory (output, state and workspace tensors) and for the current stream.
There is no CPU fallback: a missing library raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libkda.so")

KDA_F32, KDA_BF16 = 0, 1
STATUS = {
    0: "KDA_OK", 1: "KDA_ERR_NULL", 2: "KDA_ERR_SHAPE", 3: "KDA_ERR_DTYPE",
    4: "KDA_ERR_UNSUPPORTED", 5: "KDA_ERR_ALIGN", 6: "KDA_ERR_WORKSPACE", 7: "KDA_ERR_CUDA",
    8: "KDA_ERR_DEVICE_TIMEOUT", 9: "KDA_ERR_INDEX",
}
# Every symbol include/kda.h declares.
EXPORTS = ("kda_status_string", "kda_version", "kda_chunk_fwd_workspace", "kda_chunk_fwd",
           "kda_chunk_fwd_noalloc", "kda_recurrent_fwd", "kda_decode_step",
           "kda_varlen_fwd_workspace", "kda_varlen_fwd", "kda_chunk_fwd_ex", "kda_varlen_fwd_ex",
           "kda_recurrent_fwd_ex", "kda_decode_step_ex", "kda_gate_decay",
           "kda_gk_chunk_fwd", "kda_gk_varlen_fwd", "kda_gk_recurrent_fwd",
           "kda_gk_recurrent_bwd_workspace", "kda_gk_recurrent_bwd",
           "kda_recurrent_bwd_workspace", "kda_recurrent_bwd", "kda_chunk_bwd_workspace", "kda_chunk_bwd",
           "kda_gk_chunk_bwd_workspace", "kda_gk_chunk_bwd",
           "kda_gk_varlen_recurrent_fwd", "kda_gk_decode_step", "kda_query_device_error",
           "kda_diag_wait_timeout")


class KdaOptions(ctypes.Structure):
    """struct kda_options of include/kda.h."""
    _fields_ = [("decayed_read", ctypes.c_int), ("A_log", ctypes.c_void_p),
                ("dt_bias", ctypes.c_void_p), ("beta_sigmoid", ctypes.c_int),
                ("allow_neg_eigval", ctypes.c_int), ("v_heads_per_qk_head", ctypes.c_int),
                ("state_v_first", ctypes.c_int)]


def make_options(decayed_read=False, A_log=None, dt_bias=None, beta_sigmoid=False,
                 allow_neg_eigval=False, v_heads_per_qk_head=1, state_v_first=False):
    """A KdaOptions pointer (or None when every option is off).  A_log [HV] and dt_bias
    ([HV] for a per-head decay, [HV, dk] for g) are fp32 CUDA tensors; the caller keeps them
    alive for the call."""
    if not (decayed_read or A_log is not None or dt_bias is not None or beta_sigmoid or
            v_heads_per_qk_head > 1 or state_v_first):
        return None
    for t, name in ((A_log, "A_log"), (dt_bias, "dt_bias")):
        if t is not None and (not t.is_cuda or t.dtype != torch.float32 or not t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous float32 CUDA tensor")
    o = KdaOptions(int(bool(decayed_read)), None if A_log is None else A_log.data_ptr(),
                   None if dt_bias is None else dt_bias.data_ptr(), int(bool(beta_sigmoid)),
                   int(bool(allow_neg_eigval)), int(v_heads_per_qk_head), int(bool(state_v_first)))
    return ctypes.pointer(o)


class KdaError(RuntimeError):
    def __init__(self, code: int, where: str, lib=None):
        msg = STATUS.get(code, str(code))
        if lib is not None:
            msg += ": " + lib.kda_status_string(code).decode()
        super().__init__(f"{where}: {msg}")
        self.code = code


_lock = threading.Lock()
_lib = None


def load(path: str | None = None):
    """Load libkda.so (built in-tree by ``delta_rule_linear_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(
                f"libkda.so not found at {p}: build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'`")
        lib = ctypes.CDLL(p)
        P, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.kda_status_string.argtypes = [I]
        lib.kda_status_string.restype = ctypes.c_char_p
        lib.kda_version.argtypes = []
        lib.kda_version.restype = I
        lib.kda_chunk_fwd_workspace.argtypes = [I, I, I, I, I, I, I]
        lib.kda_chunk_fwd_workspace.restype = Z
        lib.kda_varlen_fwd_workspace.argtypes = [I, I, I, I, I, I, I]
        lib.kda_varlen_fwd_workspace.restype = Z
        lib.kda_chunk_fwd.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, I, F, I, I, P, Z, P]
        lib.kda_chunk_fwd.restype = I
        lib.kda_chunk_fwd_noalloc.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, I, F, I, I, P]
        lib.kda_chunk_fwd_noalloc.restype = I
        lib.kda_recurrent_fwd.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, I, F, I, P]
        lib.kda_recurrent_fwd.restype = I
        lib.kda_decode_step.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, F, I, P]
        lib.kda_decode_step.restype = I
        lib.kda_varlen_fwd.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, P, P, P, I, F, I, I,
                                       P, Z, P]
        lib.kda_varlen_fwd.restype = I
        O = ctypes.POINTER(KdaOptions)
        lib.kda_chunk_fwd_ex.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, I, F, I, I, O, P, Z, P]
        lib.kda_chunk_fwd_ex.restype = I
        lib.kda_varlen_fwd_ex.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, P, P, P, I, F, I, I,
                                          O, P, Z, P]
        lib.kda_varlen_fwd_ex.restype = I
        lib.kda_recurrent_fwd_ex.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, I, F, I, O, P]
        lib.kda_recurrent_fwd_ex.restype = I
        lib.kda_decode_step_ex.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, F, I, O, P]
        lib.kda_decode_step_ex.restype = I
        lib.kda_gk_recurrent_bwd_workspace.argtypes = [I, I, I, I, I]
        lib.kda_gk_recurrent_bwd_workspace.restype = Z
        lib.kda_gk_recurrent_bwd.argtypes = [P, P, P, P, P, P, P, P, P, P, P, P, P, P, I, I, I, I, I,
                                             I, F, I, I, P, Z, P]
        lib.kda_gk_recurrent_bwd.restype = I
        lib.kda_recurrent_bwd_workspace.argtypes = [I, I, I, I, I]
        lib.kda_recurrent_bwd_workspace.restype = Z
        lib.kda_recurrent_bwd.argtypes = [P, P, P, P, P, P, P, P, P, P, P, P, P, P, I, I, I, I, I,
                                          I, F, I, I, P, Z, P]
        lib.kda_recurrent_bwd.restype = I
        lib.kda_chunk_bwd_workspace.argtypes = [I, I, I, I, I]
        lib.kda_chunk_bwd_workspace.restype = Z
        lib.kda_chunk_bwd.argtypes = [P, P, P, P, P, P, P, P, P, P, P, P, P, P, I, I, I, I, I,
                                      I, F, I, I, P, Z, P]
        lib.kda_chunk_bwd.restype = I
        lib.kda_gk_chunk_bwd_workspace.argtypes = [I, I, I, I, I]
        lib.kda_gk_chunk_bwd_workspace.restype = Z
        lib.kda_gk_chunk_bwd.argtypes = [P, P, P, P, P, P, P, P, P, P, P, P, P, P, I, I, I, I, I,
                                         I, F, I, I, P, Z, P]
        lib.kda_gk_chunk_bwd.restype = I
        lib.kda_gate_decay.argtypes = [P, P, P, P, ctypes.c_long, I, I, P]
        lib.kda_gate_decay.restype = I
        lib.kda_gk_chunk_fwd.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, I, F, I, I, O, P,
                                         Z, P]
        lib.kda_gk_chunk_fwd.restype = I
        lib.kda_gk_varlen_fwd.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, P, P, P, I, F, I, I,
                                          O, P, Z, P]
        lib.kda_gk_varlen_fwd.restype = I
        lib.kda_gk_recurrent_fwd.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, I, F, I, O,
                                             P]
        lib.kda_gk_recurrent_fwd.restype = I
        lib.kda_gk_varlen_recurrent_fwd.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, P, P, P,
                                                    I, F, I, O, P]
        lib.kda_gk_varlen_recurrent_fwd.restype = I
        lib.kda_gk_decode_step.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, F, I, O, P]
        lib.kda_gk_decode_step.restype = I
        lib.kda_query_device_error.argtypes = [P, P]
        lib.kda_query_device_error.restype = I
        lib.kda_diag_wait_timeout.argtypes = [P, Z, ctypes.c_uint, P]
        lib.kda_diag_wait_timeout.restype = I
        _lib = lib
        return lib


def _value_heads(H, HV):
    """Value heads per q/k head (TileOPs GDNFwdOp / KDAFwdOp: HV a multiple of H)."""
    if HV < H or HV % H:
        raise ValueError(f"the value heads ({HV}) must be a multiple of the q/k heads ({H})")
    return HV // H


def _st(n, hv, dk, dv, v_first):
    """Shape of a state array: key-major [n, hv, dk, dv] or value-major [n, hv, dv, dk]."""
    return (n, hv, dv, dk) if v_first else (n, hv, dk, dv)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return KDA_BF16
    if t.dtype == torch.float32:
        return KDA_F32
    raise TypeError(f"q/k/v must be bfloat16 or float32, got {t.dtype}")


def _check(t, name, dtype=None, shape=None):
    if t is None:
        return
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _raise(code, where, lib):
    if code != 0:
        raise KdaError(code, where, lib)


def chunk_fwd_workspace_bytes(B, T, H, dk, dv, chunk_size, dtype_code):
    return int(load().kda_chunk_fwd_workspace(B, T, H, dk, dv, chunk_size, dtype_code))


def varlen_fwd_workspace_bytes(N, total_T, H, dk, dv, chunk_size, dtype_code):
    return int(load().kda_varlen_fwd_workspace(N, total_T, H, dk, dv, chunk_size, dtype_code))


def _workspace(nbytes, device, workspace):
    if workspace is not None:
        if workspace.numel() * workspace.element_size() < nbytes:
            raise ValueError("workspace too small")
        return workspace
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def chunk_fwd(q, k, v, beta, decay=None, initial_state=None, *, scale=None, chunk_size=64,
              use_qk_l2norm=True, out=None, final_state=None, workspace=None, stream=None,
              check_device=False,
              decayed_read=False, A_log=None, dt_bias=None, beta_sigmoid=False,
              allow_neg_eigval=False, state_v_first=False):
    """kda_chunk_fwd (kda_chunk_fwd_ex when an option is set): chunked prefill.  Returns
    (o [B,T,H,dv], final_state [B,H,dk,dv] fp32).

    check_device=True synchronises the stream afterwards and raises if a kernel recorded
    a device error (a bounded wait that ran out) in the workspace header.  The options are
    those of kda_options: decayed_read, the in-kernel gate (decay holds the raw gate; A_log
    [H], dt_bias [H]) and the beta transforms.
    """
    lib = load()
    B, T, H, dk = q.shape
    HV, dv = v.shape[2], v.shape[-1]
    m = _value_heads(H, HV)
    dt = _dtype_code(q)
    _check(q, "q"); _check(k, "k", q.dtype, q.shape); _check(v, "v", q.dtype, (B, T, HV, dv))
    _check(beta, "beta", torch.float32, (B, T, HV)); _check(decay, "decay", torch.float32, (B, T, HV))
    _check(initial_state, "initial_state", torch.float32, _st(B, HV, dk, dv, state_v_first))
    o = out if out is not None else torch.empty((B, T, HV, dv), dtype=q.dtype, device=q.device)
    _check(o, "out", q.dtype, (B, T, HV, dv))
    hT = final_state if final_state is not None else torch.empty(_st(B, HV, dk, dv, state_v_first),
                                                                 dtype=torch.float32, device=q.device)
    _check(hT, "final_state", torch.float32, _st(B, HV, dk, dv, state_v_first))
    need = lib.kda_chunk_fwd_workspace(B, T, HV, dk, dv, chunk_size, dt)
    if need == 0:
        raise KdaError(4, "kda_chunk_fwd_workspace", lib)
    ws = _workspace(need, q.device, workspace)
    opts = make_options(decayed_read, A_log, dt_bias, beta_sigmoid, allow_neg_eigval, m, state_v_first)
    args = (_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(decay), _ptr(initial_state), _ptr(o),
            _ptr(hT), B, T, H, dk, dv, dt, float(scale or 0.0), int(chunk_size),
            int(bool(use_qk_l2norm)))
    tail = (_ptr(ws), ws.numel() * ws.element_size(), _stream(stream))
    if opts is None:
        _raise(lib.kda_chunk_fwd(*args, *tail), "kda_chunk_fwd", lib)
    else:
        _raise(lib.kda_chunk_fwd_ex(*args, opts, *tail), "kda_chunk_fwd_ex", lib)
    if check_device:
        _raise(query_device_error(ws, stream), "kda_chunk_fwd (device)", lib)
    return o, hT


def chunk_fwd_noalloc(q, k, v, beta, decay=None, initial_state=None, *, scale=None,
                      chunk_size=64, use_qk_l2norm=True, out=None, final_state=None, stream=None):
    """kda_chunk_fwd_noalloc: chunked prefill with the library's built-in scratch.

    For callers that cannot hand over device memory for a workspace.  bf16 q/k/v with
    dk == dv in {64, 128} and chunk 64 only; the scratch is the library's built-in 48 MiB
    array, which every such problem fits.  Calls that overlap on the GPU race on that one
    buffer, so keep them ordered.  query_device_error(None) reads its error word.
    Returns (o, final_state).
    """
    lib = load()
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    dt = _dtype_code(q)
    _check(q, "q"); _check(k, "k", q.dtype, q.shape); _check(v, "v", q.dtype, (B, T, H, dv))
    _check(beta, "beta", torch.float32, (B, T, H)); _check(decay, "decay", torch.float32, (B, T, H))
    _check(initial_state, "initial_state", torch.float32, (B, H, dk, dv))
    o = out if out is not None else torch.empty((B, T, H, dv), dtype=q.dtype, device=q.device)
    _check(o, "out", q.dtype, (B, T, H, dv))
    hT = final_state if final_state is not None else torch.empty((B, H, dk, dv), dtype=torch.float32,
                                                                  device=q.device)
    _check(hT, "final_state", torch.float32, (B, H, dk, dv))
    rc = lib.kda_chunk_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(decay),
                                   _ptr(initial_state), _ptr(o), _ptr(hT), B, T, H, dk, dv, dt,
                                   float(scale or 0.0), int(chunk_size), int(bool(use_qk_l2norm)),
                                   _stream(stream))
    _raise(rc, "kda_chunk_fwd_noalloc", lib)
    return o, hT


def recurrent_fwd(q, k, v, beta, decay=None, initial_state=None, *, scale=None,
                  use_qk_l2norm=True, out=None, final_state=None, stream=None,
                  decayed_read=False, A_log=None, dt_bias=None, beta_sigmoid=False,
                  allow_neg_eigval=False, state_v_first=False):
    """kda_recurrent_fwd (_ex with options, as chunk_fwd): token-by-token prefill.
    Returns (o, final_state)."""
    lib = load()
    B, T, H, dk = q.shape
    HV, dv = v.shape[2], v.shape[-1]
    m = _value_heads(H, HV)
    dt = _dtype_code(q)
    _check(q, "q"); _check(k, "k", q.dtype, q.shape); _check(v, "v", q.dtype, (B, T, HV, dv))
    _check(beta, "beta", torch.float32, (B, T, HV)); _check(decay, "decay", torch.float32, (B, T, HV))
    _check(initial_state, "initial_state", torch.float32, _st(B, HV, dk, dv, state_v_first))
    o = out if out is not None else torch.empty((B, T, HV, dv), dtype=q.dtype, device=q.device)
    hT = final_state if final_state is not None else torch.empty(_st(B, HV, dk, dv, state_v_first),
                                                                 dtype=torch.float32, device=q.device)
    opts = make_options(decayed_read, A_log, dt_bias, beta_sigmoid, allow_neg_eigval, m, state_v_first)
    args = (_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(decay), _ptr(initial_state), _ptr(o),
            _ptr(hT), B, T, H, dk, dv, dt, float(scale or 0.0), int(bool(use_qk_l2norm)))
    if opts is None:
        _raise(lib.kda_recurrent_fwd(*args, _stream(stream)), "kda_recurrent_fwd", lib)
    else:
        _raise(lib.kda_recurrent_fwd_ex(*args, opts, _stream(stream)), "kda_recurrent_fwd_ex", lib)
    return o, hT


def decode_step(q, k, v, beta, decay, state, *, scale=None, use_qk_l2norm=True, out=None,
                stream=None,
                decayed_read=False, A_log=None, dt_bias=None, beta_sigmoid=False,
                allow_neg_eigval=False, state_v_first=False):
    """kda_decode_step: one token per sequence; ``state`` [B,HV,dk,dv] fp32 is updated in place.

    q, k: [B,1,H,dk] (or [B,H,dk]); v: [B,1,HV,dv]; beta, decay: [B,1,HV] (decay may be None);
    HV = H without grouped value heads.  Returns o with v's shape.
    """
    lib = load()
    B, HV, s2, s3 = state.shape
    dk, dv = (s3, s2) if state_v_first else (s2, s3)
    H = q.numel() // max(B * dk, 1)
    m = _value_heads(H, HV)
    dt = _dtype_code(q)
    _check(q, "q"); _check(k, "k", q.dtype); _check(v, "v", q.dtype)
    _check(beta, "beta", torch.float32); _check(decay, "decay", torch.float32)
    _check(state, "state", torch.float32)
    if q.numel() != B * H * dk or v.numel() != B * HV * dv or beta.numel() != B * HV:
        raise ValueError("decode inputs do not match the state's [B,HV,dk,dv]")
    o = out if out is not None else torch.empty_like(v)
    opts = make_options(decayed_read, A_log, dt_bias, beta_sigmoid, allow_neg_eigval, m, state_v_first)
    args = (_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(decay), _ptr(state), _ptr(o), B, H, dk,
            dv, dt, float(scale or 0.0), int(bool(use_qk_l2norm)))
    if opts is None:
        _raise(lib.kda_decode_step(*args, _stream(stream)), "kda_decode_step", lib)
    else:
        _raise(lib.kda_decode_step_ex(*args, opts, _stream(stream)), "kda_decode_step_ex", lib)
    return o


def varlen_fwd(q, k, v, beta, cu_seqlens, decay=None, initial_state=None, *, cu_seqlens_cpu=None,
               scale=None, chunk_size=64, use_qk_l2norm=True, out=None, final_state=None,
               workspace=None, stream=None, check_device=False,
               decayed_read=False, A_log=None, dt_bias=None, beta_sigmoid=False,
               allow_neg_eigval=False, state_v_first=False):
    """kda_varlen_fwd: packed sequences [1,total,H,D] split by cu_seqlens [N+1] (int32, device).

    Returns (o [1,total,H,dv], final_state [N,H,dk,dv] fp32).  check_device as in chunk_fwd.
    """
    lib = load()
    _, total, H, dk = q.shape
    HV, dv = v.shape[2], v.shape[-1]
    m = _value_heads(H, HV)
    N = cu_seqlens.numel() - 1
    dt = _dtype_code(q)
    _check(q, "q"); _check(k, "k", q.dtype, q.shape); _check(v, "v", q.dtype, (1, total, HV, dv))
    _check(beta, "beta", torch.float32, (1, total, HV))
    _check(decay, "decay", torch.float32, (1, total, HV))
    _check(cu_seqlens, "cu_seqlens", torch.int32)
    _check(initial_state, "initial_state", torch.float32, _st(N, HV, dk, dv, state_v_first))
    host = None
    if cu_seqlens_cpu is not None:
        host = cu_seqlens_cpu.to(torch.int32).contiguous()
        if host.is_cuda:
            raise ValueError("cu_seqlens_cpu must be a host tensor")
    o = out if out is not None else torch.empty((1, total, HV, dv), dtype=q.dtype, device=q.device)
    hT = final_state if final_state is not None else torch.empty(_st(N, HV, dk, dv, state_v_first),
                                                                 dtype=torch.float32, device=q.device)
    need = lib.kda_varlen_fwd_workspace(N, total, HV, dk, dv, chunk_size, dt)
    if need == 0:
        raise KdaError(4, "kda_varlen_fwd_workspace", lib)
    ws = _workspace(need, q.device, workspace)
    opts = make_options(decayed_read, A_log, dt_bias, beta_sigmoid, allow_neg_eigval, m, state_v_first)
    args = (_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(decay), _ptr(cu_seqlens), _ptr(host), N,
            total, H, dk, dv, _ptr(initial_state), _ptr(o), _ptr(hT), dt, float(scale or 0.0),
            int(chunk_size), int(bool(use_qk_l2norm)))
    tail = (_ptr(ws), ws.numel() * ws.element_size(), _stream(stream))
    if opts is None:
        _raise(lib.kda_varlen_fwd(*args, *tail), "kda_varlen_fwd", lib)
    else:
        _raise(lib.kda_varlen_fwd_ex(*args, opts, *tail), "kda_varlen_fwd_ex", lib)
    if check_device:
        _raise(query_device_error(ws, stream), "kda_varlen_fwd (device)", lib)
    return o, hT


def gk_chunk_fwd(q, k, v, beta, g=None, initial_state=None, *, cu_seqlens=None, cu_seqlens_cpu=None,
                 scale=None, chunk_size=64, use_qk_l2norm=True, out=None, final_state=None,
                 workspace=None, stream=None, check_device=False,
                 decayed_read=False, A_log=None, dt_bias=None, beta_sigmoid=False,
                 allow_neg_eigval=False, state_v_first=False):
    """kda_gk_chunk_fwd / kda_gk_varlen_fwd: chunked prefill with one log decay per key
    channel (g with q's shape, fp32).  Packed when ``cu_seqlens`` is given (as
    gk_recurrent_fwd).  check_device as in chunk_fwd.  Returns (o, final_state)."""
    lib = load()
    Bq, T, H, dk = q.shape
    HV, dv = v.shape[2], v.shape[-1]
    m = _value_heads(H, HV)
    opts = make_options(decayed_read, A_log, dt_bias, beta_sigmoid, allow_neg_eigval, m, state_v_first)
    dt = _dtype_code(q)
    N = Bq if cu_seqlens is None else cu_seqlens.numel() - 1
    _check(q, "q"); _check(k, "k", q.dtype, q.shape); _check(v, "v", q.dtype, (Bq, T, HV, dv))
    _check(beta, "beta", torch.float32, (Bq, T, HV)); _check(g, "g", torch.float32, (Bq, T, HV, dk))
    _check(initial_state, "initial_state", torch.float32, _st(N, HV, dk, dv, state_v_first))
    o = out if out is not None else torch.empty((Bq, T, HV, dv), dtype=q.dtype, device=q.device)
    _check(o, "out", q.dtype, (Bq, T, HV, dv))
    hT = final_state if final_state is not None else torch.empty(_st(N, HV, dk, dv, state_v_first),
                                                                 dtype=torch.float32, device=q.device)
    _check(hT, "final_state", torch.float32, _st(N, HV, dk, dv, state_v_first))
    if cu_seqlens is None:
        need = lib.kda_chunk_fwd_workspace(Bq, T, HV, dk, dv, chunk_size, dt)
        if need == 0:
            raise KdaError(4, "kda_chunk_fwd_workspace", lib)
        ws = _workspace(need, q.device, workspace)
        rc = lib.kda_gk_chunk_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g), _ptr(initial_state),
                                  _ptr(o), _ptr(hT), Bq, T, H, dk, dv, dt, float(scale or 0.0),
                                  int(chunk_size), int(bool(use_qk_l2norm)), opts,
                                  _ptr(ws), ws.numel() * ws.element_size(), _stream(stream))
        _raise(rc, "kda_gk_chunk_fwd", lib)
    else:
        if Bq != 1:
            raise ValueError("packed sequences need token arrays with B == 1")
        _check(cu_seqlens, "cu_seqlens", torch.int32)
        host = None
        if cu_seqlens_cpu is not None:
            host = cu_seqlens_cpu.to(torch.int32).contiguous()
            if host.is_cuda:
                raise ValueError("cu_seqlens_cpu must be a host tensor")
        need = lib.kda_varlen_fwd_workspace(N, T, HV, dk, dv, chunk_size, dt)
        if need == 0:
            raise KdaError(4, "kda_varlen_fwd_workspace", lib)
        ws = _workspace(need, q.device, workspace)
        rc = lib.kda_gk_varlen_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g), _ptr(cu_seqlens),
                                   _ptr(host), N, T, H, dk, dv, _ptr(initial_state), _ptr(o), _ptr(hT),
                                   dt, float(scale or 0.0), int(chunk_size), int(bool(use_qk_l2norm)),
                                   opts, _ptr(ws), ws.numel() * ws.element_size(),
                                   _stream(stream))
        _raise(rc, "kda_gk_varlen_fwd", lib)
    if check_device:
        _raise(query_device_error(ws, stream), "kda_gk_chunk_fwd (device)", lib)
    return o, hT


def gk_recurrent_fwd(q, k, v, beta, g=None, initial_state=None, *, cu_seqlens=None,
                     cu_seqlens_cpu=None, scale=None, use_qk_l2norm=True, out=None,
                     final_state=None, stream=None,
                     decayed_read=False, A_log=None, dt_bias=None, beta_sigmoid=False,
                     allow_neg_eigval=False, state_v_first=False):
    """kda_gk_recurrent_fwd / kda_gk_varlen_recurrent_fwd: token-by-token prefill with one
    log decay per key channel, g with q's shape (fp32).  ``decayed_read`` selects where the
    delta term reads the memory.  With ``cu_seqlens`` (int32, device, [N+1]) the token
    arrays are packed [1,total,H,.] and the states are [N,H,dk,dv].  Returns (o, final_state).
    """
    lib = load()
    Bq, T, H, dk = q.shape
    HV, dv = v.shape[2], v.shape[-1]
    m = _value_heads(H, HV)
    opts = make_options(decayed_read, A_log, dt_bias, beta_sigmoid, allow_neg_eigval, m, state_v_first)
    dt = _dtype_code(q)
    N = Bq if cu_seqlens is None else cu_seqlens.numel() - 1
    _check(q, "q"); _check(k, "k", q.dtype, q.shape); _check(v, "v", q.dtype, (Bq, T, HV, dv))
    _check(beta, "beta", torch.float32, (Bq, T, HV)); _check(g, "g", torch.float32, (Bq, T, HV, dk))
    _check(initial_state, "initial_state", torch.float32, _st(N, HV, dk, dv, state_v_first))
    o = out if out is not None else torch.empty((Bq, T, HV, dv), dtype=q.dtype, device=q.device)
    _check(o, "out", q.dtype, (Bq, T, HV, dv))
    hT = final_state if final_state is not None else torch.empty(_st(N, HV, dk, dv, state_v_first),
                                                                 dtype=torch.float32, device=q.device)
    _check(hT, "final_state", torch.float32, _st(N, HV, dk, dv, state_v_first))
    if cu_seqlens is None:
        rc = lib.kda_gk_recurrent_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g),
                                      _ptr(initial_state), _ptr(o), _ptr(hT), Bq, T, H, dk, dv, dt,
                                      float(scale or 0.0), int(bool(use_qk_l2norm)),
                                      opts, _stream(stream))
        _raise(rc, "kda_gk_recurrent_fwd", lib)
        return o, hT
    if Bq != 1:
        raise ValueError("packed sequences need token arrays with B == 1")
    _check(cu_seqlens, "cu_seqlens", torch.int32)
    host = None
    if cu_seqlens_cpu is not None:
        host = cu_seqlens_cpu.to(torch.int32).contiguous()
        if host.is_cuda:
            raise ValueError("cu_seqlens_cpu must be a host tensor")
    rc = lib.kda_gk_varlen_recurrent_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g),
                                         _ptr(cu_seqlens), _ptr(host), N, T, H, dk, dv,
                                         _ptr(initial_state), _ptr(o), _ptr(hT), dt,
                                         float(scale or 0.0), int(bool(use_qk_l2norm)),
                                         opts, _stream(stream))
    _raise(rc, "kda_gk_varlen_recurrent_fwd", lib)
    return o, hT


def gk_decode_step(q, k, v, beta, g, state, *, scale=None, use_qk_l2norm=True, out=None,
                   stream=None,
                   decayed_read=False, A_log=None, dt_bias=None, beta_sigmoid=False,
                   allow_neg_eigval=False, state_v_first=False):
    """kda_gk_decode_step: one token per sequence with per-channel decay g [B,1,H,dk] fp32
    (or None); ``state`` [B,H,dk,dv] fp32 is updated in place.  Returns o with v's shape."""
    lib = load()
    B, HV, s2, s3 = state.shape
    dk, dv = (s3, s2) if state_v_first else (s2, s3)
    H = q.numel() // max(B * dk, 1)
    m = _value_heads(H, HV)
    opts = make_options(decayed_read, A_log, dt_bias, beta_sigmoid, allow_neg_eigval, m, state_v_first)
    dt = _dtype_code(q)
    _check(q, "q"); _check(k, "k", q.dtype); _check(v, "v", q.dtype)
    _check(beta, "beta", torch.float32); _check(g, "g", torch.float32)
    _check(state, "state", torch.float32)
    if q.numel() != B * H * dk or v.numel() != B * HV * dv or beta.numel() != B * HV or (
            g is not None and g.numel() != B * HV * dk):
        raise ValueError("decode inputs do not match the state's [B,HV,dk,dv]")
    o = out if out is not None else torch.empty_like(v)
    rc = lib.kda_gk_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g), _ptr(state),
                                _ptr(o), B, H, dk, dv, dt, float(scale or 0.0),
                                int(bool(use_qk_l2norm)), opts,
                                _stream(stream))
    _raise(rc, "kda_gk_decode_step", lib)
    return o


def query_device_error(workspace, stream=None) -> int:
    """kda_query_device_error: device error word of the last call on ``workspace`` (0 = none);
    ``workspace=None``: the built-in array of chunk_fwd_noalloc on the current device."""
    return int(load().kda_query_device_error(_ptr(workspace), _stream(stream)))


def diag_wait_timeout(workspace, limit_us, stream=None) -> None:
    """kda_diag_wait_timeout: enqueue the failure-detection probe on ``workspace``; its
    bounded waits run out after ``limit_us`` each and record KDA_ERR_DEVICE_TIMEOUT, which
    query_device_error(workspace) then returns."""
    lib = load()
    nbytes = workspace.numel() * workspace.element_size()
    _raise(lib.kda_diag_wait_timeout(_ptr(workspace), nbytes, int(limit_us), _stream(stream)),
           "kda_diag_wait_timeout", lib)


def gate_decay(gate, A_log, dt_bias=None, *, out=None, stream=None):
    """kda_gate_decay (ejkernel kda_decay): -exp(A_log[h]) softplus(gate + dt_bias).
    gate [..., H] with A_log, dt_bias [H], or [..., H, K] with dt_bias [H, K]; fp32 CUDA."""
    lib = load()
    H = A_log.numel()
    K = 1 if gate.shape[-1] == H and (dt_bias is None or dt_bias.dim() == 1) else gate.shape[-1]
    _check(gate, "gate", torch.float32); _check(A_log, "A_log", torch.float32)
    _check(dt_bias, "dt_bias", torch.float32)
    if dt_bias is not None and dt_bias.numel() != H * K:
        raise ValueError("dt_bias must have H * K elements")
    o = out if out is not None else torch.empty_like(gate)
    rows = gate.numel() // (H * K)
    _raise(lib.kda_gate_decay(_ptr(gate), _ptr(A_log), _ptr(dt_bias), _ptr(o), rows, H, K,
                              _stream(stream)), "kda_gate_decay", lib)
    return o


def gk_recurrent_bwd(q, k, v, beta, g, initial_state, d_o, dfinal_state=None, *, scale=None,
                     use_qk_l2norm=True, decayed_read=False, workspace=None, stream=None):
    """kda_gk_recurrent_bwd: fp32 gradients of the per-channel recurrence with respect to q, k,
    v, beta, g and initial_state, given dL/do (dtype of q) and dL/dfinal_state (fp32 or None).
    Returns a dict dq, dk, dv, dbeta, dg, dh0."""
    lib = load()
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    dt = _dtype_code(q)
    _check(q, "q"); _check(k, "k", q.dtype, q.shape); _check(v, "v", q.dtype, (B, T, H, dv))
    _check(beta, "beta", torch.float32, (B, T, H)); _check(g, "g", torch.float32, q.shape)
    _check(initial_state, "initial_state", torch.float32, (B, H, dk, dv))
    _check(d_o, "d_o", q.dtype, (B, T, H, dv))
    _check(dfinal_state, "dfinal_state", torch.float32, (B, H, dk, dv))
    f32 = dict(dtype=torch.float32, device=q.device)
    out = dict(dq=torch.empty((B, T, H, dk), **f32), dk=torch.empty((B, T, H, dk), **f32),
               dv=torch.empty((B, T, H, dv), **f32), dbeta=torch.empty((B, T, H), **f32),
               dg=torch.empty((B, T, H, dk), **f32), dh0=torch.empty((B, H, dk, dv), **f32))
    need = lib.kda_gk_recurrent_bwd_workspace(B, T, H, dk, dv)
    if need == 0:
        raise KdaError(4, "kda_gk_recurrent_bwd_workspace", lib)
    ws = _workspace(need, q.device, workspace)
    rc = lib.kda_gk_recurrent_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g), _ptr(initial_state),
                                  _ptr(d_o), _ptr(dfinal_state), _ptr(out["dq"]), _ptr(out["dk"]),
                                  _ptr(out["dv"]), _ptr(out["dbeta"]), _ptr(out["dg"]), _ptr(out["dh0"]),
                                  B, T, H, dk, dv, dt, float(scale or 0.0), int(bool(use_qk_l2norm)),
                                  int(bool(decayed_read)), _ptr(ws), ws.numel() * ws.element_size(),
                                  _stream(stream))
    _raise(rc, "kda_gk_recurrent_bwd", lib)
    return out


def recurrent_bwd(q, k, v, beta, decay, initial_state, d_o, dfinal_state=None, *, scale=None,
                  use_qk_l2norm=True, decayed_read=False, workspace=None, stream=None):
    """kda_recurrent_bwd: fp32 gradients of the recurrence with one decay per head (decay
    [B,T,H] or None) with respect to q, k, v, beta, decay and initial_state, given dL/do
    (dtype of q) and dL/dfinal_state (fp32 or None).  Returns a dict dq, dk, dv, dbeta,
    ddecay, dh0."""
    lib = load()
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    dt = _dtype_code(q)
    _check(q, "q"); _check(k, "k", q.dtype, q.shape); _check(v, "v", q.dtype, (B, T, H, dv))
    _check(beta, "beta", torch.float32, (B, T, H)); _check(decay, "decay", torch.float32, (B, T, H))
    _check(initial_state, "initial_state", torch.float32, (B, H, dk, dv))
    _check(d_o, "d_o", q.dtype, (B, T, H, dv))
    _check(dfinal_state, "dfinal_state", torch.float32, (B, H, dk, dv))
    f32 = dict(dtype=torch.float32, device=q.device)
    out = dict(dq=torch.empty((B, T, H, dk), **f32), dk=torch.empty((B, T, H, dk), **f32),
               dv=torch.empty((B, T, H, dv), **f32), dbeta=torch.empty((B, T, H), **f32),
               ddecay=torch.empty((B, T, H), **f32), dh0=torch.empty((B, H, dk, dv), **f32))
    need = lib.kda_recurrent_bwd_workspace(B, T, H, dk, dv)
    if need == 0:
        raise KdaError(4, "kda_recurrent_bwd_workspace", lib)
    ws = _workspace(need, q.device, workspace)
    rc = lib.kda_recurrent_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(decay), _ptr(initial_state),
                               _ptr(d_o), _ptr(dfinal_state), _ptr(out["dq"]), _ptr(out["dk"]),
                               _ptr(out["dv"]), _ptr(out["dbeta"]), _ptr(out["ddecay"]), _ptr(out["dh0"]),
                               B, T, H, dk, dv, dt, float(scale or 0.0), int(bool(use_qk_l2norm)),
                               int(bool(decayed_read)), _ptr(ws), ws.numel() * ws.element_size(),
                               _stream(stream))
    _raise(rc, "kda_recurrent_bwd", lib)
    return out


def chunk_bwd(q, k, v, beta, decay, initial_state, d_o, dfinal_state=None, *, scale=None,
                  use_qk_l2norm=True, decayed_read=False, workspace=None, stream=None):
    """kda_chunk_bwd: the gradients of recurrent_bwd computed by chunks on the tensor cores
    (bf16 q/k/v/d_o, dk == dv in {64, 128}).  Returns a dict dq, dk, dv, dbeta, ddecay, dh0."""
    lib = load()
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    dt = _dtype_code(q)
    _check(q, "q"); _check(k, "k", q.dtype, q.shape); _check(v, "v", q.dtype, (B, T, H, dv))
    _check(beta, "beta", torch.float32, (B, T, H)); _check(decay, "decay", torch.float32, (B, T, H))
    _check(initial_state, "initial_state", torch.float32, (B, H, dk, dv))
    _check(d_o, "d_o", q.dtype, (B, T, H, dv))
    _check(dfinal_state, "dfinal_state", torch.float32, (B, H, dk, dv))
    f32 = dict(dtype=torch.float32, device=q.device)
    out = dict(dq=torch.empty((B, T, H, dk), **f32), dk=torch.empty((B, T, H, dk), **f32),
               dv=torch.empty((B, T, H, dv), **f32), dbeta=torch.empty((B, T, H), **f32),
               ddecay=torch.empty((B, T, H), **f32), dh0=torch.empty((B, H, dk, dv), **f32))
    need = lib.kda_chunk_bwd_workspace(B, T, H, dk, dv)
    if need == 0:
        raise KdaError(4, "kda_chunk_bwd_workspace", lib)
    ws = _workspace(need, q.device, workspace)
    rc = lib.kda_chunk_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(decay), _ptr(initial_state),
                               _ptr(d_o), _ptr(dfinal_state), _ptr(out["dq"]), _ptr(out["dk"]),
                               _ptr(out["dv"]), _ptr(out["dbeta"]), _ptr(out["ddecay"]), _ptr(out["dh0"]),
                               B, T, H, dk, dv, dt, float(scale or 0.0), int(bool(use_qk_l2norm)),
                               int(bool(decayed_read)), _ptr(ws), ws.numel() * ws.element_size(),
                               _stream(stream))
    _raise(rc, "kda_chunk_bwd", lib)
    return out


def gk_chunk_bwd(q, k, v, beta, g, initial_state, d_o, dfinal_state=None, *, scale=None,
                 use_qk_l2norm=True, decayed_read=False, workspace=None, stream=None):
    """kda_gk_chunk_bwd: the gradients of gk_recurrent_bwd with the two walks on the tensor
    cores and every chunk's token walk at once (bf16 q/k/v/d_o, dk == dv in {64, 128}).
    Returns a dict dq, dk, dv, dbeta, dg, dh0."""
    lib = load()
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    dt = _dtype_code(q)
    _check(q, "q"); _check(k, "k", q.dtype, q.shape); _check(v, "v", q.dtype, (B, T, H, dv))
    _check(beta, "beta", torch.float32, (B, T, H)); _check(g, "g", torch.float32, q.shape)
    _check(initial_state, "initial_state", torch.float32, (B, H, dk, dv))
    _check(d_o, "d_o", q.dtype, (B, T, H, dv))
    _check(dfinal_state, "dfinal_state", torch.float32, (B, H, dk, dv))
    f32 = dict(dtype=torch.float32, device=q.device)
    out = dict(dq=torch.empty((B, T, H, dk), **f32), dk=torch.empty((B, T, H, dk), **f32),
               dv=torch.empty((B, T, H, dv), **f32), dbeta=torch.empty((B, T, H), **f32),
               dg=torch.empty((B, T, H, dk), **f32), dh0=torch.empty((B, H, dk, dv), **f32))
    need = lib.kda_gk_chunk_bwd_workspace(B, T, H, dk, dv)
    if need == 0:
        raise KdaError(4, "kda_gk_chunk_bwd_workspace", lib)
    ws = _workspace(need, q.device, workspace)
    rc = lib.kda_gk_chunk_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g), _ptr(initial_state),
                              _ptr(d_o), _ptr(dfinal_state), _ptr(out["dq"]), _ptr(out["dk"]),
                              _ptr(out["dv"]), _ptr(out["dbeta"]), _ptr(out["dg"]), _ptr(out["dh0"]),
                              B, T, H, dk, dv, dt, float(scale or 0.0), int(bool(use_qk_l2norm)),
                              int(bool(decayed_read)), _ptr(ws), ws.numel() * ws.element_size(),
                              _stream(stream))
    _raise(rc, "kda_gk_chunk_bwd", lib)
    return out
