"""fp64 gradients of the per-key-channel recurrence -- TEST INFRASTRUCTURE.

Only ``tests/`` and the benchmark's reference leg may import this module; the GPU library
never does.  The forward is the per-channel recurrence of TileOPs "Linear Attention
Operators", KDAFwdOp (one log decay per key channel, D_t = diag(exp g_t)), in the order of
ejkernel kda() "The core recurrence" or, with ``decayed_read``, the gated delta rule:

    u_t = beta_t (v_t - R_t^T k^_t),   R_t = h_{t-1} or D_t h_{t-1}
    h_t = D_t h_{t-1} + k^_t u_t^T,    o_t = h_t^T q~_t,   k^ = l2(k),  q~ = scale l2(q)

written with plain PyTorch CPU ops in float64, one token at a time, and differentiated by
torch.autograd (the backward of the training mode named in the kda-neuron-kernels README,
"kda_chunk_step_exact_bwd": dq, dk, dv, dg, dbeta and the state gradient).  The pins in
tests/ compare it with central finite differences and with the C oracle's forward.
"""
from __future__ import annotations

import numpy as np
import torch


def _l2(x):
    return x / torch.clamp(torch.linalg.vector_norm(x, dim=-1, keepdim=True), min=1e-12)


def forward_torch(q, k, v, beta, g, h0, *, scale=None, use_l2=True, decayed_read=False):
    """q, k, g [B,T,H,dk]; v [B,T,H,dv]; beta [B,T,H]; h0 [B,H,dk,dv]: float64 tensors.
    Returns (o [B,T,H,dv], hT [B,H,dk,dv])."""
    B, T, H, dk = q.shape
    s = scale if scale else dk ** -0.5
    kk = _l2(k) if use_l2 else k
    qq = (_l2(q) if use_l2 else q) * s
    h = h0
    outs = []
    for t in range(T):
        a = torch.exp(g[:, t])                                   # [B,H,dk]
        hd = a[..., None] * h
        read = hd if decayed_read else h
        r = torch.einsum("bhij,bhi->bhj", read, kk[:, t])
        u = beta[:, t, :, None] * (v[:, t] - r)
        h = hd + kk[:, t, ..., None] * u[:, :, None, :]
        outs.append(torch.einsum("bhij,bhi->bhj", h, qq[:, t]))
    return torch.stack(outs, dim=1), h


def backward(q, k, v, beta, g, h0, do, dhT=None, *, scale=None, use_l2=True, decayed_read=False):
    """Gradients of sum(o * do) + sum(hT * dhT) with respect to q, k, v, beta, g and h0 (numpy
    in, numpy float64 out).  Returns a dict with keys dq, dk, dv, dbeta, dg, dh0."""
    t = {n: torch.tensor(np.asarray(x, np.float64), requires_grad=True)
         for n, x in (("q", q), ("k", k), ("v", v), ("beta", beta), ("g", g), ("h0", h0))}
    o, hT = forward_torch(t["q"], t["k"], t["v"], t["beta"], t["g"], t["h0"], scale=scale,
                          use_l2=use_l2, decayed_read=decayed_read)
    loss = (o * torch.tensor(np.asarray(do, np.float64))).sum()
    if dhT is not None:
        loss = loss + (hT * torch.tensor(np.asarray(dhT, np.float64))).sum()
    grads = torch.autograd.grad(loss, [t[n] for n in ("q", "k", "v", "beta", "g", "h0")])
    return {n: gr.detach().numpy() for n, gr in zip(("dq", "dk", "dv", "dbeta", "dg", "dh0"), grads)}
