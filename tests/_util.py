"""Shared test helpers: tolerances and tensor marshalling (no method arithmetic)."""
import numpy as np

# Tolerances of the parity bar:
#   fp32 inputs: max relative error <= 1e-4 on o and on final_state, read normwise
#                (max |diff| / max |ref|) per tensor;
#   bf16 inputs with an fp32 state, against the oracle on the same bf16-rounded inputs:
#                max |do| <= 2e-2 * max |o|  and  ||d final_state||_F / ||final_state||_F <= 1e-2.
F32_REL = 1e-4
BF16_O = 2e-2
BF16_STATE_FROB = 1e-2


def max_rel(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    den = np.max(np.abs(ref)) if ref.size else 0.0
    if den == 0.0:
        return float(np.max(np.abs(got))) if got.size else 0.0
    return float(np.max(np.abs(got - ref)) / den)


def frob_rel(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    den = np.linalg.norm(ref)
    if den == 0.0:
        return float(np.linalg.norm(got))
    return float(np.linalg.norm(got - ref) / den)


def assert_parity(dtype, o, ro, h=None, rh=None, tag=""):
    """Apply the bar for the input dtype ("f32" or "bf16")."""
    if dtype == "f32":
        eo = max_rel(o, ro)
        assert eo <= F32_REL, f"{tag} o max-rel {eo:.3e} > {F32_REL}"
        if h is not None:
            eh = max_rel(h, rh)
            assert eh <= F32_REL, f"{tag} final_state max-rel {eh:.3e} > {F32_REL}"
    else:
        eo = max_rel(o, ro)
        assert eo <= BF16_O, f"{tag} o max-abs/max|o| {eo:.3e} > {BF16_O}"
        if h is not None:
            eh = frob_rel(h, rh)
            assert eh <= BF16_STATE_FROB, f"{tag} final_state frob-rel {eh:.3e} > {BF16_STATE_FROB}"


def to_dev(x, dev, dtype):
    import torch
    if x is None:
        return None
    return torch.from_numpy(np.ascontiguousarray(x)).to(device=dev, dtype=dtype)


def inputs_to_dev(d, dev, dtype):
    """q/k/v in the compute dtype, beta/decay/h0 fp32 (values are exact in both)."""
    import torch
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    out = {n: to_dev(d[n], dev, tdt) for n in ("q", "k", "v")}
    for n in ("beta", "decay", "h0"):
        out[n] = to_dev(d.get(n), dev, torch.float32)
    if "cu_seqlens" in d:
        out["cu_seqlens"] = to_dev(d["cu_seqlens"], dev, torch.int32)
    return out


def to_np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)
