"""kda_chunk_fwd_noalloc: the prefill for callers that cannot hand us device memory.

Such callers (a plugin inside a framework that owns the memory pool, code on a
latency-critical path where cudaMalloc would synchronise the device) call this entry
point, which keeps its scratch in one built-in array instead of a caller workspace.
These tests call it through the C ABI and check it against kda_chunk_fwd (the
workspace entry point) on two calls in a row with different inputs, so that the
contents the array keeps from the first call cannot leak into the second, and that
a problem too big for the array is refused up front.  This file is collected last.
"""
import numpy as np
import pytest

from kda_inputs import make_custom
from _util import BF16_O, BF16_STATE_FROB, frob_rel, inputs_to_dev, max_rel, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kda():
    import delta_rule_linear_gb300 as m
    from delta_rule_linear_gb300 import build as b
    b.build()
    m.load()
    return m


def test_noalloc_matches_workspace_entry_point_on_consecutive_calls(kda):
    import torch
    dev = torch.device("cuda:0")
    cases = [((1, 1000, 8, 128), "long", "normal002", 11),
             ((2, 300, 4, 64), "train", "zero", 12),
             ((4, 70, 20, 64), "train", "normal002", 13)]   # B*H = 80: the two-launch path
    for (B, T, H, D), decay, h0, seed in cases:
        d = make_custom(B, T, H, D, D, dtype="bf16", decay=decay, h0=h0, seed=seed)
        t = inputs_to_dev(d, dev, "bf16")
        o_ref, h_ref = kda.chunk_fwd(t["q"], t["k"], t["v"], t["beta"], t["decay"], t["h0"],
                                     check_device=True)
        o, h = kda.chunk_fwd_noalloc(t["q"], t["k"], t["v"], t["beta"], t["decay"], t["h0"])
        torch.cuda.synchronize()
        assert max_rel(to_np(o), to_np(o_ref)) <= BF16_O
        assert frob_rel(to_np(h), to_np(h_ref)) <= BF16_STATE_FROB
        assert np.all(np.isfinite(to_np(o)))


def test_noalloc_refuses_problems_beyond_its_scratch(kda):
    import torch
    from delta_rule_linear_gb300 import KdaError
    dev = torch.device("cuda:0")
    # 16 chunks x 64 heads = 1024 (chunk, head) pairs of 72 KB > 64 MiB
    B, T, H, D = 1, 1024, 64, 128
    q = torch.zeros(B, T, H, D, dtype=torch.bfloat16, device=dev)
    beta = torch.zeros(B, T, H, dtype=torch.float32, device=dev)
    with pytest.raises(KdaError) as ei:
        kda.chunk_fwd_noalloc(q, q, q, beta)
    assert ei.value.code == 6   # KDA_ERR_WORKSPACE
