"""kda_chunk_fwd_noalloc: the prefill for callers that cannot hand us device memory.

Such callers (a plugin inside a framework that owns the memory pool, code on a
latency-critical path where cudaMalloc would synchronise the device) call this entry
point, which keeps its scratch in one built-in array instead of a caller workspace.
These tests call it through the C ABI on several calls in a row with different inputs
and check each result against kda_chunk_fwd (the workspace entry point: the same kernels
on the same inputs, so the results must be identical bit for bit -- contents that the
array keeps from an earlier call must not leak into a later one) and against the oracle,
and read the array's error word after every call.  This file is collected last.
"""
import pytest

from kda_inputs import make_custom
from _util import assert_parity, inputs_to_dev, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kda():
    import delta_rule_linear_gb300 as m
    from delta_rule_linear_gb300 import build as b
    b.build()
    m.load()
    return m


def _check_case(kda, oracle_mod, dev, B, T, H, D, decay, h0, seed):
    import torch
    d = make_custom(B, T, H, D, D, dtype="bf16", decay=decay, h0=h0, seed=seed)
    t = inputs_to_dev(d, dev, "bf16")
    o_ref, h_ref = kda.chunk_fwd(t["q"], t["k"], t["v"], t["beta"], t["decay"], t["h0"],
                                 check_device=True)
    o, h = kda.chunk_fwd_noalloc(t["q"], t["k"], t["v"], t["beta"], t["decay"], t["h0"])
    torch.cuda.synchronize()
    assert kda.query_device_error(None) == 0, "a wait of the no-alloc call timed out"
    assert torch.equal(o, o_ref), f"o differs from the workspace call (B={B} T={T} H={H} D={D})"
    assert torch.equal(h, h_ref), f"final state differs from the workspace call (B={B} T={T} H={H} D={D})"
    ro, rh = oracle_mod.forward(d["q"], d["k"], d["v"], d["beta"], d["decay"], d["h0"])
    assert_parity("bf16", to_np(o), ro, to_np(h), rh, tag=f"noalloc B={B} T={T} H={H} D={D}")


def test_noalloc_matches_workspace_entry_point_and_oracle_on_consecutive_calls(kda, oracle_mod):
    import torch
    dev = torch.device("cuda:0")
    # one more (sequence, head) pair than a quarter of the SMs: more pairs than chains,
    # two rounds
    pairs = torch.cuda.get_device_properties(dev).multi_processor_count // 4 + 1
    H = next(h for h in (19, 17, 13, 11, 7, 5, 3, 2, 1) if pairs % h == 0)
    cases = [(1, 1000, 8, 128, "long", "normal002", 11),
             (2, 300, 4, 64, "train", "zero", 12),
             (pairs // H, 1100, H, 64, "train", "normal002", 13)]
    for B, T, H_, D, decay, h0, seed in cases:
        _check_case(kda, oracle_mod, dev, B, T, H_, D, decay, h0, seed)


def test_noalloc_serves_long_problems(kda, oracle_mod):
    """4096 (chunk, head) pairs at head dim 128: the scratch does not grow with the problem."""
    import torch
    _check_case(kda, oracle_mod, torch.device("cuda:0"), 1, 4096, 64, 128, "long", "normal002", 14)


def test_noalloc_refuses_unsupported_shapes(kda):
    import torch
    from delta_rule_linear_gb300 import KdaError
    dev = torch.device("cuda:0")
    q = torch.zeros(1, 64, 2, 32, dtype=torch.bfloat16, device=dev)   # head dim 32: not served
    beta = torch.zeros(1, 64, 2, dtype=torch.float32, device=dev)
    with pytest.raises(KdaError) as ei:
        kda.chunk_fwd_noalloc(q, q, q, beta)
    assert ei.value.code == 4   # KDA_ERR_UNSUPPORTED
