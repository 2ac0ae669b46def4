"""Failure detection without a GPU fault.

The tensor-core prefill bounds every wait (mbarrier phases, the publication flags between
its prep and chain roles) and records KDA_ERR_DEVICE_TIMEOUT in the workspace header when a
limit runs out.  kda_diag_wait_timeout runs those same waits against events that never
happen, with a short limit: the test checks that the time-out is reported once, that the
report is cleared by reading it, and that the context still runs a prefill correctly.
"""
import time

import pytest

from kda_inputs import make_custom
from _util import assert_parity, inputs_to_dev, to_np

pytestmark = pytest.mark.gpu

KDA_ERR_DEVICE_TIMEOUT = 8


@pytest.fixture(scope="module")
def kda():
    import delta_rule_linear_gb300 as m
    from delta_rule_linear_gb300 import build as b
    b.build()
    m.load()
    return m


def test_bounded_waits_report_and_recover(kda, oracle_mod):
    import torch
    dev = torch.device("cuda:0")
    ws = torch.zeros(4096, dtype=torch.uint8, device=dev)
    t0 = time.perf_counter()
    kda.diag_wait_timeout(ws, 2000)          # two waits of 2 ms each, nothing ever signals
    assert kda.query_device_error(ws) == KDA_ERR_DEVICE_TIMEOUT
    assert time.perf_counter() - t0 < 5.0    # the waits gave up: no hang
    assert kda.query_device_error(ws) == 0   # reading the report cleared it

    # the context is still usable: a tensor-core prefill right after is correct
    d = make_custom(1, 200, 4, 128, 128, dtype="bf16", decay="train", h0="normal002", seed=21)
    t = inputs_to_dev(d, dev, "bf16")
    o, h = kda.chunk_fwd(t["q"], t["k"], t["v"], t["beta"], t["decay"], t["h0"], check_device=True)
    ro, rh = oracle_mod.forward(d["q"], d["k"], d["v"], d["beta"], d["decay"], d["h0"])
    assert_parity("bf16", to_np(o), ro, to_np(h), rh, tag="after probe")


def test_probe_rejects_bad_arguments(kda):
    import torch
    from delta_rule_linear_gb300 import KdaError
    dev = torch.device("cuda:0")
    ws = torch.zeros(4096, dtype=torch.uint8, device=dev)
    for limit in (0, 2_000_001):
        with pytest.raises(KdaError) as ei:
            kda.diag_wait_timeout(ws, limit)
        assert ei.value.code == 2            # KDA_ERR_SHAPE
    with pytest.raises(KdaError) as ei:
        kda.diag_wait_timeout(ws[:128], 1000)
    assert ei.value.code == 6                # KDA_ERR_WORKSPACE
