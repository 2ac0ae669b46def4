"""The multi-process path of the benchmark on CPU: two `gloo` ranks (127.0.0.1).

The method shards as independent problems (sequences and heads never exchange anything), so
N GPUs run N replicas with no data-path collective; the only cross-rank traffic is the
benchmark's barrier and the max over ranks of the timed region.  These tests run that
host logic with world_size 2 and check that a batch split across ranks gives, per rank,
exactly the oracle's result on the whole batch for its sequences (what the replicas rely
on), and that the reference arm does its work on rank 0 alone.
"""
import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
WORLD = 2


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, outdir):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    import bench
    import oracle
    import torch.distributed as dist
    from kda_inputs import make_custom

    w, r, _ = bench.dist_setup()
    assert (w, r) == (world, rank)
    assert dist.get_backend() == "gloo"
    bench.barrier(w)
    # the max over ranks of each rank's time
    m = bench.max_over_ranks(1.5 * (rank + 1), w)
    # this rank's shard of a 4-sequence batch: sequences [2 rank, 2 rank + 2)
    d = make_custom(2 * world, 40, 2, 16, 16, dtype="f32", decay="train", h0="normal002", seed=11)
    sl = slice(2 * rank, 2 * rank + 2)
    o, hT = oracle.forward(d["q"][sl], d["k"][sl], d["v"][sl], d["beta"][sl], d["decay"][sl], d["h0"][sl])
    # the reference arm: rank 0 prints one line, the other ranks return without work
    args = type("A", (), dict(steps=1, warmup=0, gpus=world))()
    buf = io.StringIO()
    if rank != 0:
        with redirect_stdout(buf):
            bench.run_reference(args, w, r)
    np.savez(os.path.join(outdir, f"rank{rank}.npz"), o=o, hT=hT, m=m, ref_out=buf.getvalue())
    bench.barrier(w)
    dist.destroy_process_group()


@pytest.fixture(scope="module")
def ranks(tmp_path_factory, oracle_mod):
    import torch.multiprocessing as mp
    out = tmp_path_factory.mktemp("ranks")
    mp.start_processes(_worker, args=(WORLD, _free_port(), str(out)), nprocs=WORLD, join=True,
                       start_method="spawn")
    return [dict(np.load(out / f"rank{r}.npz")) for r in range(WORLD)]


def test_max_over_ranks(ranks):
    for r in ranks:
        assert float(r["m"]) == pytest.approx(1.5 * WORLD)


def test_shards_match_the_whole_batch(ranks, oracle_mod):
    from kda_inputs import make_custom
    d = make_custom(2 * WORLD, 40, 2, 16, 16, dtype="f32", decay="train", h0="normal002", seed=11)
    o, hT = oracle_mod.forward(d["q"], d["k"], d["v"], d["beta"], d["decay"], d["h0"])
    np.testing.assert_array_equal(np.concatenate([r["o"] for r in ranks]), o)
    np.testing.assert_array_equal(np.concatenate([r["hT"] for r in ranks]), hT)


def test_reference_arm_rank0_only(ranks):
    assert str(ranks[1]["ref_out"]) == ""


def test_reference_arm_line_keys():
    """The line the reference arm prints on rank 0 (checked on a stub oracle timing)."""
    import bench
    args = type("A", (), dict(steps=1, warmup=0, gpus=1))()
    orig = bench.oracle_prefill_sample
    bench.oracle_prefill_sample = lambda d, heads, threads=0: (1000.0, 0.5, 4)
    orig_make = bench.make_prefill
    bench.make_prefill = lambda wl, seed=0: None
    try:
        buf = io.StringIO()
        with redirect_stdout(buf):
            bench.run_reference(args, 1, 0)
    finally:
        bench.oracle_prefill_sample = orig
        bench.make_prefill = orig_make
    line = json.loads(buf.getvalue().strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] == 1000.0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] == 4
    assert line["e2e"] == {"value": 1000.0, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}


def test_clock_summary_uses_the_timed_region():
    """The clock record: samples inside the region when there are any, else the ones around it;
    throttle reasons are read from the same samples."""
    import datetime
    import bench

    def line(t, mhz, thermal="Not Active", power="Not Active"):
        ts = datetime.datetime.fromtimestamp(t).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
        return (t, f"{ts}, {mhz}, 2070, 900.0, 0x0, Not Active, {thermal}, Not Active, {power}")

    c = bench.ClockSampler(0)
    c.t0, c.t1 = 1000.0, 1000.5
    c.lines = [line(999.9, 1500, thermal="Active"), line(1000.1, 2070), line(1000.3, 2060, power="Active"),
               line(1000.6, 1800)]
    s = c.summary()
    assert s["samples"] == 2 and s["sm_mhz"] == 2065 and s["reasons"] == ["sw_power_cap"]
    assert s["samples_where"] == "inside the timed region"
    c.t0, c.t1 = 1000.11, 1000.12   # shorter than the interval: the samples on either side
    s = c.summary()
    assert s["samples"] == 2 and s["sm_mhz"] == 2065 and "bracketing" in s["samples_where"]
