#!/usr/bin/env python3
"""Benchmark of the delta-rule linear-attention forward on GB300.

One JSON line on rank 0.  Headline (``value``): chunked prefill tokens/s on the
long-sequence workload (B=1, T=32768, H=32, dk=dv=128, bf16 q/k/v, fp32
state carried in from N(0, 0.02^2), decay = -softplus(N(-4,1)), chunk 64),
with the counted chunk-GEMM FLOPs reported against the bf16 tensor peak.  The
same line carries the decode workload (B=256, H=32, d=128, 128 single-token
steps over a 512 MiB fp32 state) as state GB/s against the HBM peak.

  python bench.py [--gpus N --steps K --warmup W] [--impl reference]

Under torchrun (N > 1) every rank runs its own independent copy of the
workload on its own GPU (different seed; heads are independent, no collective
on the data path) and rank 0 reports the aggregate over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from kda_inputs import (WORKLOADS, make_custom, make_decode_state, make_decode_step,  # noqa: E402
                        make_gate_params, make_gk, make_gk_decode_step, make_prefill, make_varlen)

METRIC = "prefill tokens/s & % bf16 TC peak; decode state GB/s vs HBM peak (1×GB300)"
NOMINAL_HBM_GBS = 8000.0
# Counters of one ncu capture per kernel (DRAM bytes read + written per launch, tensor-pipe
# activity) live in profiles/ncu_counters.txt together with a hash of the kernel's sources
# at capture time; a figure is reported only while those sources are unchanged (null
# otherwise), and `--record-counters` writes a new capture's figures there.
COUNTERS_FILE = os.path.join(ROOT, "profiles", "ncu_counters.txt")
COUNTER_SOURCES = {   # the sources each kernel's counters depend on
    "prefill": ["delta_rule_linear_gb300/csrc/chunk_tc.cu", "delta_rule_linear_gb300/csrc/tc_ptx.cuh"],
    "decode": ["delta_rule_linear_gb300/csrc/scan.cu"],
}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def sources_hash(kind):
    import hashlib
    h = hashlib.sha256()
    for rel in COUNTER_SOURCES[kind]:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(rel.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def recorded_counters(kind):
    """The recorded ncu figures of `kind` if its sources are unchanged since the capture:
    {"dram_bytes_per_launch", "tensor_pipe_active", "capture"}, else None."""
    try:
        with open(COUNTERS_FILE) as f:
            rec = json.load(f).get(kind)
    except (OSError, ValueError):
        return None
    if not rec or rec.get("sources") != sources_hash(kind):
        return None
    return rec


KEPT_METRICS = ("dram__bytes_read.sum", "dram__bytes_write.sum",
                "sm__pipe_tensor_cycles_active.avg.pct_of_peak_sustained_active")


def _capture_metrics(csv_path, kernel_regex):
    """{launch: {metric: value}} for the DRAM-byte and tensor-pipe metrics of the launches
    of kernels matching kernel_regex in an ncu --csv file (raw page or --metrics list)."""
    import csv
    import re
    rows = list(csv.reader(open(csv_path, newline="")))
    head_i = next(i for i, r in enumerate(rows) if "Kernel Name" in r)
    head = rows[head_i]
    kcol = head.index("Kernel Name")
    launches = {}
    if "Metric Name" in head:   # --metrics list: one row per (launch, metric)
        idcol, mcol, vcol = head.index("ID"), head.index("Metric Name"), head.index("Metric Value")
        for r in rows[head_i + 1:]:
            if len(r) > vcol and re.search(kernel_regex, r[kcol]):
                launches.setdefault(r[idcol], {})[r[mcol]] = float(r[vcol].replace(",", ""))
    else:                       # raw page: one row per launch, one column per metric, a units row
        units = rows[head_i + 1]
        mult = {"byte": 1.0, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9}
        for n, r in enumerate(rows[head_i + 2:]):
            if len(r) > kcol and re.search(kernel_regex, r[kcol]):
                launches[n] = {m: float(r[i].replace(",", "")) * mult.get(units[i], 1.0)
                               for i, m in enumerate(head) if m in KEPT_METRICS and r[i].strip()}
    return {k: {m: v for m, v in l.items() if m in KEPT_METRICS} for k, l in launches.items()}


def record_counters(kind, csv_path, kernel_regex, scale=1.0, note="", tensor_csv=None):
    """Parse an ncu --csv capture (raw page or --metrics list), average the DRAM bytes and
    tensor-pipe activity over the launches of the kernels matching `kernel_regex`, scale
    the bytes to one full launch (`scale`: units of the full launch / units captured) and
    store them with the current hash of the kernel's sources.  `tensor_csv`: a second
    capture (e.g. a full set on a smaller case) that supplies the tensor-pipe activity."""
    import csv
    import re
    if tensor_csv:
        tp_only = _capture_metrics(tensor_csv, kernel_regex)
    launches = _capture_metrics(csv_path, kernel_regex)
    if not launches:
        raise SystemExit(f"no launch of {kernel_regex!r} in {csv_path}")
    rd = [l.get("dram__bytes_read.sum", 0.0) + l.get("dram__bytes_write.sum", 0.0) for l in launches.values()]
    tp = [l[m] for l in (tp_only if tensor_csv else launches).values() for m in l
          if m.startswith("sm__pipe_tensor_cycles_active")]
    try:
        with open(COUNTERS_FILE) as f:
            allrec = json.load(f)
    except (OSError, ValueError):
        allrec = {}
    allrec[kind] = {"sources": sources_hash(kind),
                    "dram_bytes_per_launch": statistics.mean(rd) * scale if any(rd) else None,
                    "tensor_pipe_active": (statistics.mean(tp) / 100.0) if tp else None,
                    "launches_captured": len(launches), "scale_to_full_launch": scale,
                    "capture": note}
    with open(COUNTERS_FILE, "w") as f:
        json.dump(allrec, f, indent=1, sort_keys=True)
        f.write("\n")
    print(json.dumps(allrec[kind]))


def headline_config(wl, world):
    """The config dict both arms print for the headline workload."""
    return {"workload": wl.name, "B": wl.B, "T": wl.T, "H": wl.H, "dk": wl.dk,
            "dv": wl.dv, "chunk_size": wl.chunk, "state": "fp32 carried in",
            "l2_flush": "none: inputs (805 MB) and decode state (512 MiB) exceed L2",
            "parallelism": f"replicas x{world}"}


def counted_prefill_flops(B, T, H, dk, dv, C):
    """Chunk-GEMM FLOPs counted per token-head: 2C(3dk + 2dv) + 6 dk dv
    (Gram/scores/WY products at chunk C with triangular products counted dense,
    plus the three state products), times B*T*H."""
    return float(B) * T * H * (2 * C * (3 * dk + 2 * dv) + 6 * dk * dv)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle sampling around the timed region.

    Sampling starts (and the first sample is awaited) before the region opens and goes on
    until a sample after it has arrived; every sample carries nvidia-smi's timestamp, and
    the summary uses the samples taken inside the region (host wall clock marks set by
    `begin()` / `end()`), or, when the region is shorter than the sampling interval, the
    samples that bracket it, and says which."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    INTERVAL_MS = 20

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []   # (host time received, line)
        self.t0 = self.t1 = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.INTERVAL_MS)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True, bufsize=1)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            self._await(1, 5.0)   # sampling is live before the region opens
        except Exception:
            self.proc = None
        self.begin()
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def _await(self, n, timeout):
        t = time.time() + timeout
        while len(self.lines) < n and time.time() < t and self.proc.poll() is None:
            time.sleep(0.002)

    def begin(self):
        self.t0 = time.time()

    def end(self):
        self.t1 = time.time()

    def __exit__(self, *a):
        if self.t1 is None:
            self.end()
        if self.proc is not None:
            self._await(len(self.lines) + 1, 1.0)   # a sample after the region
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.thread.join(timeout=2)

    @staticmethod
    def _stamp(text):
        import datetime
        try:
            return datetime.datetime.strptime(text.strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
        except ValueError:
            return None

    def summary(self):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        rows = []
        for recv, ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((self._stamp(parts[0]) or recv, float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        inside = [r for r in rows if self.t0 is not None and self.t0 <= r[0] <= self.t1]
        if inside:
            use, where = inside, "inside the timed region"
        else:   # the region is shorter than the interval: the samples just before and after it
            before = [r for r in rows if r[0] < (self.t0 or 0)][-1:]
            after = [r for r in rows if r[0] > (self.t1 or 0)][:1]
            use, where = before + after, "bracketing the timed region (shorter than the sampling interval)"
        reasons = sorted({nm for r in use for nm, val in zip(names, r[3]) if val.lower() == "active"})
        return {"sm_mhz": statistics.median([r[1] for r in use]) if use else None,
                "sm_max_mhz": use[-1][2] if use else None, "reasons": reasons,
                "samples": len(use), "samples_where": where,
                "region_ms": round(1e3 * (self.t1 - self.t0), 1) if self.t0 and self.t1 else None,
                "interval_ms": self.INTERVAL_MS}


def dist_setup():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def pin_to_gpu_cpus(index):
    """Run this process on the CPUs beside GPU `index` (the local_cpulist of its PCI device),
    so that pinned host buffers allocated afterwards sit in the memory node next to the GPU:
    the host-device copy rate depends on it.  Returns the CPU list in use ("unchanged" when
    the list cannot be read or covers every allowed CPU)."""
    try:
        bus_id = subprocess.run(["nvidia-smi", "-i", str(index), "--query-gpu=pci.bus_id",
                                 "--format=csv,noheader"], capture_output=True, text=True,
                                timeout=30).stdout.strip()
        dom, bus, rest = bus_id.split(":")
        path = f"/sys/bus/pci/devices/{int(dom, 16):04x}:{bus.lower()}:{rest.lower()}/local_cpulist"
        with open(path) as f:
            spec = f.read().strip()
        cpus = set()
        for part in spec.split(","):
            lo, _, hi = part.partition("-")
            cpus.update(range(int(lo), int(hi or lo) + 1))
        allowed = os.sched_getaffinity(0)
        cpus &= allowed
        if not cpus or cpus == allowed:
            return "unchanged"
        os.sched_setaffinity(0, cpus)
        return spec
    except Exception:
        return "unchanged"


def to_dev(x, dev, dtype):
    import torch
    return None if x is None else torch.from_numpy(np.ascontiguousarray(x)).to(dev, dtype)


# --------------------------------------------------------------------------- prefill
def prefill_workload(args):
    """The long-sequence workload, or the same with T overridden (profiling captures only)."""
    wl = WORKLOADS[3]
    if args.prefill_T:
        wl = dataclasses.replace(wl, T=args.prefill_T, name=f"{wl.name} [T overridden: {args.prefill_T}]")
    return wl


# Kernels of ours per call.  The tensor-core prefill is one cooperative launch of tc_kernel
# (its ring flags are cleared by a cudaMemsetAsync, not a kernel of ours); packed varlen adds
# the kernel that orders the sequences longest first; the chunked backward is three launches
# (the forward keeping every chunk's map and state, the reverse walk, the chunk-local
# gradients); the token-by-token backward is three (checkpoints, reverse walk, finish).
TC_PREFILL_LAUNCHES, VARLEN_LAUNCHES, CHUNK_BWD_LAUNCHES, RECURRENT_BWD_LAUNCHES = 1, 2, 3, 3
GK_CHUNK_BWD_LAUNCHES = 4   # kept-map forward, reverse walk, chunk-parallel token walks, q/k finish


def prefill_min_bytes(tokens, H, dk, dv, has_decay, nseq, h0_in):
    """Bytes a prefill call cannot avoid: q, k, v read and o written once (bf16), beta (and
    the decay) read once, the final state written (and the initial state read) once."""
    per_token_head = (2 * dk + 2 * dv) * 2 + 4 + (4 if has_decay else 0)
    return tokens * H * per_token_head + nseq * H * dk * dv * 4 * (2 if h0_in else 1)


def memory_ceiling(flops, min_bytes, ms, peaks):
    """How the call stands against HBM: the achieved bandwidth on its minimum bytes as a
    fraction of the measured HBM peak, and the tensor fraction it could reach at most if it
    moved exactly those bytes at that peak (the FLOP time over the larger of the FLOP and
    byte times)."""
    t_flops = flops / (peaks["bf16_tflops"] * 1e12)
    t_bytes = min_bytes / (peaks["hbm_gbs"] * 1e9)
    return {"min_bytes": int(min_bytes),
            "hbm_frac_of_min_bytes": round(min_bytes / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 5),
            "tc_frac_ceiling_at_hbm_peak": round(t_flops / max(t_flops, t_bytes), 4)}


def bench_prefill(args, world, rank, dev, peaks, d):
    import torch
    import delta_rule_linear_gb300 as kda

    wl = prefill_workload(args)
    q, k, v = (to_dev(d[n], dev, torch.bfloat16) for n in ("q", "k", "v"))
    beta, decay, h0 = (to_dev(d[n], dev, torch.float32) for n in ("beta", "decay", "h0"))
    B, T, H, dk, dv, C = wl.B, wl.T, wl.H, wl.dk, wl.dv, wl.chunk
    o = torch.empty((B, T, H, dv), dtype=torch.bfloat16, device=dev)
    hT = torch.empty((B, H, dk, dv), dtype=torch.float32, device=dev)
    from delta_rule_linear_gb300 import _lib
    ws = torch.empty(_lib.chunk_fwd_workspace_bytes(B, T, H, dk, dv, C, _lib.KDA_BF16),
                     dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        kda.chunk_fwd(q, k, v, beta, decay, h0, chunk_size=C, out=o, final_state=hT,
                      workspace=ws, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index) as clk:
        clk.begin()
        ev0.record(stream)
        for _ in range(args.steps):
            step()
        ev1.record(stream)
        torch.cuda.synchronize()
        clk.end()
    barrier(world)
    ms = ev0.elapsed_time(ev1) / args.steps
    ms_max = max_over_ranks(ms, world)
    if kda.query_device_error(ws) != 0:
        raise RuntimeError("device error recorded during the prefill benchmark")

    # End to end through the C ABI with host buffers: every step copies its inputs from
    # pinned host memory, runs the kernels and reads o and the final state back.  Steps are
    # pipelined over three streams (H2D, compute, D2H) with two device buffer sets, so that
    # step i's read-back and step i+1's upload (opposite copy directions) and step i's
    # kernels overlap; every byte of every step still crosses the link inside the timed
    # region.
    host_cpus = pin_to_gpu_cpus(dev.index if dev.index is not None else 0)
    pin = lambda x: x.cpu().pin_memory()  # noqa: E731
    hin = [pin(x) for x in (q, k, v, beta, decay, h0)]
    hout = [[torch.empty_like(x, device="cpu").pin_memory() for x in (o, hT)] for _ in range(2)]
    din = [[torch.empty_like(x) for x in (q, k, v, beta, decay, h0)] for _ in range(2)]
    dout = [[torch.empty_like(x) for x in (o, hT)] for _ in range(2)]
    h2d = sum(x.numel() * x.element_size() for x in hin)
    d2h = sum(x.numel() * x.element_size() for x in hout[0])
    s_h2d, s_d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    freed = [None, None]   # per buffer set: the event after which its inputs/outputs are free

    def e2e_step(i):
        j = i & 1
        if freed[j] is not None:
            s_h2d.wait_event(freed[j])
        with torch.cuda.stream(s_h2d):
            for dst, src in zip(din[j], hin):
                dst.copy_(src, non_blocking=True)
        up = torch.cuda.Event()
        up.record(s_h2d)
        stream.wait_event(up)
        dq, dk_, dv_, db, dd, dh0 = din[j]
        kda.chunk_fwd(dq, dk_, dv_, db, dd, dh0, chunk_size=C, out=dout[j][0],
                      final_state=dout[j][1], workspace=ws, stream=stream)
        done = torch.cuda.Event()
        done.record(stream)
        s_d2h.wait_event(done)
        with torch.cuda.stream(s_d2h):
            for dst, src in zip(hout[j], dout[j]):
                dst.copy_(src, non_blocking=True)
        back = torch.cuda.Event()
        back.record(s_d2h)
        freed[j] = back

    e2e_steps = max(3, min(args.steps, 10))
    e2e_step(0)
    torch.cuda.synchronize()
    freed[0] = freed[1] = None
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_h2d)
    stream.wait_stream(s_h2d)
    for i in range(e2e_steps):
        e2e_step(i)
    stream.wait_stream(s_d2h)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, world)

    tokens = B * T
    flops = counted_prefill_flops(B, T, H, dk, dv, C)
    peak_tf = peaks["bf16_tflops"]
    achieved_tf = flops / (ms * 1e-3) / 1e12
    min_bytes = B * T * H * (2 * dk + 2 * dv) * 2 + B * T * H * 8 + 2 * B * H * dk * dv * 4
    ctr = recorded_counters("prefill") if not args.prefill_T else None
    return {
        "ms": ms_max, "tokens_per_s": tokens * world / (ms_max * 1e-3),
        "clocks": clk.summary(),
        "roofline": {"bound": "tensor", "achieved": round(achieved_tf, 3), "peak": peak_tf,
                     "unit": "TFLOP/s", "frac": round(achieved_tf / peak_tf, 5),
                     "traffic": (ctr or {}).get("dram_bytes_per_launch"),
                     "traffic_capture": (ctr or {}).get("capture", "none for the kernel as built"),
                     "kernel": "tc_kernel (the whole step: one launch holds the prep groups and the chains)",
                     "flops_per_launch": flops,
                     "recurrence_min_flops": 6.0 * B * T * H * dk * dv,
                     "ncu_tensor_pipe_active": (ctr or {}).get("tensor_pipe_active"),
                     "hbm_frac_of_min_bytes": round(min_bytes / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 5)},
        "e2e": {"value": tokens * world / (e2e_ms * 1e-3), "unit": "tokens/s",
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "ms_per_step": e2e_ms, "steps": e2e_steps,
                "pipelining": "H2D, kernels and D2H on three streams, two buffer sets",
                "host_cpus": host_cpus},
        "gpu_launches": args.steps * TC_PREFILL_LAUNCHES,
        "shape": dict(B=B, T=T, H=H, dk=dk, dv=dv, chunk=C),
    }


# --------------------------------------------------------------------------- other prefill configs
SECONDARY_PARTS = ("tiny", "training", "backward", "gated", "varlen")


def bench_secondary(args, world, rank, dev, peaks, parts=SECONDARY_PARTS):
    """The tiny fp32 workload (1, the CUDA-core chunk path), the training-shape prefill
    (workload 2) and its backward, the long-sequence prefill with the gate prologues, and the
    packed varlen prefill (workload 5), reported beside the headline: tokens/s and counted
    FLOPs against the bf16 peak.  `parts` selects a subset (profiling captures)."""
    import torch
    import delta_rule_linear_gb300 as kda
    from delta_rule_linear_gb300 import _lib
    stream = torch.cuda.current_stream()
    out = {}

    def timed(step):
        for _ in range(args.warmup):
            step()
        torch.cuda.synchronize()
        barrier(world)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        return max_over_ranks(e0.elapsed_time(e1) / args.steps, world)

    if "tiny" in parts:
        tiny_prefill(out, timed, kda, _lib, rank, dev, stream, world)
    wl = WORKLOADS[2]
    d = make_prefill(wl, seed=rank)
    q, k, v = (to_dev(d[n], dev, torch.bfloat16) for n in ("q", "k", "v"))
    beta, decay = (to_dev(d[n], dev, torch.float32) for n in ("beta", "decay"))
    o = torch.empty_like(v)
    hT = torch.empty((wl.B, wl.H, wl.dk, wl.dv), dtype=torch.float32, device=dev)
    ws = torch.empty(_lib.chunk_fwd_workspace_bytes(wl.B, wl.T, wl.H, wl.dk, wl.dv, wl.chunk,
                                                    _lib.KDA_BF16), dtype=torch.uint8, device=dev)
    if "training" in parts:
        training_prefill(out, timed, kda, wl, q, k, v, beta, decay, o, hT, ws, stream, world, peaks)
    if "backward" in parts:
        training_backward(out, timed, kda, _lib, wl, q, k, v, beta, decay, o, stream, dev, world)
    del q, k, v, beta, decay, o, hT, ws
    if "gated" in parts:
        gated_prefill(out, timed, kda, _lib, rank, dev, stream, world)
    if "varlen" in parts:
        varlen_prefill(out, timed, kda, _lib, rank, dev, stream, world, peaks)
    return out


def tiny_prefill(out, timed, kda, _lib, rank, dev, stream, world):
    """Workload 1: fp32, B=1 T=64 H=2 d=32, chunk 16 -- the CUDA-core chunk path."""
    import torch
    wl = WORKLOADS[1]
    d = make_prefill(wl, seed=rank)
    q, k, v, beta, decay = (to_dev(d[n], dev, torch.float32) for n in ("q", "k", "v", "beta", "decay"))
    o = torch.empty_like(v)
    hT = torch.empty((wl.B, wl.H, wl.dk, wl.dv), dtype=torch.float32, device=dev)
    ws = torch.empty(max(256, _lib.chunk_fwd_workspace_bytes(wl.B, wl.T, wl.H, wl.dk, wl.dv, wl.chunk,
                                                             _lib.KDA_F32)), dtype=torch.uint8, device=dev)
    ms = timed(lambda: kda.chunk_fwd(q, k, v, beta, decay, None, chunk_size=wl.chunk, out=o,
                                     final_state=hT, workspace=ws, stream=stream))
    out["tiny_prefill"] = {
        "workload": wl.name, "ms_per_call": ms, "tokens_per_s": wl.B * wl.T * world / (ms * 1e-3),
        "gpu_launches_per_call": 1, "note": "fp32 CUDA-core chunk path (chunk_simt_kernel): launch-bound at this size"}


def training_prefill(out, timed, kda, wl, q, k, v, beta, decay, o, hT, ws, stream, world, peaks):
    ms = timed(lambda: kda.chunk_fwd(q, k, v, beta, decay, None, chunk_size=wl.chunk, out=o,
                                     final_state=hT, workspace=ws, stream=stream))
    flops = counted_prefill_flops(wl.B, wl.T, wl.H, wl.dk, wl.dv, wl.chunk)
    out["training_prefill"] = {
        "workload": wl.name, "ms_per_call": ms, "tokens_per_s": wl.B * wl.T * world / (ms * 1e-3),
        "tc_frac": round(flops / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"], 5),
        **memory_ceiling(flops, prefill_min_bytes(wl.B * wl.T, wl.H, wl.dk, wl.dv, True, wl.B, False), ms, peaks),
        "gpu_launches_per_call": TC_PREFILL_LAUNCHES}


def training_backward(out, timed, kda, _lib, wl, q, k, v, beta, decay, o, stream, dev, world):
    import torch
    # the backward of the same call (one decay per head): gradients for q, k, v, beta, the
    # decay and the initial state, by chunks on the tensor cores and token by token
    d_o = torch.randn_like(o)
    h0z = torch.zeros((wl.B, wl.H, wl.dk, wl.dv), dtype=torch.float32, device=dev)
    wsc = torch.empty(_lib.load().kda_chunk_bwd_workspace(wl.B, wl.T, wl.H, wl.dk, wl.dv),
                      dtype=torch.uint8, device=dev)
    cms = timed(lambda: kda.chunk_bwd(q, k, v, beta, decay, h0z, d_o, None, workspace=wsc, stream=stream))
    out["training_backward"] = {
        "workload": wl.name + ", backward", "ms_per_call": cms,
        "tokens_per_s": wl.B * wl.T * world / (cms * 1e-3), "gpu_launches_per_call": CHUNK_BWD_LAUNCHES,
        "workspace_bytes": int(wsc.numel()),
        "note": "chunked on the tensor cores: the forward keeping every chunk's map and state, "
                "the reverse walk over the maps (state gradients), the chunk-local gradients of q, "
                "k, v, beta and the decay (tf32 warp MMAs, persistent CTAs)"}
    del wsc
    wsb = torch.empty(_lib.load().kda_recurrent_bwd_workspace(wl.B, wl.T, wl.H, wl.dk, wl.dv),
                      dtype=torch.uint8, device=dev)
    bms = timed(lambda: kda.recurrent_bwd(q, k, v, beta, decay, h0z, d_o, None, workspace=wsb,
                                          stream=stream))
    out["training_backward_recurrent"] = {
        "workload": wl.name + ", backward", "ms_per_call": bms,
        "tokens_per_s": wl.B * wl.T * world / (bms * 1e-3), "gpu_launches_per_call": RECURRENT_BWD_LAUNCHES,
        "note": "token by token on CUDA cores: 32-token checkpoints, recompute, reverse walk"}
    del d_o, h0z, wsb


def gated_prefill(out, timed, kda, _lib, rank, dev, stream, world):
    import torch
    # the long-sequence workload with the prologues in the kernel: decay from a raw gate
    # (kda_decay), beta from logits (sigmoid), the decayed read
    wl = WORKLOADS[3]
    d = make_prefill(wl, seed=rank)
    gate, A_log, dt_bias = make_gate_params((wl.B, wl.T, wl.H), wl.H, seed=rank)
    q, k, v = (to_dev(d[n], dev, torch.bfloat16) for n in ("q", "k", "v"))
    braw = to_dev(((2.0 * d["beta"] - 1.0) * 3).astype(np.float32), dev, torch.float32)
    graw, al, db, h0 = (to_dev(x, dev, torch.float32) for x in (gate, A_log, dt_bias, d["h0"]))
    o = torch.empty_like(v)
    hT = torch.empty((wl.B, wl.H, wl.dk, wl.dv), dtype=torch.float32, device=dev)
    ws = torch.empty(_lib.chunk_fwd_workspace_bytes(wl.B, wl.T, wl.H, wl.dk, wl.dv, wl.chunk,
                                                    _lib.KDA_BF16), dtype=torch.uint8, device=dev)
    ms = timed(lambda: kda.chunk_fwd(q, k, v, braw, graw, h0, chunk_size=wl.chunk, out=o,
                                     final_state=hT, workspace=ws, stream=stream, decayed_read=True,
                                     A_log=al, dt_bias=db, beta_sigmoid=True))
    out["gated_long_prefill"] = {
        "workload": wl.name + ", raw gate + beta logits + decayed read in the kernel",
        "ms_per_call": ms, "tokens_per_s": wl.B * wl.T * world / (ms * 1e-3),
        "gpu_launches_per_call": TC_PREFILL_LAUNCHES}
    del q, k, v, braw, graw, al, db, h0, o, hT, ws


def varlen_prefill(out, timed, kda, _lib, rank, dev, stream, world, peaks):
    import torch
    wl = WORKLOADS[5]
    d = make_varlen(wl, seed=rank)
    q, k, v = (to_dev(d[n], dev, torch.bfloat16) for n in ("q", "k", "v"))
    beta = to_dev(d["beta"], dev, torch.float32)
    cu_cpu = torch.from_numpy(d["cu_seqlens"])
    cu = cu_cpu.to(dev)
    N, total = len(d["cu_seqlens"]) - 1, int(d["cu_seqlens"][-1])
    o = torch.empty_like(v)
    hT = torch.empty((N, wl.H, wl.dk, wl.dv), dtype=torch.float32, device=dev)
    ws = torch.empty(_lib.varlen_fwd_workspace_bytes(N, total, wl.H, wl.dk, wl.dv, wl.chunk,
                                                     _lib.KDA_BF16), dtype=torch.uint8, device=dev)
    ms = timed(lambda: kda.varlen_fwd(q, k, v, beta, cu, None, None, cu_seqlens_cpu=cu_cpu,
                                      chunk_size=wl.chunk, out=o, final_state=hT, workspace=ws,
                                      stream=stream))
    flops = counted_prefill_flops(1, total, wl.H, wl.dk, wl.dv, wl.chunk)
    out["varlen_prefill"] = {
        "workload": wl.name, "tokens": total, "ms_per_call": ms,
        "tokens_per_s": total * world / (ms * 1e-3),
        "tc_frac": round(flops / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"], 5),
        **memory_ceiling(flops, prefill_min_bytes(total, wl.H, wl.dk, wl.dv, False, N, False), ms, peaks),
        "gpu_launches_per_call": VARLEN_LAUNCHES}


# --------------------------------------------------------------------------- per-channel decay
def bench_gk_chunk(args, world, rank, dev, peaks, out, D, e0, e1, long_only):
    """Per-channel chunked prefill (tensor cores) at the long-sequence and training shapes."""
    import torch
    import delta_rule_linear_gb300 as kda
    stream = torch.cuda.current_stream()
    from delta_rule_linear_gb300 import _lib
    shapes = [("gk_chunk_prefill_long", (1, args.prefill_T or 32768, 32)),
              ("gk_chunk_prefill_training", (2, 2048, 16))]
    if long_only:
        shapes = shapes[:1]
    for name, (Bp, T, Hp) in shapes:
        d = make_gk(Bp, T, Hp, D, D, dtype="bf16", gate_scale=0.01, h0="normal002", seed=rank)
        q, k, v = (to_dev(d[n], dev, torch.bfloat16) for n in ("q", "k", "v"))
        beta, g, h0 = (to_dev(d[n], dev, torch.float32) for n in ("beta", "g", "h0"))
        o = torch.empty_like(v)
        hT = torch.empty((Bp, Hp, D, D), dtype=torch.float32, device=dev)
        ws = torch.empty(_lib.chunk_fwd_workspace_bytes(Bp, T, Hp, D, D, 64, _lib.KDA_BF16),
                         dtype=torch.uint8, device=dev)

        def cstep():
            kda.gk_chunk_fwd(q, k, v, beta, g, h0, decayed_read=True, out=o, final_state=hT,
                             workspace=ws, stream=stream)

        for _ in range(args.warmup):
            cstep()
        torch.cuda.synchronize()
        barrier(world)
        e0.record(stream)
        for _ in range(args.steps):
            cstep()
        e1.record(stream)
        torch.cuda.synchronize()
        ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world)
        if kda.query_device_error(ws) != 0:
            raise RuntimeError("device error recorded during the per-channel prefill benchmark")
        flops = counted_prefill_flops(Bp, T, Hp, D, D, 64)
        out[name] = {
            "shape": dict(B=Bp, T=T, H=Hp, dk=D, dv=D, chunk=64), "decayed_read": True,
            "ms_per_call": ms, "tokens_per_s": Bp * T * world / (ms * 1e-3),
            "tc_frac": round(flops / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"], 5),
            "gpu_launches_per_call": TC_PREFILL_LAUNCHES}
        del q, k, v, beta, g, h0, o, hT, ws
    return out


def bench_gk(args, world, rank, dev, peaks):
    """Per-key-channel decay (TileOPs KDAFwdOp, g [B,T,H,K] = -0.01 U[0,1), the draw of the
    kda-neuron-kernels README's examples): the batched decode step at the decode workload's
    shape (HBM-bound: the fp32 state in and out), and the token-by-token prefill at the
    training shape."""
    import torch
    import delta_rule_linear_gb300 as kda
    stream = torch.cuda.current_stream()
    out = {}

    B, H, D, nsteps = 256, 32, 128, 32
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if args.only == "gk_prefill":   # profiling: the long-sequence chunked prefill alone
        return bench_gk_chunk(args, world, rank, dev, peaks, out, D, e0, e1, long_only=True)
    rng = np.random.Generator(np.random.PCG64([rank, 7]))
    state = torch.from_numpy((0.02 * rng.standard_normal((B, H, D, D), dtype=np.float32))).to(dev)
    toks = []
    for s in range(nsteps):
        st = make_gk_decode_step(B, H, D, D, s, dtype="bf16", gate_scale=0.01, seed=rank)
        toks.append(tuple(to_dev(st[n], dev, torch.bfloat16) for n in ("q", "k", "v")) +
                    tuple(to_dev(st[n], dev, torch.float32) for n in ("beta", "g")))
    o = torch.empty((B, 1, H, D), dtype=torch.bfloat16, device=dev)

    def run(n):
        for s in range(n):
            q, k, v, b, g = toks[s % nsteps]
            kda.gk_decode_step(q, k, v, b, g, state, decayed_read=True, out=o, stream=stream)

    run(3)
    torch.cuda.synchronize()
    barrier(world)
    e0.record(stream)
    run(nsteps)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1) / nsteps, world)
    nbytes = 2.0 * B * H * D * D * 4 + B * H * D * 4      # state in + out, and g
    gbs = nbytes / (ms * 1e-3) / 1e9
    out["gk_decode"] = {
        "shape": dict(B=B, H=H, dk=D, dv=D), "decayed_read": True, "ms_per_step": ms,
        "steps": nsteps, "gpu_launches": nsteps,
        "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": round(gbs / peaks["hbm_gbs"], 4),
                     "bytes_per_launch": nbytes}}

    bench_gk_chunk(args, world, rank, dev, peaks, out, D, e0, e1, long_only=False)

    Bp, T, Hp = 2, 2048, 16
    d = make_gk(Bp, T, Hp, D, D, dtype="bf16", gate_scale=0.01, seed=rank)
    q, k, v = (to_dev(d[n], dev, torch.bfloat16) for n in ("q", "k", "v"))
    beta, g = (to_dev(d[n], dev, torch.float32) for n in ("beta", "g"))
    o = torch.empty_like(v)
    hT = torch.empty((Bp, Hp, D, D), dtype=torch.float32, device=dev)
    nrep = max(1, min(args.steps, 5))

    def step():
        kda.gk_recurrent_fwd(q, k, v, beta, g, None, decayed_read=True, out=o, final_state=hT,
                             stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    barrier(world)
    e0.record(stream)
    for _ in range(nrep):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1) / nrep, world)
    # the backward of the same call: gradients for q, k, v, beta, g and the initial state
    d_o = torch.randn_like(o)
    gates = to_dev(d["g"], dev, torch.float32)
    h0z = torch.zeros((Bp, Hp, D, D), dtype=torch.float32, device=dev)
    from delta_rule_linear_gb300 import _lib
    wsb = torch.empty(_lib.load().kda_gk_recurrent_bwd_workspace(Bp, T, Hp, D, D), dtype=torch.uint8,
                      device=dev)

    def bstep():
        kda.gk_recurrent_bwd(q, k, v, beta, gates, h0z, d_o, None, decayed_read=True, workspace=wsb,
                             stream=stream)

    bstep()
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(nrep):
        bstep()
    e1.record(stream)
    torch.cuda.synchronize()
    bms = max_over_ranks(e0.elapsed_time(e1) / nrep, world)
    out["gk_recurrent_bwd"] = {
        "shape": dict(B=Bp, T=T, H=Hp, dk=D, dv=D), "decayed_read": True, "ms_per_call": bms,
        "tokens_per_s": Bp * T * world / (bms * 1e-3), "calls": nrep, "gpu_launches_per_call": RECURRENT_BWD_LAUNCHES,
        "note": "token by token on CUDA cores: 32-token checkpoints, recompute, reverse walk"}
    del wsb
    wsc = torch.empty(_lib.load().kda_gk_chunk_bwd_workspace(Bp, T, Hp, D, D), dtype=torch.uint8,
                      device=dev)

    def cstep():
        kda.gk_chunk_bwd(q, k, v, beta, gates, h0z, d_o, None, decayed_read=True, workspace=wsc,
                         stream=stream)

    for _ in range(max(1, args.warmup)):
        cstep()
    torch.cuda.synchronize()
    crep = max(1, min(args.steps, 10))
    e0.record(stream)
    for _ in range(crep):
        cstep()
    e1.record(stream)
    torch.cuda.synchronize()
    cms = max_over_ranks(e0.elapsed_time(e1) / crep, world)
    out["gk_chunk_bwd"] = {
        "shape": dict(B=Bp, T=T, H=Hp, dk=D, dv=D), "decayed_read": True, "ms_per_call": cms,
        "tokens_per_s": Bp * T * world / (cms * 1e-3), "calls": crep,
        "gpu_launches_per_call": GK_CHUNK_BWD_LAUNCHES, "workspace_bytes": int(wsc.numel()),
        "note": "the forward keeping every chunk's per-channel map and state and the reverse walk "
                "over the maps on the tensor cores, then every 64-token chunk's token walk at once "
                "(CUDA cores, persistent CTAs)"}
    del wsc
    out["gk_recurrent_prefill"] = {
        "shape": dict(B=Bp, T=T, H=Hp, dk=D, dv=D), "decayed_read": True, "ms_per_call": ms,
        "tokens_per_s": Bp * T * world / (ms * 1e-3), "calls": nrep, "gpu_launches_per_call": 1,
        "note": "CUDA-core token-by-token scan (latency-bound per token)"}
    return out


# --------------------------------------------------------------------------- layouts
def bench_layouts(args, world, rank, dev, peaks):
    """Layout options: the decode step with value-major states (TileOPs state_v_first) at the
    decode workload's shape, against the HBM roofline; and the training-shape prefill with
    grouped value heads (4 q/k heads, 16 value heads)."""
    import torch
    import delta_rule_linear_gb300 as kda
    from delta_rule_linear_gb300 import _lib
    stream = torch.cuda.current_stream()
    out = {}
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    wl = WORKLOADS[4]
    state = to_dev(np.ascontiguousarray(np.swapaxes(make_decode_state(wl, seed=rank), -1, -2)), dev,
                   torch.float32)
    nsteps = 32
    toks = []
    for s_ in range(nsteps):
        st = make_decode_step(wl, s_, seed=rank)
        toks.append(tuple(to_dev(st[n], dev, torch.bfloat16) for n in ("q", "k", "v")) +
                    tuple(to_dev(st[n], dev, torch.float32) for n in ("beta", "decay")))
    o = torch.empty((wl.B, 1, wl.H, wl.dv), dtype=torch.bfloat16, device=dev)

    def run(n):
        for i in range(n):
            q, k, v, b, g = toks[i % nsteps]
            kda.decode_step(q, k, v, b, g, state, out=o, stream=stream, state_v_first=True)

    run(3)
    torch.cuda.synchronize()
    barrier(world)
    e0.record(stream)
    run(nsteps)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1) / nsteps, world)
    nbytes = 2.0 * wl.B * wl.H * wl.dk * wl.dv * 4
    gbs = nbytes / (ms * 1e-3) / 1e9
    out["decode_state_v_first"] = {
        "workload": wl.name + ", value-major state", "ms_per_step": ms, "gpu_launches": nsteps,
        "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": round(gbs / peaks["hbm_gbs"], 4), "bytes_per_launch": nbytes}}
    del state, toks

    B, T, H, m, D = 2, 2048, 4, 4, 128
    d = make_custom(B, T, H * m, D, D, dtype="bf16", decay="train", seed=rank)
    q, k = (to_dev(np.ascontiguousarray(d[n][:, :, ::m]), dev, torch.bfloat16) for n in ("q", "k"))
    v = to_dev(d["v"], dev, torch.bfloat16)
    beta, decay = (to_dev(d[n], dev, torch.float32) for n in ("beta", "decay"))
    o = torch.empty_like(v)
    hT = torch.empty((B, H * m, D, D), dtype=torch.float32, device=dev)
    ws = torch.empty(_lib.chunk_fwd_workspace_bytes(B, T, H * m, D, D, 64, _lib.KDA_BF16),
                     dtype=torch.uint8, device=dev)

    def step():
        kda.chunk_fwd(q, k, v, beta, decay, None, out=o, final_state=hT, workspace=ws, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    barrier(world)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world)
    out["grouped_heads_prefill"] = {
        "shape": dict(B=B, T=T, qk_heads=H, v_heads=H * m, dk=D, dv=D, chunk=64), "ms_per_call": ms,
        "tokens_per_s": B * T * world / (ms * 1e-3),
        "gpu_launches_per_call": TC_PREFILL_LAUNCHES}
    return out


# --------------------------------------------------------------------------- decode
def bench_decode(args, world, rank, dev, peaks):
    import torch
    import delta_rule_linear_gb300 as kda

    wl = WORKLOADS[4]
    state = to_dev(make_decode_state(wl, seed=rank), dev, torch.float32)
    nsteps = wl.steps
    toks = []
    for s in range(nsteps):
        st = make_decode_step(wl, s, seed=rank)
        toks.append(tuple(to_dev(st[n], dev, torch.bfloat16) for n in ("q", "k", "v")) +
                    tuple(to_dev(st[n], dev, torch.float32) for n in ("beta", "decay")))
    o = torch.empty((wl.B, 1, wl.H, wl.dv), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()

    def run(n):
        for s in range(n):
            q, k, v, b, g = toks[s % nsteps]
            kda.decode_step(q, k, v, b, g, state, out=o, stream=stream)

    run(3)
    torch.cuda.synchronize()
    barrier(world)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index) as clk:
        clk.begin()
        ev0.record(stream)
        run(nsteps)
        ev1.record(stream)
        torch.cuda.synchronize()
        clk.end()
    barrier(world)
    ms = ev0.elapsed_time(ev1) / nsteps
    ms_max = max_over_ranks(ms, world)
    state_bytes = 2.0 * wl.B * wl.H * wl.dk * wl.dv * 4
    gbs = state_bytes / (ms * 1e-3) / 1e9
    ctr = recorded_counters("decode")
    return {
        "ms_per_decode_step": ms_max, "steps": nsteps,
        "state_GBps": state_bytes * world / (ms_max * 1e-3) / 1e9,
        "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": round(gbs / peaks["hbm_gbs"], 4),
                     "frac_of_8TBps_nominal": round(gbs / NOMINAL_HBM_GBS, 4),
                     "traffic": (ctr or {}).get("dram_bytes_per_launch"),
                     "traffic_capture": (ctr or {}).get("capture", "none for the kernel as built"),
                     "kernel": "decode step", "bytes_per_launch": state_bytes},
        "clocks": clk.summary(),
        "gpu_launches": nsteps,
        "shape": dict(B=wl.B, H=wl.H, dk=wl.dk, dv=wl.dv),
    }


# --------------------------------------------------------------------------- CPU oracle
def oracle_prefill_sample(d, heads_in_sample, threads=0):
    """Time the fp64 oracle on the first `heads_in_sample` heads of the long-sequence workload."""
    import oracle
    wl = WORKLOADS[3]
    sel = list(range(heads_in_sample))
    sub = {n: (None if d[n] is None else np.ascontiguousarray(d[n][:, :, sel]))
           for n in ("q", "k", "v", "beta", "decay")}
    h0 = np.ascontiguousarray(d["h0"][:, sel])
    t0 = time.perf_counter()
    _, _, used = oracle.forward(sub["q"], sub["k"], sub["v"], sub["beta"], sub["decay"], h0,
                                threads=threads, return_threads=True)
    dt = time.perf_counter() - t0
    tokens_equiv = wl.B * wl.T * heads_in_sample / wl.H
    return tokens_equiv / dt, dt, used


def run_reference(args, world, rank):
    """The reference arm: the fp64 CPU oracle on the host cores, same workload.

    Each step runs the oracle on as many of the 32 heads as the host has cores (one
    thread per head) over the full T, about a second of wall time; tokens/s is scaled by
    the head fraction."""
    if rank != 0:
        return
    import oracle
    oracle.build()
    wl = WORKLOADS[3]
    d = make_prefill(wl, seed=0)
    heads = max(1, min(wl.H, os.cpu_count() or 1))   # one oracle thread per head: every host core busy
    for _ in range(min(args.warmup, 1)):
        oracle_prefill_sample(d, 1)
    vals, secs, used = [], 0.0, 0
    for _ in range(args.steps):
        v, dt, used = oracle_prefill_sample(d, heads)
        vals.append(v)
        secs += dt
    value = statistics.median(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * secs / max(1, args.steps), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": headline_config(wl, args.gpus),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": used, "kind": "oracle",
                         "sample": f"{heads} of {wl.H} heads x full T={wl.T}, per step; "
                                   "tokens/s scaled by heads/H"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", choices=["prefill", "decode", "secondary", "gk", "gk_prefill", "layouts"] + list(SECONDARY_PARTS),
                    default=None,
                    help="run one workload (profiling); the default runs them all")
    ap.add_argument("--prefill-T", type=int, default=0,
                    help="profiling only: override T of the prefill workload (no CPU baseline)")
    ap.add_argument("--record-counters", nargs=3, metavar=("KIND", "CSV", "KERNEL_REGEX"),
                    help="store the DRAM bytes and tensor-pipe activity of an ncu --csv capture "
                         "as the counters of KIND (prefill|decode) for the current sources; no GPU")
    ap.add_argument("--scale", type=float, default=1.0,
                    help="with --record-counters: full-launch units / captured units")
    ap.add_argument("--note", default="", help="with --record-counters: the capture command")
    ap.add_argument("--tensor-csv", default=None,
                    help="with --record-counters: a second capture that supplies the tensor-pipe activity")
    args = ap.parse_args()
    if args.record_counters:
        kind, csv_path, regex = args.record_counters
        record_counters(kind, csv_path, regex, args.scale, args.note, args.tensor_csv)
        return

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        run_reference(args, world, rank)
        return

    # inputs of the prefill workload are drawn once; the CPU baseline runs on them
    # first, before any CUDA work starts in this process
    d = make_prefill(prefill_workload(args), seed=rank) if args.only in (None, "prefill") else None
    cpu = None
    if rank == 0 and not args.no_cpu_baseline and not args.prefill_T and d is not None:
        import oracle
        oracle.build()
        heads = WORKLOADS[3].H
        v, dt, used = oracle_prefill_sample(d, heads)
        cpu = {"value": v, "unit": "tokens/s", "cores": used, "kind": "oracle",
               "sample": f"all {heads} heads x full T=32768, fp64 per-token scan, "
                         f"{dt:.1f} s wall on {used} threads"}

    import torch
    world, rank, local = dist_setup()
    from delta_rule_linear_gb300 import build as b
    if rank == 0 or world == 1:
        b.build()
    barrier(world)
    import delta_rule_linear_gb300 as kda
    kda.load()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    peaks, peak_src = load_peaks()

    pre = bench_prefill(args, world, rank, dev, peaks, d) if d is not None else None
    dec = bench_decode(args, world, rank, dev, peaks) if args.only in (None, "decode") else None
    sec = bench_secondary(args, world, rank, dev, peaks) if args.only in (None, "secondary") else None
    if args.only in SECONDARY_PARTS:
        sec = bench_secondary(args, world, rank, dev, peaks, parts=(args.only,))
    if args.only in (None, "secondary", "gk", "gk_prefill"):
        sec = dict(sec or {}, kda_gk=bench_gk(args, world, rank, dev, peaks))
    if args.only in (None, "secondary", "layouts"):
        sec = dict(sec or {}, layouts=bench_layouts(args, world, rank, dev, peaks))
    if rank != 0:
        return
    if pre is None:
        print(json.dumps({"metric": METRIC, "workload": f"{args.only} only", "decode": dec,
                          "secondary": sec}), flush=True)
        return
    wl = prefill_workload(args)
    pre["roofline"]["peak_source"] = peak_src
    line = {
        "metric": METRIC, "value": pre["tokens_per_s"], "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": pre["ms"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": headline_config(wl, world),
        "roofline": pre["roofline"],
        "cpu_baseline": cpu,
        "e2e": pre["e2e"],
        "gpu_launches": pre["gpu_launches"],
        "clocks": pre["clocks"],
    }
    if dec is not None:
        dec["roofline"]["peak_source"] = peak_src
        line["decode"] = dec
    if sec is not None:
        line.update(sec)
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
