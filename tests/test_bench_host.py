"""Host logic of bench.py (no GPU): the roofline arithmetic against the workloads' stated
figures, the parsing of ncu --csv captures in both layouts, and the recorded counters'
invalidation when a kernel's sources change."""
import importlib.util
import json
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_counted_flops_match_the_workload_figures(bench):
    # per token-head 2C(3dk + 2dv) + 6 dk dv: 180,224 at C = 64, d = 128; 65,536 at d = 64
    assert bench.counted_prefill_flops(1, 1, 1, 128, 128, 64) == 180224
    assert bench.counted_prefill_flops(1, 1, 1, 64, 64, 64) == 65536
    # long-sequence prefill (B=1, T=32768, H=32): 189.0 GFLOP; training shape: 11.81 GFLOP
    assert bench.counted_prefill_flops(1, 32768, 32, 128, 128, 64) == 188978561024
    assert round(bench.counted_prefill_flops(2, 2048, 16, 128, 128, 64) / 1e9, 2) == 11.81


def test_minimum_bytes_and_memory_ceiling(bench):
    # q, k, v, o bf16 + beta + decay per token-head, the fp32 state in and out: 1.086 GB
    b = bench.prefill_min_bytes(32768, 32, 128, 128, True, 1, True)
    assert b == 32768 * 32 * (4 * 128 * 2 + 8) + 2 * 32 * 128 * 128 * 4 == 1086324736
    # no decay and no initial state: 4 bytes less per token-head, one state only
    assert bench.prefill_min_bytes(10, 2, 64, 64, False, 3, False) == 10 * 2 * (4 * 64 * 2 + 4) + 3 * 2 * 64 * 64 * 4
    peaks = {"bf16_tflops": 1928.4, "hbm_gbs": 6677.8}
    flops = bench.counted_prefill_flops(1, 32768, 32, 128, 128, 64)
    mc = bench.memory_ceiling(flops, b, 0.695, peaks)
    # its FLOPs take 98 us at the tensor peak, its bytes 162.7 us at the copy peak: the
    # reachable tensor fraction is about 0.60
    assert abs(mc["tc_frac_ceiling_at_hbm_peak"] - (flops / 1928.4e12) / (b / 6677.8e9)) < 1e-4
    assert 0.59 < mc["tc_frac_ceiling_at_hbm_peak"] < 0.61
    assert abs(mc["hbm_frac_of_min_bytes"] - b / 0.695e-3 / 6677.8e9) < 1e-5
    # a compute-bound call's ceiling is 1
    assert bench.memory_ceiling(1e15, 1e6, 1.0, peaks)["tc_frac_ceiling_at_hbm_peak"] == 1.0


METRICS_CSV = '''==WARNING== Note: Running with unmodified GPU clocks.
==PROF== Connected to process 1
"ID","Process ID","Process Name","Host Name","Kernel Name","Context","Stream","Block Size","Grid Size","Device","CC","Section Name","Metric Name","Metric Unit","Metric Value"
"0","1","python","h","void k::other_kernel(int)","1","7","(32, 1, 1)","(1, 1, 1)","0","10.3","Command line profiler metrics","dram__bytes_read.sum","byte","5"
"1","1","python","h","void k::tc_kernel<128, 0, 0>(P)","1","7","(512, 1, 1)","(152, 1, 1)","0","10.3","Command line profiler metrics","dram__bytes_read.sum","byte","816,862,464"
"1","1","python","h","void k::tc_kernel<128, 0, 0>(P)","1","7","(512, 1, 1)","(152, 1, 1)","0","10.3","Command line profiler metrics","dram__bytes_write.sum","byte","358,486,016"
"1","1","python","h","void k::tc_kernel<128, 0, 0>(P)","1","7","(512, 1, 1)","(152, 1, 1)","0","10.3","Command line profiler metrics","gpu__time_duration.sum","ns","700,992"
'''

RAW_CSV = '''"ID","Kernel Name","dram__bytes_read.sum","dram__bytes_write.sum","sm__pipe_tensor_cycles_active.avg.pct_of_peak_sustained_active","gpu__time_duration.sum"
"","","Mbyte","Mbyte","%","us"
"0","void k::tc_kernel<128, 0, 0>(P)","206.0","78.0","21.2","198.2"
"1","void k::tc_kernel<128, 0, 0>(P)","210.0","80.0","20.8","199.0"
"2","void k::scan_kernel(Q)","1.0","1.0","0.0","5.0"
'''


def test_capture_parsing_both_layouts(bench, tmp_path):
    m = tmp_path / "metrics.csv"
    m.write_text(METRICS_CSV)
    got = bench._capture_metrics(str(m), r"tc_kernel<128, 0, 0>")
    assert list(got) == ["1"]
    assert got["1"] == {"dram__bytes_read.sum": 816862464.0, "dram__bytes_write.sum": 358486016.0}
    r = tmp_path / "raw.csv"
    r.write_text(RAW_CSV)
    got = bench._capture_metrics(str(r), r"tc_kernel")
    assert len(got) == 2
    first = got[0]
    assert first["dram__bytes_read.sum"] == pytest.approx(206.0e6)
    assert first["dram__bytes_write.sum"] == pytest.approx(78.0e6)
    assert first["sm__pipe_tensor_cycles_active.avg.pct_of_peak_sustained_active"] == pytest.approx(21.2)


def test_recorded_counters_follow_the_sources(bench, tmp_path, monkeypatch):
    src = tmp_path / "kernel.cu"
    src.write_text("// version 1\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "COUNTERS_FILE", str(tmp_path / "counters.txt"))
    monkeypatch.setattr(bench, "COUNTER_SOURCES", {"prefill": ["kernel.cu"]})
    m = tmp_path / "metrics.csv"
    m.write_text(METRICS_CSV)
    r = tmp_path / "raw.csv"
    r.write_text(RAW_CSV)
    bench.record_counters("prefill", str(m), r"tc_kernel<128, 0, 0>", scale=2.0, note="capture X",
                          tensor_csv=str(r))
    rec = bench.recorded_counters("prefill")
    assert rec is not None
    assert rec["dram_bytes_per_launch"] == pytest.approx(2.0 * (816862464 + 358486016))
    assert rec["tensor_pipe_active"] == pytest.approx((0.212 + 0.208) / 2)
    assert rec["capture"] == "capture X" and rec["launches_captured"] == 1
    assert json.loads((tmp_path / "counters.txt").read_text())["prefill"]["sources"] == bench.sources_hash("prefill")
    src.write_text("// version 2\n")   # the kernel changed since the capture: no figures
    assert bench.recorded_counters("prefill") is None
    assert bench.recorded_counters("decode") is None
