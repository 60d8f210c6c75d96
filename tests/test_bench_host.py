"""Host-side logic of bench.py (CPU): the clock summary that decides whether a run is valid,
the recorded-traffic lookup keyed by the kernel sources' hash, the measured peak, and the
confidence interval of the generation loop."""
import importlib.util
import json
import math
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_clock_summary_median_and_reasons(bench):
    cs = bench.ClockSampler(0)
    rows = ["2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active",
            "1995, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active",
            "2070, 2070, 950.0, 0x0, Not Active, Not Active, Not Active, Not Active",
            "[N/A], 2070, 0, 0x0, Not Active, Not Active, Not Active, Not Active",
            "garbage"]
    cs.samples = [(10.0 + 0.1 * i, r) for i, r in enumerate(rows)]
    s = cs.summary(10.0, 10.5)
    assert s["sm_mhz"] == 2070.0 and s["sm_max_mhz"] == 2070.0 and s["samples"] == 3
    assert s["reasons"] == ["sw_power_cap"]
    cs.samples.append((10.3, "1200, 2070, 800, 0x8, Active, Not Active, Active, Not Active"))
    s = cs.summary(10.0, 10.5)
    assert s["reasons"] == ["hw_slowdown", "sw_power_cap", "sw_thermal_slowdown"]
    # outside the window: falls back to every sample
    assert cs.summary(100.0, 101.0)["samples"] == 4


def test_recorded_traffic_needs_the_same_sources_and_workload(bench, tmp_path, monkeypatch):
    sha = bench.kernel_source_sha()
    assert len(sha) == 16 and sha == bench.kernel_source_sha()
    rec = tmp_path / "traffic.json"
    rec.write_text(json.dumps({"kernel_source_sha": sha, "workload": "w",
                               "dram_bytes_per_launch": 123.0}))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(rec))
    assert bench.recorded_traffic("w") == 123.0
    assert bench.recorded_traffic("other") is None
    rec.write_text(json.dumps({"kernel_source_sha": "0" * 16, "workload": "w",
                               "dram_bytes_per_launch": 123.0}))
    assert bench.recorded_traffic("w") is None


def test_measured_peak(bench):
    peak, kind = bench.measured_peak()
    if os.path.exists(os.path.join(ROOT, "MEASURED_PEAKS.json")):
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            assert (peak, kind) == (float(json.load(f)["hbm_gbs"]), "measured")
    else:
        assert (peak, kind) == (bench.FALLBACK_HBM_GBS, "fallback")


def test_mean_ci(bench):
    xs = [1.0, 2.0, 3.0, 4.0]
    m, ci = bench._mean_ci(xs)
    sd = math.sqrt(sum((x - 2.5) ** 2 for x in xs) / 3)
    assert m == 2.5 and abs(ci - 1.96 * sd / 2.0) < 1e-12
    assert bench._mean_ci([5.0]) == (5.0, 0.0)


def test_traffic_record_from_an_ncu_log(bench, tmp_path):
    """--record-traffic reads ncu's one-row-per-metric CSV (units scaled or in bytes), keeps
    the decode launches only, and keys the record by the current kernel sources' hash."""
    hdr = ('"ID","Process ID","Process Name","Host Name","Kernel Name","Context","Stream",'
           '"Block Size","Grid Size","Device","CC","Section Name","Metric Name","Metric Unit",'
           '"Metric Value"\n')

    def row(i, kern, metric, unit, val):
        return (f'"{i}","1","python","h","{kern}","1","7","(256, 1, 1)","(16, 4, 1)","0",'
                f'"10.3","Command line profiler metrics","{metric}","{unit}","{val}"\n')

    k = "void santa::decode_kernel<true, 128, 7, true>(santa::DecodeParams)"
    text = ("==PROF== Connected to process 1\n" + hdr +
            row(0, k, "dram__bytes_read.sum", "Mbyte", "8.17") +
            row(0, k, "dram__bytes_write.sum", "byte", "0") +
            row(1, "void at::native::fill_kernel()", "dram__bytes_read.sum", "byte", "5") +
            row(1, "void at::native::fill_kernel()", "dram__bytes_write.sum", "byte", "5") +
            row(2, k, "dram__bytes_read.sum", "byte", "7,915,008") +
            row(2, k, "dram__bytes_write.sum", "Kbyte", "1.5"))
    csv_path = tmp_path / "traffic.csv"
    csv_path.write_text(text)
    out = tmp_path / "rec.json"
    rec = bench.record_traffic_file(str(csv_path), str(out), "w", "ncu ...")
    assert rec["dram_bytes_read_per_launch"] == [8.17e6, 7915008.0]
    assert rec["dram_bytes_write_per_launch"] == [0.0, 1500.0]
    assert rec["dram_bytes_per_launch"] == (8.17e6 + 7915008.0 + 1500.0) / 2
    assert rec["kernel_source_sha"] == bench.kernel_source_sha()
    assert json.loads(out.read_text()) == rec


def test_host_stall_filter(bench):
    """Loop-mode steps far above the median (the host fell behind the spin kernel) are left
    out of the mean and counted; ordinary spread is kept."""
    us = [17.0, 17.2, 16.9, 17.1, 50000.0, 17.0, 30.0]
    kept, dropped = bench._drop_host_stalls(us)
    assert dropped == 1 and 50000.0 not in kept and 30.0 in kept
    assert bench._drop_host_stalls([5.0] * 10) == ([5.0] * 10, 0)
