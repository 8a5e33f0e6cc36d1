"""Host-side helpers of bench.py, on the CPU: clock-sample parsing, the
kernel source hash and the gate on recorded DRAM traffic."""

import importlib.util
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    argv = sys.argv
    sys.argv = ["bench.py"]
    try:
        spec = importlib.util.spec_from_file_location("bench_under_test",
                                                      os.path.join(ROOT, "bench.py"))
        mod = importlib.util.module_from_spec(spec)
        spec.loader.exec_module(mod)
    finally:
        sys.argv = argv
    return mod


def test_clock_summary_reports_median_and_reasons(bench):
    s = bench.ClockSampler(0)
    s.lines = [
        "2070, 2070, 900.0, Not Active, Not Active, Not Active, Not Active",
        "2055, 2070, 1100.0, Not Active, Not Active, Not Active, Active",
        "2070, 2070, 1000.0, Not Active, Not Active, Not Active, Not Active",
        "garbage line",
    ]
    out = bench.ClockSampler.summary(s)
    assert out["sm_mhz"] == 2070.0 and out["sm_max_mhz"] == 2070.0
    assert out["reasons"] == ["sw_power_cap"] and out["samples"] == 3
    s.lines = ["1500, 2070, 800.0, Active, Not Active, Active, Not Active"]
    out = bench.ClockSampler.summary(s)
    assert out["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]
    s.lines = []
    assert bench.ClockSampler.summary(s)["samples"] == 0


def test_source_hash_ignores_comments_only(bench):
    a = "int f(int x) { return x + 1; }  // one\n/* block\n comment */\n"
    b = "int f(int x)\n{\n  return x + 1;  // changed comment\n}\n"
    c = "int f(int x) { return x + 2; }\n"
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only(a) != bench._code_only(c)


def test_recorded_traffic_is_used_only_for_the_current_sources(bench, tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_sha", lambda: "abc123")
    assert bench.ncu_traffic("c3") is None                 # no file
    (prof / "dram_traffic_c3.txt").write_text("kernel_source_sha: abc123\ndram_bytes_per_call: 1234\n")
    assert bench.ncu_traffic("c3") == 1234.0
    (prof / "dram_traffic_c3.txt").write_text("kernel_source_sha: other\ndram_bytes_per_call: 1234\n")
    assert bench.ncu_traffic("c3") is None                 # taken on other sources


def test_rank_rows_do_not_overlap(bench):
    assert bench.rank_row0(0) == 0
    assert bench.rank_row0(1) - bench.rank_row0(0) >= 100000
