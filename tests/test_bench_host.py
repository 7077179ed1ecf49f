"""Host-side logic of bench.py that needs no GPU: the clock sampler's reading of nvidia-smi lines
(samples kept to the timed region, throttle reasons, missing samples) and the DRAM-traffic lookup
that is dropped once the main kernel's source changes."""
import json

import bench


def _line(sm, smax=2070, reasons=("Not Active",) * 4):
    return f"0, {sm}, {smax}, 900.0, 0x0000000000000000, " + ", ".join(reasons)


def test_clock_summary_keeps_the_timed_region():
    s = bench.ClockSampler(0, period_ms=20)
    s.lines = [(0.0, _line(1400)), (1.0, _line(2070)), (1.02, _line(2055)), (1.04, _line(2070)), (3.0, _line(900))]
    s.mark(0.99, 1.03)
    out = s.summary()
    assert out["samples"] == 3 and out["scope"] == "timed region"
    assert out["sm_mhz"] == 2070 and out["sm_max_mhz"] == 2070 and out["reasons"] == []


def test_clock_summary_reports_throttle_reasons():
    s = bench.ClockSampler(0)
    s.lines = [(1.0, _line(1942, reasons=("Not Active", "Not Active", "Not Active", "Active"))),
               (1.01, _line(1900, reasons=("Active", "Not Active", "Not Active", "Not Active")))]
    out = s.summary()
    assert out["scope"] == "whole run"
    assert out["reasons"] == ["hw_slowdown", "sw_power_cap"]
    assert out["sm_mhz"] == (1942 + 1900) / 2


def test_clock_summary_without_samples():
    s = bench.ClockSampler(0)
    s.lines = [(1.0, "garbage")]
    assert s.summary()["reasons"] == ["no samples"]


def test_traffic_only_for_the_captured_source(tmp_path, monkeypatch):
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(
        {"kv_kernel/w": {"dram_bytes_per_launch": 123.0, "source_sha": "abc"}}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench._traffic("kv_kernel/w", "abc") == 123.0
    assert bench._traffic("kv_kernel/w", "def") is None
    assert bench._traffic("kv_kernel/other", "abc") is None
