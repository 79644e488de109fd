"""Host logic of the benchmark that decides whether a number is kept: the
clock record (median SM clock under load, throttle reasons seen) and the
roofline peaks (the measured file, else the stated fallback). No GPU."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _summary(lines):
    s = bench.ClockSampler(0)
    s.out = "\n".join(lines)
    return s.summary()


def test_clock_summary_reports_reasons_and_loaded_median():
    lines = [
        "2070, 2070, 150.0, Not Active, Not Active, Not Active, Not Active",   # idle: left out of the median
        "1965, 2070, 900.5, Not Active, Not Active, Not Active, Active",
        "1980, 2070, 950.0, Not Active, Not Active, Not Active, Active",
        "2010, 2070, 905.0, Not Active, Not Active, Not Active, Not Active",
        "garbage line",
        "2070, 2070, [N/A], Not Active, Not Active, Not Active, Not Active",  # unparsable power
    ]
    d = _summary(lines)
    assert d["samples"] == 4
    assert d["sm_mhz"] == 1980.0            # median of the three loaded samples
    assert d["sm_max_mhz"] == 2070.0
    assert d["reasons"] == ["sw_power_cap"]
    assert d["power_w_max"] == 950.0


def test_clock_summary_flags_thermal_and_hardware_slowdown():
    lines = ["1500, 2070, 800.0, Active, Not Active, Active, Not Active",
             "1400, 2070, 820.0, Not Active, Active, Not Active, Not Active"]
    d = _summary(lines)
    assert d["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"]
    assert d["sm_mhz"] == 1450.0


def test_clock_summary_without_samples():
    d = _summary([])
    assert d == {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}


def test_clock_summary_all_idle_uses_every_sample():
    d = _summary(["2070, 2070, 120.0, Not Active, Not Active, Not Active, Not Active",
                  "1000, 2070, 110.0, Not Active, Not Active, Not Active, Not Active"])
    assert d["sm_mhz"] == 1535.0 and d["samples"] == 2


def test_peaks_from_the_measured_file_else_the_fallback(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    pk = bench.load_peaks()
    assert pk == {"bf16": 1900.0, "bf16_sustained": 1700.0, "source": "fallback"}
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"bf16_tflops": 1946.0,
                                                               "bf16_tflops_sustained": 1710.5,
                                                               "hbm_gbs": 6781.0}))
    pk = bench.load_peaks()
    assert pk == {"bf16": 1946.0, "bf16_sustained": 1710.5, "source": "measured"}
    (tmp_path / "MEASURED_PEAKS.json").write_text("{not json")
    assert bench.load_peaks()["source"] == "fallback"
