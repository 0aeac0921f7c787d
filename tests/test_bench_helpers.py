"""Host checks of the benchmark's bookkeeping: the clock record it adds to
its line, the roofline peak it divides by, and when it reports a stored DRAM
traffic figure.  Runs without a GPU."""
import json
import os

import pytest

import bench


def sampler_with(lines):
    s = bench.ClockSampler(0)
    s.lines = list(lines)
    return s


def test_clock_summary_median_max_and_reasons():
    # index, clocks.sm, clocks.max.sm, power, reasons.active, hw_slowdown,
    # hw_thermal_slowdown, sw_thermal_slowdown, sw_power_cap
    lines = [
        "0, 2070, 2070, 800.1, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 1980, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 2070, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "garbage line",
        "0, [N/A], 2070, 1.0, 0x0, Not Active, Not Active, Not Active, Not Active",
    ]
    s = sampler_with(lines).summary()
    assert s == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"],
                 "samples": 3}


def test_clock_summary_reports_every_slowdown_kind():
    lines = ["0, 1500, 2070, 1000, 0x8, Active, Not Active, Not Active, Not Active",
             "0, 1400, 2070, 1000, 0x8, Not Active, Active, Not Active, Not Active",
             "0, 1300, 2070, 1000, 0x8, Not Active, Not Active, Active, Not Active"]
    s = sampler_with(lines).summary()
    assert s["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"]
    assert s["sm_mhz"] == 1400.0 and s["samples"] == 3


def test_clock_summary_without_samples_is_none():
    assert sampler_with([]).summary() is None
    assert sampler_with(["not, a, sample"]).summary() is None


def test_measured_peak_and_fallback(monkeypatch, tmp_path):
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 6795.8}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_peaks() == (6795.8, "measured")
    os.remove(tmp_path / "MEASURED_PEAKS.json")
    assert bench.measured_peaks() == (bench.FALLBACK_HBM_GBS, "fallback")


def test_stored_traffic_only_for_the_source_it_was_taken_on(monkeypatch, tmp_path):
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "pa_decode_demo.md").write_text(
        "# demo\n\nsource_sha256_16: 0123456789abcdef\ntraffic_bytes_per_launch: 4.5e+09\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "source_digest", lambda: "0123456789abcdef")
    assert bench.stored_traffic("demo") == 4.5e9
    monkeypatch.setattr(bench, "source_digest", lambda: "fedcba9876543210")
    assert bench.stored_traffic("demo") is None   # the kernel changed since
    assert bench.stored_traffic("absent") is None


@pytest.mark.parametrize("name", sorted(
    f[len("pa_decode_"):-len(".md")]
    for f in os.listdir(os.path.join(os.path.dirname(bench.__file__), "profiles"))
    if f.startswith("pa_decode_") and f.endswith(".md")))
def test_committed_profiles_carry_a_hash_and_a_traffic_figure(name):
    """Every decode summary ends with the two lines the benchmark parses."""
    with open(os.path.join(os.path.dirname(bench.__file__), "profiles",
                           f"pa_decode_{name}.md")) as fh:
        text = fh.read()
    tail = text.strip().splitlines()[-2:]
    assert tail[0].startswith("source_sha256_16: ") and len(tail[0].split()[-1]) == 16
    assert tail[1].startswith("traffic_bytes_per_launch: ") and float(tail[1].split()[-1]) > 0
