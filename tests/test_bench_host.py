"""Host-side logic of the benchmark: clock-record summary, the DRAM-traffic
record's tie to the kernel sources, fixed-plan parsing and the peak lookup.
No GPU is needed."""
import json
import os

import pytest

import bench


def _row(sm, mx, hw="Not Active", hwt="Not Active", swt="Not Active", cap="Not Active"):
    return ["0", str(sm), str(mx), "900.0", "0x0", hw, hwt, swt, cap]


def test_clock_summary_median_max_and_reasons():
    rows = [_row(2070, 2070), _row(1900, 2070, cap="Active"), _row(2000, 2070)]
    s = bench.ClockSampler.summarize(rows)
    assert s["sm_mhz"] == 2000.0
    assert s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]
    assert s["samples"] == 3


def test_clock_summary_reports_every_throttle_reason():
    rows = [_row(1200, 2070, hw="Active"), _row(1300, 2070, hwt="Active", swt="Active")]
    s = bench.ClockSampler.summarize(rows)
    assert s["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"]


def test_clock_summary_without_samples():
    s = bench.ClockSampler.summarize([])
    assert s["samples"] == 0 and s["sm_mhz"] is None and s["reasons"] == ["no samples"]


def test_clock_summary_skips_unparsable_fields():
    s = bench.ClockSampler.summarize([_row("[N/A]", "[N/A]"), _row(1980, 2070)])
    assert s["sm_mhz"] == 1980.0 and s["sm_max_mhz"] == 2070.0 and s["samples"] == 2


def test_traffic_record_used_only_for_the_kernel_it_describes():
    # The committed record is reported only while the kernel sources hash as
    # they did when the counters were taken; otherwise traffic is null.
    path = os.path.join(bench.ROOT, "profiles", "fused_gemv_gate_proj_b1.traffic.json")
    with open(path) as f:
        rec = json.load(f)
    assert rec["dram_bytes_per_launch"] == rec["dram_bytes_read"] + rec["dram_bytes_write"]
    if rec["kernel_hash"] == bench.kernel_hash():
        assert bench.profiled_traffic() == float(rec["dram_bytes_per_launch"])
    else:
        assert bench.profiled_traffic() is None


def test_traffic_record_is_dropped_once_the_kernel_changes(monkeypatch):
    monkeypatch.setattr(bench, "kernel_hash", lambda: "0" * 16)
    assert bench.profiled_traffic() is None


def test_fixed_plan_names_a_variant():
    import lossless_bf16_weight_gb300 as uw
    plan = bench.fixed_plan(uw, "fused:col_w16x1")
    assert plan.strategy == uw.STRATEGY_FUSED
    assert uw.variant_name(uw.STRATEGY_FUSED, plan.variant) == "col_w16x1"
    plan = bench.fixed_plan(uw, "exponent:tc_g3")
    assert plan.strategy == uw.STRATEGY_EXPONENT
    assert uw.variant_name(uw.STRATEGY_EXPONENT, plan.variant) == "tc_g3"


def test_fixed_plan_rejects_an_unknown_variant():
    import lossless_bf16_weight_gb300 as uw
    with pytest.raises(SystemExit):
        bench.fixed_plan(uw, "fused:no_such_variant")


def test_peak_comes_from_the_measured_file_when_present():
    path = os.path.join(bench.ROOT, "MEASURED_PEAKS.json")
    value, kind = bench.peaks()
    if os.path.exists(path):
        with open(path) as f:
            assert value == float(json.load(f)["hbm_gbs"])
        assert kind == "measured"
    else:
        assert (value, kind) == (bench.FALLBACK_HBM_GBS, "fallback")


def test_clock_sampler_without_nvidia_smi(monkeypatch):
    # No nvidia-smi on the path: no samples, and the temporary file is gone.
    monkeypatch.setenv("PATH", "")
    c = bench.ClockSampler(0)
    c.start()
    assert c.stop() == []
    assert not os.path.exists(c.path)
