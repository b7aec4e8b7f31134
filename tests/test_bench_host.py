"""Host-only parts of bench.py: the oracle table (the CPU oracle timed with all
host cores and with one) on the smallest workload, the reference arm's line,
the clock summary's throttle reasons, power and fallbacks (its time window is
also covered with the replica tests), and the DRAM, traffic and peak figures of
the roofline object.  No GPU is involved."""
import argparse
import json

import pytest


def test_oracle_table_times_every_workload_with_all_cores_and_one(monkeypatch, capsys):
    import bench
    from dense_fp32_gemm_02_gb300 import workloads
    small = {"sgemm_256": workloads.WORKLOADS["sgemm_256"]}
    monkeypatch.setattr(workloads, "WORKLOADS", small)
    monkeypatch.delenv("RANK", raising=False)
    args = argparse.Namespace(oracle_budget=0.05)
    assert bench.run_oracle_table(args) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["kind"] == "oracle" and line["unit"] == "GFLOP/s"
    assert line["host"]["cores"] == bench.host_cores()
    rows = line["oracle_table"]
    assert [(r["workload"], r["threads"]) for r in rows] == \
        [("sgemm_256", bench.host_cores()), ("sgemm_256", 1)]
    for r in rows:
        assert 1 <= r["rows"] <= 256 and r["secs"] > 0 and r["gflops"] > 0
        # the rate is 2 N K per row over the measured seconds (printed to the ms)
        assert r["gflops"] == pytest.approx(2.0 * r["rows"] * 256 * 256 / r["secs"] / 1e9,
                                            rel=0.05)


def test_dram_use_is_traffic_over_time_against_the_measured_copy_bandwidth():
    import os
    import bench
    if os.path.exists(bench.PEAKS_FILE):      # driver-written; the fallback otherwise
        with open(bench.PEAKS_FILE) as f:
            peak = json.load(f)["hbm_gbs"]
    else:
        peak = bench.HBM_FALLBACK_GBS
    d = bench.dram_use(3.0e9, 15.0)              # 3 GB in 15 ms = 200 GB/s
    assert d["dram_gbs"] == pytest.approx(200.0)
    assert d["dram_frac"] == pytest.approx(200.0 / peak, abs=1e-4)
    assert bench.dram_use(None, 15.0) == {"dram_gbs": None, "dram_frac": None}
    assert bench.dram_use(3.0e9, 0.0) == {"dram_gbs": None, "dram_frac": None}


def test_reference_arm_prints_the_contract_line(monkeypatch, capsys):
    """Rank 0 of the reference arm times the oracle on rows of the workload and
    prints one JSON line with the bench contract's keys (no GPU)."""
    import bench
    monkeypatch.delenv("RANK", raising=False)
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    args = argparse.Namespace(workload="sgemm_256", steps=2, warmup=1, gpus=1)
    assert bench.run_reference(args) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC
    assert line["unit"] == "GFLOP/s" and line["value"] > 0 and line["higher_is_better"] is True
    assert (line["steps"], line["warmup"], line["n_gpus"]) == (2, 1, 1)
    cpu = line["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["cores"] == bench.host_cores()
    assert cpu["value"] == line["value"] and "rows" in cpu["sample"]
    assert line["e2e"] == {"value": line["value"], "unit": "GFLOP/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    assert line["config"]["workload"] == "sgemm_256"


def _smi_row(ts, sm, sm_max, power, reasons=()):
    """One line of `nvidia-smi --format=csv,noheader,nounits` for ClockSampler.FIELDS."""
    flags = ["Active" if n in reasons else "Not Active"
             for n in ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")]
    stamp = ts.strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    return ", ".join([stamp, "0", str(sm), str(sm_max), f"{power:.2f}", "0x0000000000000000"] + flags)


def test_clock_summary_reasons_power_and_fallback_to_all_samples(tmp_path):
    """Median SM clock, maximum clock, throttle reasons and power come from the
    samples inside the marked windows; the idle samples around them (low clock,
    a power-cap flag) do not count, and malformed lines are skipped."""
    import datetime
    import bench
    t = datetime.datetime(2026, 1, 5, 12, 0, 0)
    sec = datetime.timedelta(seconds=1)
    lines = [_smi_row(t, 345, 2070, 90.0, {"sw_power_cap"}),            # before the window
             "garbage line",
             _smi_row(t + 2 * sec, 1965, 2070, 1100.0),
             _smi_row(t + 3 * sec, 1980, 2070, 1150.0, {"sw_power_cap"}),
             _smi_row(t + 4 * sec, 1950, 2070, 1120.0),
             _smi_row(t + 9 * sec, 400, 2070, 95.0, {"hw_slowdown"})]        # after it
    path = tmp_path / "clocks.csv"
    path.write_text("\n".join(lines) + "\n")
    s = bench.ClockSampler(0)
    s.path = str(path)
    s.mark((t + 2 * sec).timestamp(), (t + 4 * sec).timestamp())
    out = s.summary()
    assert out["samples"] == 3 and out["in_window"] is True
    assert out["sm_mhz"] == 1965 and out["sm_max_mhz"] == 2070
    assert out["reasons"] == ["sw_power_cap"]
    assert out["power_w_median"] == pytest.approx(1120.0)
    # a window with no samples falls back to every sample, and says so
    late = (t + 60 * sec).timestamp()
    out = s.summary(windows=[(late, late + 1)])
    assert out["samples"] == 5 and out["in_window"] is False
    assert out["reasons"] == ["hw_slowdown", "sw_power_cap"]


def test_clock_summary_without_samples(tmp_path):
    import bench
    s = bench.ClockSampler(0)
    s.path = str(tmp_path / "missing.csv")
    out = s.summary()
    assert out["sm_mhz"] is None and out["samples"] == 0
    assert out["reasons"] == ["no nvidia-smi samples"]


def test_l2_note_says_whether_the_inputs_outgrow_l2():
    import bench
    from dense_fp32_gemm_02_gb300.workloads import WORKLOADS
    assert bench.l2_note(WORKLOADS["sgemm_8192_ab"]).startswith("inputs larger than L2 (A, B, C 805 MB")
    assert "not larger than" in bench.l2_note(WORKLOADS["sgemm_256"])


def test_traffic_figure_counts_only_for_the_kernel_sources_it_was_taken_on(monkeypatch):
    import bench
    with open(bench.PROFILE_SUMMARY) as f:
        stored = json.load(f)["sgemm_8192_ab"]
    monkeypatch.setattr(bench, "kernel_revision", lambda: stored["kernel_revision"])
    assert bench.load_traffic("sgemm_8192_ab") == stored["dram_bytes_per_launch"]
    assert bench.load_traffic("no_such_workload") is None
    monkeypatch.setattr(bench, "kernel_revision", lambda: "0" * 16)
    assert bench.load_traffic("sgemm_8192_ab") is None


def test_tensor_peak_comes_from_the_measured_bf16_figure_else_the_fallback(monkeypatch, tmp_path):
    import bench
    monkeypatch.setattr(bench, "PEAKS_FILE", str(tmp_path / "absent.json"))
    peak, src = bench.tensor_peak_tf32()
    assert peak == pytest.approx(bench.BF16_FALLBACK_TFLOPS * bench.TF32_PER_BF16)
    assert src.startswith("fallback")
    p = tmp_path / "peaks.json"
    p.write_text(json.dumps({"bf16_tflops": 2000.0, "hbm_gbs": 7000.0}))
    monkeypatch.setattr(bench, "PEAKS_FILE", str(p))
    peak, src = bench.tensor_peak_tf32()
    assert peak == pytest.approx(2000.0 * bench.TF32_PER_BF16) and src.startswith("measured")
    assert bench.dram_use(7.0e9, 10.0)["dram_frac"] == pytest.approx(0.1)


def test_probed_mma_fraction_uses_the_unit_rate_at_max_and_measured_clock():
    import bench
    # 152 SMs x 4096 TF32 FLOP/clk x 2070 MHz = 1288.8 TFLOP/s
    f = bench.probed_mma_fields(1071.0, 152, 1960.0)
    assert abs(f["probed_mma_peak"] - 152 * 4096 * 2070e6 / 1e12) < 1e-3
    assert abs(f["frac_of_probed_mma"] - 1071.0 / 1288.8) < 1e-3
    assert abs(f["frac_of_probed_mma_at_measured_clock"] - 1071.0 / (152 * 4096 * 1960e6 / 1e12)) < 1e-3
    assert bench.probed_mma_fields(None, 152)["frac_of_probed_mma"] is None
    assert bench.probed_mma_fields(1071.0, 152)["frac_of_probed_mma_at_measured_clock"] is None
