"""Host-only parts of bench.py: the oracle table (the CPU oracle timed with all
host cores and with one) on the smallest workload.  No GPU is involved."""
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
