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
