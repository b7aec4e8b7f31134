"""Host logic of the multi-GPU (replica) benchmark path, run as two gloo ranks
on the CPU: rendezvous, the barrier around the timed region, the max over
ranks of the step time and the whole-job rate.  No GPU and no data-path
collective are involved: each rank would run the whole GEMM on its own GPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    import torch.distributed as dist
    w, r, local = bench.dist_setup(None)
    assert (w, r, local) == (world, rank, rank)
    bench.dist_init(w, "gloo")
    bench.barrier(w)
    # rank 1 is the slow one: every rank must see its time
    slowest = bench.max_over_ranks(w, 10.0 + 5.0 * rank)
    out[rank] = slowest
    bench.barrier(w)
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_step_time():
    world, port = 2, _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        assert dict(out) == {0: 15.0, 1: 15.0}


def test_whole_job_rate_counts_every_replica():
    import bench
    flops = 2.0 * 8192 ** 3
    one = bench.aggregate_gflops(flops, 16.0, 1)
    assert one == pytest.approx(flops / 16e-3 / 1e9)
    assert bench.aggregate_gflops(flops, 16.0, 8) == pytest.approx(8 * one)


def test_reference_arm_is_rank_zero_only(monkeypatch):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class Args:
        workload = None
        steps = 1
        warmup = 0
        gpus = 2
    # a non-zero rank returns at once, without touching inputs or the oracle
    assert bench.run_reference(Args()) == 0


def test_clock_sampler_summary_keeps_samples_inside_the_timed_window(tmp_path):
    import datetime
    import bench
    t0 = datetime.datetime(2026, 1, 1, 12, 0, 0)
    lines = []
    for i, (mhz, slow) in enumerate([(1200, "Not Active"), (2070, "Not Active"),
                                     (2040, "Not Active"), (900, "Active")]):
        ts = (t0 + datetime.timedelta(seconds=i)).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
        lines.append(f"{ts}, 0, {mhz}, 2070, 500.0, 0x0, {slow}, Not Active, Not Active, Not Active")
    path = tmp_path / "clocks.csv"
    path.write_text("\n".join(lines) + "\n")
    cs = bench.ClockSampler(0)
    cs.path = str(path)
    start = (t0 + datetime.timedelta(seconds=1)).timestamp()
    cs.mark(start, start + 1.0)
    summary = cs.summary()
    assert summary["samples"] == 2 and summary["in_window"]
    assert summary["sm_mhz"] == pytest.approx(2055.0)
    assert summary["reasons"] == []
