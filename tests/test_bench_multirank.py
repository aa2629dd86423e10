"""Multi-rank host logic of bench.py on CPU: two gloo ranks.

Every GPU run available here has one GPU, so the N > 1 path of the bench
(replicas, barrier, the job time as the maximum over ranks, the whole-job
throughput) is checked with the gloo backend on CPU.
"""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, times_ms, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        dist.barrier()
        worst = bench.max_over_ranks(times_ms[rank], world, "cpu")
        value = bench.job_tflops(world, 5, 2.0e12, worst)
        dist.barrier()
        out.put((rank, worst, value))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    out = ctx.SimpleQueue()
    times = [10.0, 12.5]
    mp.start_processes(_rank, args=(2, _free_port(), times, out), nprocs=2, join=True,
                       start_method="spawn")
    got = sorted(out.get() for _ in range(2))
    for rank, worst, value in got:
        assert worst == pytest.approx(12.5)               # slowest rank
        # two replicas x 5 steps x 2 TFLOP in 12.5 ms
        assert value == pytest.approx(2 * 5 * 2.0e12 / 0.0125 / 1e12)


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.25, 1) == 3.25
    assert bench.job_tflops(1, 4, 1.0e12, 2.0) == pytest.approx(2000.0)


def test_clock_sampler_keeps_only_samples_inside_the_timed_region():
    import datetime
    import bench
    t0 = 1_800_000_000.0

    def line(t, clk, hw="Not Active", cap="Not Active"):
        ts = datetime.datetime.fromtimestamp(t).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
        return f"{ts}, 0, {clk}, 2070, 1200.0, 0x0, {hw}, Not Active, Not Active, {cap}"

    out = "\n".join([line(t0 - 0.5, 2070), line(t0 + 0.1, 1900, cap="Active"),
                     line(t0 + 0.2, 1800), line(t0 + 0.3, 1850), line(t0 + 2.0, 345, hw="Active")])
    r = bench.ClockSampler.parse(out, t0, t0 + 1.0)
    assert r["samples"] == 3 and r["sm_mhz"] == 1850.0 and r["sm_min_mhz"] == 1800.0
    assert r["reasons"] == ["sw_power_cap"]              # the hw_slowdown sample was outside
    assert "error" in bench.ClockSampler.parse(out, t0 + 5, t0 + 6)
    # a region between two samples takes the one just before and the one just after it
    r = bench.ClockSampler.parse(out, t0 + 0.21, t0 + 0.25)
    assert r["samples"] == 2 and r["sm_min_mhz"] == 1800.0 and r["sm_max_mhz"] == 2070.0
    assert "nearest_samples" in r and r["reasons"] == []
