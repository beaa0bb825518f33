"""Host logic of bench.py that needs no GPU: multi-rank timing aggregation over gloo (2 CPU
ranks), whole-job throughput, the CPU-baseline sample accounting and the reference arm's rank
handling."""
import os
import socket

import pytest

import bench
from comm_overlap_gb300 import synth


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local = [10.0 + rank, 20.0 - rank]   # rank 1 is slower in the first entry, faster in the second
        q.put((rank, bench.max_over_ranks(local, world, "cpu")))
    finally:
        torch.distributed.destroy_process_group()


def test_max_over_ranks_gloo_two_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0] == [11.0, 20.0] and res[1] == [11.0, 20.0]


def test_job_throughput_counts_all_ranks():
    s = synth.SHAPES["llama3_8b_swiglu_fwdbwd"]
    one = bench.job_tflops(s.gemm_flops(), 10, 1, 250.0)
    assert abs(one - 10 * s.gemm_flops() / 0.25 / 1e12) < 1e-9
    assert abs(bench.job_tflops(s.gemm_flops(), 10, 4, 250.0) - 4 * one) < 1e-9


def test_gemm_flops_of_the_workloads():
    # forward: 2 M h R + 2 M F h (R = 2F gated); backward = 2 x forward
    s = synth.SHAPES["llama3_8b_swiglu_fwdbwd"]
    fwd = 2 * 32768 * 4096 * 2 * 14336 + 2 * 32768 * 14336 * 4096
    assert s.gemm_flops() == 3 * fwd
    s = synth.SHAPES["gpt3_6.7b_stack4"]
    assert s.gemm_flops() == 4 * (2 * 32768 * 4096 * 16384 * 2)


def test_kernel_work_sums_to_step_flops():
    # the per-launch algorithmic flops of the GEMM kinds, times their launches per step, add up to
    # the step's GEMM flops (p launches of each kind per step, q of the column-chunked ones)
    s = synth.SHAPES["llama3_8b_swiglu_fwdbwd"]
    w = bench.kernel_work(s)
    per_step = (s.p * (w["gemm_fwd1"][1] + w["gemm_dgrad_h"][1] + w["gemm_wgrad_b"][1] + w["gemm_wgrad_a"][1])
                + s.p * s.q * (w["gemm_fwd2"][1] + w["gemm_dgrad_x"][1]))
    assert abs(per_step - s.gemm_flops()) / s.gemm_flops() < 1e-12


def test_reference_arm_only_rank0_reports():
    class A:
        pass
    a = A()
    a.shape = synth.SHAPES["tiny_gelu"]
    assert bench.run_reference(a, rank=1) is None


def test_reduction_roofline_and_traffic_lookup():
    s = synth.SHAPES["llama3_8b_swiglu_fwdbwd"]
    work = bench.kernel_work(s)
    peaks = {"hbm_gbs": 6794.5}
    kern = {"shard_sum": {"launches": 4, "total_ms": 4 * 0.34}}
    r = bench.reduction_roofline(kern, work, peaks, s.name)
    m, n = s.M // s.p, s.h // s.q
    assert r["algorithmic_bytes_per_launch"] == s.t * m * n * 4 + m * n * 2
    assert abs(r["achieved"] - r["algorithmic_bytes_per_launch"] / 0.34e-3 / 1e9) < 1e-6
    assert abs(r["frac"] - r["achieved"] / 6794.5) < 1e-12
    # the fused schedule launches no shard-sum: no reduction roofline
    assert bench.reduction_roofline({}, work, peaks, s.name) is None


def test_traffic_is_reported_only_for_the_code_it_was_captured_on(monkeypatch):
    s = synth.SHAPES["llama3_8b_swiglu_fwdbwd"]
    cur = bench.kernel_source_sha("elementwise")
    monkeypatch.setattr(bench, "NCU_TRAFFIC", {(s.name, "shard_sum"): {"bytes_per_launch": 2.0e9, "src_sha": cur},
                                               (s.name, "gemm_fwd1"): {"bytes_per_launch": 5.0e9,
                                                                       "src_sha": "0" * 16}})
    assert bench.traffic_per_launch(s.name, "shard_sum") == 2.0e9
    assert bench.traffic_per_launch(s.name, "shard_sum", "0" * 16) is None
    assert bench.traffic_per_launch("tiny_gelu", "shard_sum") is None
    # a GEMM entry keyed to other GEMM code is not reported
    assert bench.traffic_per_launch(s.name, "gemm_fwd1") is None
    # each kind is keyed to its own sources: the GEMM and shard-sum hashes differ
    assert bench.source_group("gemm_dgrad_x") == "gemm" and bench.source_group("shard_sum") == "elementwise"
    assert bench.kernel_source_sha("gemm") != cur


def test_kernel_hash_ignores_comments():
    code = "int a; // note\n/* block\n comment */ int b;\n\n"
    assert bench._code_only(code) == bench._code_only("int a;\n int b;")


def test_clock_summary_keeps_the_timed_window():
    """Only nvidia-smi rows stamped inside the timed loop's window count: an idle lead-in at a high
    clock and low power must not enter the median, and throttle reasons outside it are ignored."""
    import datetime
    import bench

    def row(sec, mhz, watts, cap="Not Active", thermal="Not Active"):
        ts = datetime.datetime(2026, 12, 2, 11, 25, 0) + datetime.timedelta(seconds=sec)
        return ", ".join([ts.strftime("%Y/%m/%d %H:%M:%S.%f")[:-3], "0", str(mhz), "2070", str(watts), "0x0",
                          "Not Active", thermal, "Not Active", cap])

    lines = [row(0.00, 2070, 180.0, thermal="Active"), row(0.05, 2070, 185.0),         # idle lead-in
             row(0.10, 1500, 1390.0, cap="Active"), row(0.15, 1470, 1400.0, cap="Active"),
             row(0.20, 1485, 1395.0, cap="Active"),                                      # timed loop
             row(0.30, 2070, 300.0)]                                                     # after it
    text = "\n".join(lines) + "\n"
    t0 = datetime.datetime(2026, 12, 2, 11, 25, 0).timestamp() + 0.08
    c = bench.summarize_clocks(text, t0, t0 + 0.15)
    assert c["samples"] == 3 and c["in_window"]
    assert c["sm_mhz"] == 1485.0 and c["power_w_max"] == 1400.0 and c["sm_max_mhz"] == 2070.0
    assert c["reasons"] == ["sw_power_cap"]
    every = bench.summarize_clocks(text)
    assert every["samples"] == 6 and "in_window" not in every
    assert "hw_thermal_slowdown" in every["reasons"]
    empty = bench.summarize_clocks(text, t0 + 10.0, t0 + 11.0)
    assert empty["in_window"] is False and empty["samples"] == 6


def test_reduction_alone_on_a_timeline():
    """The exposed part of each shard-sum is its time minus the union of the other kernels' spans."""
    K_RED, K_G1, K_G2 = 2, 0, 1
    trace = [(K_G1, 0.0, 10.0),      # GEMM of chunk 0
             (K_G2, 9.0, 20.0),      # next GEMM, overlapping the first
             (K_RED, 8.0, 12.0),     # reduction fully under the GEMMs
             (K_RED, 19.0, 23.0),    # reduction half exposed: 20 .. 23
             (K_G1, 22.0, 30.0),     # GEMM starting before that reduction ends: 22 .. 23 hidden
             (K_RED, 31.0, 32.5)]    # reduction after everything: exposed
    total, alone = bench.reduction_alone_ms(trace, K_RED)
    assert abs(total - (4.0 + 4.0 + 1.5)) < 1e-12
    assert abs(alone - (0.0 + 2.0 + 1.5)) < 1e-12
    assert bench.reduction_alone_ms([(K_G1, 0.0, 1.0)], K_RED) == (0.0, 0.0)


def test_exposure_summary_of_alternating_windows():
    steps = 50
    wins = [("normal", 50 * 22.0, 1500.0), ("noreduce", 50 * 21.0, 1540.0),
            ("normal", 50 * 22.2, 1510.0), ("noreduce", 50 * 21.2, 1530.0)]
    e = bench.exposure_summary(wins, steps)
    t_n, t_0, f_n, f_0 = 22.1, 21.1, 1505.0, 1535.0
    assert abs(e["ms_per_step_normal"] - t_n) < 1e-9 and abs(e["ms_per_step_noreduce"] - t_0) < 1e-9
    assert abs(e["ms"] - 1.0) < 1e-9 and abs(e["frac"] - 1.0 / t_n) < 1e-12
    assert e["sm_mhz_normal"] == f_n and e["sm_mhz_noreduce"] == f_0
    assert abs(e["frac_equal_clock"] - (t_n * f_n - t_0 * f_0) / (t_n * f_n)) < 1e-12
    assert len(e["windows"]) == 4 and e["steps_per_window"] == steps
    # without clock samples the equal-clock figure is left out
    assert "frac_equal_clock" not in bench.exposure_summary([(a, ms, None) for a, ms, _ in wins], steps)
