"""bench.py's JSON line, assembled on CPU from synthetic stage times: the
keys the benchmark contract asks for, the roofline arithmetic and the
traffic figure (only for the unmodified named workload)."""
import argparse
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
from moe_inputs import WORKLOADS  # noqa: E402


def _args(**kw):
    a = dict(workload="imagegen-16k", no_cpu_baseline=True, cpu_seconds=0.1, gpus=1, steps=10,
             warmup=3, T=None, E=None, I=None, Is=None, tp=1, shared_stream="off", seed=0,
             no_e2e=False, impl="ours", gate_sequential=False, y_f32=False, steady_seconds=0.0)
    a.update(kw)
    return argparse.Namespace(**a)


def _stages(ms):
    import moe_expert_routing_fp32_gb300 as moe
    return {n: ms for n in moe.STAGE_NAMES}


CLK = {"sm_mhz": 1700.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"]}


def test_json_line_keys_and_roofline():
    args = _args()
    wl = WORKLOADS["imagegen-16k"]
    stages = _stages(1.0)
    stages["gemm_w13_swiglu"] = 4.5
    res = bench.finish_ours(args, wl, 1, 0, 10, 3, 80.0, stages, CLK, 1.9e6, {})
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "e2e", "gpu_launches", "clocks"):
        assert key in res, key
    assert res["value"] == pytest.approx(16384 * 10 / 0.080)
    assert res["ms_per_step"] == pytest.approx(8.0)
    r = res["roofline"]
    flops = 4.0 * wl.T * wl.k * wl.H * wl.I + 4.0 * wl.T * wl.H * wl.I_s
    assert r["achieved"] == pytest.approx(flops / 4.5e-3 / 1e12, rel=1e-3)
    assert r["frac"] == pytest.approx(r["achieved"] / r["peak"], rel=1e-3)
    assert r["traffic"] is None or r["traffic"] > 4e9      # recorded for this workload
    assert res["e2e"]["h2d_bytes_per_step"] == wl.T * wl.H * 2
    assert res["config"]["workload"] == "imagegen-16k"


def test_traffic_not_reported_for_a_resized_workload():
    args = _args(I=128, Is=128)
    wl = bench.workload_of(args)
    res = bench.finish_ours(args, wl, 1, 0, 10, 3, 10.0, _stages(0.5), CLK, None, {})
    assert res["roofline"]["traffic"] is None
    assert res["e2e"] is None


def test_launch_count_follows_the_gate_path():
    """gpu_launches is the library's kernels per step times the steps: the
    tensor-core gate adds RMSNorm, split, GEMM and combine launches above 512
    tokens; the small-batch router and the sequential gate are fewer."""
    img = WORKLOADS["imagegen-16k"]
    assert bench.launches_per_step(img) == 10
    assert bench.launches_per_step(img, gate_sequential=True) == 7
    assert bench.launches_per_step(img, two_streams=True) == 11
    assert bench.launches_per_step(WORKLOADS["skewed-32k"]) == 9          # no RMSNorm
    assert bench.launches_per_step(WORKLOADS["smallbatch-8"]) == 7   # histogram in the scan
    res = bench.finish_ours(_args(), img, 1, 0, 10, 3, 80.0, _stages(1.0), CLK, None, {})
    assert res["gpu_launches"] == 100
    assert "tensor cores" in res["config"]["gate"]
    res = bench.finish_ours(_args(gate_sequential=True), img, 1, 0, 10, 3, 80.0, _stages(1.0),
                            CLK, None, {})
    assert res["gpu_launches"] == 70 and "sequential" in res["config"]["gate"]


def test_roofline_bound_follows_the_arithmetic_intensity():
    """Thousands of rows per expert make the matmul tensor-bound; a few rows
    per expert make it stream the weights, and the roofline is then HBM
    bytes (the experts that get rows, each weight once) against the HBM peak."""
    img, small = WORKLOADS["imagegen-16k"], WORKLOADS["smallbatch-8"]
    w = bench.stage_bytes_flops(img, active=img.E)["gemm_w13_swiglu"]
    assert bench.gemm_bound(w["flops"], w["bytes"], 1699.4, 6769.8) == "tensor"
    w = bench.stage_bytes_flops(small, active=41)["gemm_w13_swiglu"]
    H, I, Is, N = small.H, small.I, small.I_s, small.T * small.k
    weights = 41 * 2 * I * H * 2 + 2 * Is * H * 2
    assert weights < w["bytes"] < weights * 1.01          # the weights are nearly all of it
    assert bench.gemm_bound(w["flops"], w["bytes"], 1699.4, 6769.8) == "hbm"
    d = bench.stage_bytes_flops(small, active=41)["gemm_down"]["bytes"]
    assert 41 * H * I * 2 + H * Is * 2 < d < (41 * H * I * 2 + H * Is * 2) * 1.01
    stages = _stages(0.01)
    stages["gemm_w13_swiglu"] = 0.32
    res = bench.finish_ours(_args(workload="smallbatch-8"), small, 1, 0, 10, 3, 5.7, stages, CLK,
                            None, {}, active=41)
    r = res["roofline"]
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["achieved"] == pytest.approx(w["bytes"] / 0.32e-3 / 1e9, rel=1e-3)
    assert res["stages"]["gemm_w13_swiglu"]["frac_hbm"] == pytest.approx(r["frac"], rel=1e-3)
    assert bench.finish_ours(_args(), img, 1, 0, 10, 3, 80.0, _stages(1.0), CLK, None,
                             {})["roofline"]["bound"] == "tensor"


def test_tensor_peak_follows_the_clock_record():
    """The matmul is measured against the burst matmul rate when the median
    SM clock of its timed steps stayed within 3% of the maximum (whatever an
    isolated power-cap sample says), else, and with no clock record, against
    the sustained rate.  Both measured rates and the nominal dense bf16 rate
    appear beside it."""
    wl = WORKLOADS["balanced-4k"]
    peaks, _ = bench.load_peaks()
    burst = peaks["bf16_tflops"]
    full = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []}
    capped_sample = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"]}
    for clk in (full, capped_sample):
        p, how = bench.tensor_peak(peaks, clk)
        assert p == pytest.approx(burst) and how.startswith("bf16_tflops (burst")
    p, how = bench.tensor_peak(peaks, CLK)
    assert p == pytest.approx(peaks["bf16_tflops_sustained"]) and "sustained" in how
    p, how = bench.tensor_peak(peaks, {})
    assert p == pytest.approx(peaks["bf16_tflops_sustained"])
    stages = _stages(0.1)
    stages["gemm_w13_swiglu"] = 0.2
    r = bench.finish_ours(_args(workload="balanced-4k"), wl, 1, 0, 10, 3, 4.5, stages, full,
                          None, {})["roofline"]
    flops = 4.0 * wl.T * wl.k * wl.H * wl.I
    assert r["peak"] == pytest.approx(burst, rel=1e-3)
    assert r["frac"] == pytest.approx(flops / 0.2e-3 / 1e12 / burst, rel=1e-3)
    assert r["frac_nominal_dense_bf16"] == pytest.approx(flops / 0.2e-3 / 1e12 / 2250.0, rel=1e-3)
    assert r["frac_of_sustained"] == pytest.approx(
        flops / 0.2e-3 / 1e12 / peaks["bf16_tflops_sustained"], rel=1e-3)
    r = bench.finish_ours(_args(workload="balanced-4k"), wl, 1, 0, 10, 3, 4.5, stages, CLK,
                          None, {})["roofline"]
    assert r["peak"] == pytest.approx(peaks["bf16_tflops_sustained"], rel=1e-3)
    assert r["frac_of_burst"] == pytest.approx(flops / 0.2e-3 / 1e12 / burst, rel=1e-3)
    assert r["frac_nominal_at_sampled_clock"] == pytest.approx(
        flops / 0.2e-3 / 1e12 / (2250.0 * 1700.0 / 2070.0), rel=1e-3)


def test_y_f32_mode_counts_fp32_routed_rows():
    """With fp32 routed expert outputs the down matmul writes and finalize
    reads four bytes per element instead of two."""
    wl = WORKLOADS["imagegen-16k"]
    N, H = wl.T * wl.k, wl.H
    a = bench.stage_bytes_flops(wl, active=wl.E)
    b = bench.stage_bytes_flops(wl, active=wl.E, y_f32=True)
    assert b["finalize"]["bytes"] - a["finalize"]["bytes"] == N * H * 2
    assert b["gemm_down"]["bytes"] - a["gemm_down"]["bytes"] == N * H * 2
    res = bench.finish_ours(_args(y_f32=True), wl, 1, 0, 10, 3, 80.0, _stages(1.0), CLK, None, {})
    assert res["config"]["routed_expert_outputs"].startswith("fp32")
    assert res["roofline"]["traffic"] is None


def test_gathered_rows_count_no_permute_pass():
    """With the rows gathered inside the w13 matmul (MOE_GATHER_A) the permute
    stage has no bytes, the step one launch fewer, and the recorded w13
    traffic (taken on the permute path's kernel) does not apply."""
    wl = WORKLOADS["imagegen-16k"]
    a = bench.stage_bytes_flops(wl, active=wl.E)
    b = bench.stage_bytes_flops(wl, active=wl.E, gather=True)
    assert a["permute"]["bytes"] > 0 and b["permute"]["bytes"] == 0
    assert b["gemm_w13_swiglu"] == a["gemm_w13_swiglu"]
    plain = bench.finish_ours(_args(), wl, 1, 0, 10, 3, 80.0, _stages(1.0), CLK, None, {})
    gath = bench.finish_ours(_args(), wl, 1, 0, 10, 3, 80.0, _stages(1.0), CLK, None, {},
                             gather=True)
    assert gath["gpu_launches"] == plain["gpu_launches"] - 10
    assert gath["roofline"]["traffic"] is None
    assert "gathered" in gath["config"]["w13_rows"]


def test_clock_summary_keeps_the_timed_window():
    """nvidia-smi samples before and after the timed region (idle clocks,
    low power) are left out of the clock record."""
    import datetime

    def line(t, mhz, watts, cap="Not Active"):
        ts = datetime.datetime.fromtimestamp(t).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
        return (f"{ts}, {mhz}, 2070, {watts}, 0x0, Not Active, Not Active, Not Active, "
                f"{cap}\n")
    t0 = 1_800_000_000.0
    lines = [line(t0 - 0.5, 2070, 150), line(t0 - 0.2, 2070, 160)]
    lines += [line(t0 + 0.05 * i, 1800 + i, 1300, "Active") for i in range(1, 8)]
    lines += [line(t0 + 0.9, 2070, 200)]
    s = bench.ClockSampler.summary(lines, t0, t0 + 0.4)
    assert s["samples"] == 7
    assert s["sm_mhz"] == 1804
    assert s["power_w_median"] == 1300
    assert s["reasons"] == ["sw_power_cap"]
    assert s["window_s"] == pytest.approx(0.4)
    everything = bench.ClockSampler.summary(lines)
    assert everything["samples"] == 10
