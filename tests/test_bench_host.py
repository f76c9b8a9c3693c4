"""Host logic of bench.py (no GPU): the algorithmic work it divides by, the
stage and roofline arithmetic, and the clock sampler's parsing.

The byte and FLOP counts are pinned to the figures of the hot-path scope
table for the Mixtral-shaped layers (router 33.7 MB, dispatch ~101 MB,
combine ~168 MB, experts 2.886 TFLOP at prefill; 2.819 GB of activated
expert weights at decode), which follow from the configurations' shapes
alone, not from bench.py."""
import json
import os
import time

import pytest

import bench
import synth


def work_of(name, counts=None):
    shape = synth.WORKLOADS[name]
    if counts is None:
        counts = [1] * shape.E  # every expert active
    return shape, bench.algorithmic_work(shape, counts)


def test_prefill_work_matches_the_scope_table():
    shape, w = work_of("mixtral_prefill")
    assert w["router_bytes"] == pytest.approx(33.7e6, rel=2e-3)
    assert w["dispatch_bytes"] == pytest.approx(101e6, rel=1e-2)
    assert w["combine_bytes"] == pytest.approx(168e6, rel=1e-2)
    assert w["gateup_flops"] + w["down_flops"] == pytest.approx(2.886e12, rel=1e-3)
    # x crosses HBM once in the one-launch form: the router's and the dispatch's bytes less one x
    x = shape.T * shape.d * 2
    assert w["route_dispatch_fused_bytes"] == w["router_bytes"] + w["dispatch_bytes"] - x


def test_decode_weight_bytes_match_the_scope_table():
    _, w = work_of("mixtral_decode")
    assert w["active_expert_weight_bytes"] == pytest.approx(2.819e9, rel=1e-3)
    assert w["gateup_weight_bytes"] + w["down_weight_bytes"] == w["active_expert_weight_bytes"]


def test_quantised_weight_bytes_count_the_scales():
    shape, w = work_of("int8")
    d, f, E = shape.d, shape.f, shape.E
    assert w["active_expert_weight_bytes"] == 3 * d * f * E + E * (2 * f + d) * 4
    assert w["active_expert_weight_bytes"] == pytest.approx(1.2096e9, rel=1e-3)


def test_inactive_experts_carry_no_weight_bytes():
    shape = synth.WORKLOADS["skewed"]
    counts = [0] * shape.E
    counts[3] = 10
    counts[7] = 5
    w = bench.algorithmic_work(shape, counts)
    assert w["active_expert_weight_bytes"] == 2 * 3 * shape.d * shape.f * 2


PEAKS = {"hbm_gbs": 6783.8, "bf16_tflops": 1909.0, "bf16_tflops_sustained": 1725.4}
NAMES = ["router", "dispatch", "gateup_gemm", "down_gemm", "combine"]


def test_stage_report_with_the_one_launch_router_and_dispatch():
    shape, w = work_of("skewed")
    mean = [0.0585, 0.0021, 0.1423, 0.0988, 0.0564]   # ms
    st = bench.stage_report(shape, w, mean, NAMES, PEAKS, fused_rd=True)
    assert st["router"]["gbs"] == pytest.approx(w["route_dispatch_fused_bytes"] / 0.0585e-3 / 1e9)
    assert "gbs" not in st["dispatch"]
    assert st["router_dispatch"]["bytes"] == w["route_dispatch_fused_bytes"]
    assert st["router_dispatch"]["ms"] == pytest.approx(0.0606)
    tf = w["gateup_flops"] / 0.1423e-3 / 1e12
    assert st["gateup_gemm"]["tflops"] == pytest.approx(tf)
    assert st["gateup_gemm"]["frac_tc"] == pytest.approx(tf / 1909.0)
    assert st["grouped_gemms"]["ms"] == pytest.approx(0.1423 + 0.0988)
    sep = bench.stage_report(shape, w, mean, NAMES, PEAKS, fused_rd=False)
    assert sep["router_dispatch"]["bytes"] == w["router_bytes"] + w["dispatch_bytes"]


def test_roofline_picks_the_bound_by_intensity():
    shape, w = work_of("mixtral_prefill")
    roof = bench.roofline_of(shape, w, [0.034, 0.002, 1.116, 0.583, 0.030], NAMES, PEAKS, "measured")
    assert roof["kernel"] == "gateup_gemm" and roof["bound"] == "tensor" and roof["unit"] == "TFLOP/s"
    assert roof["peak"] == 1909.0                       # the burst peak, not the sustained one
    assert roof["frac"] == pytest.approx(w["gateup_flops"] / 1.116e-3 / 1e12 / 1909.0)
    shape, w = work_of("mixtral_decode")
    roof = bench.roofline_of(shape, w, [0.015, 0.002, 0.300, 0.156, 0.008], NAMES, PEAKS, "measured")
    assert roof["bound"] == "hbm" and roof["unit"] == "GB/s"
    assert roof["achieved"] == pytest.approx(w["gateup_weight_bytes"] / 0.300e-3 / 1e9)


def write_samples(sampler, rows):
    with open(sampler.file.name, "w") as f:
        for ts, mhz, reasons in rows:
            stamp = time.strftime("%Y/%m/%d %H:%M:%S", time.localtime(ts)) + f".{int((ts % 1) * 1000):03d}"
            act = ["Active" if r in reasons else "Not Active" for r in
                   ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")]
            f.write(f"{stamp}, {mhz}, 2070, 900.00, 0x0000000000000000, {', '.join(act)}\n")


def test_clock_samples_inside_the_timed_region():
    s = bench.ClockSampler(device=0)
    s.stop()
    t0 = float(int(time.time())) + 0.5
    write_samples(s, [(t0 - 1.0, 1000, ()), (t0 + 0.01, 2070, ()), (t0 + 0.03, 1950, ("sw_power_cap",)),
                      (t0 + 0.05, 2070, ()), (t0 + 1.0, 900, ("hw_slowdown",))])
    c = s.summary(t0, t0 + 0.05)
    assert c["samples"] == 3 and c["sm_mhz"] == 2070 and c["reasons"] == ["sw_power_cap"]
    assert "nearest" not in c


def test_clock_samples_nearest_when_none_fall_inside():
    s = bench.ClockSampler(device=0)
    s.stop()
    t0 = float(int(time.time())) + 0.5
    write_samples(s, [(t0 - 0.2, 2070, ()), (t0 + 0.15, 2000, ()), (t0 + 0.6, 800, ("hw_slowdown",))])
    c = s.summary(t0, t0 + 0.01)
    assert c["nearest"] is True and c["samples"] == 2
    assert c["reasons"] == [] and c["sm_mhz"] == pytest.approx(2035)
