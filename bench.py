#!/usr/bin/env python
"""Benchmark of the GB300 MoE FFN layer forward (router -> dispatch -> grouped
SwiGLU GEMMs -> combine) through the C ABI of libcbmoe.so.

One step = one forward of the whole layer over one batch of T tokens of the
workload (default: the Mixtral-8x7B-shaped prefill layer, T=4096, d=4096,
f=14336, E=8, top-2, bf16).  Inputs are seeded synthetic data resident in HBM;
L2 is flushed (a 512 MB write) between timed steps, outside the timed events.
After the headline layer the metric's other layers are timed the same way
(decode-size weight streaming, the skewed 128-expert layer, the int8 layer)
and reported under "workloads"; `--workloads none` skips them.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--workloads A,B|none] [--impl reference]

Under torchrun each rank runs an independent replica of the layer on its own
GPU over its own T tokens (weak scaling, no collective in the data path); the
time is the max over ranks and `value` counts the tokens of all ranks.
`--impl reference` times the fp64 CPU oracle on the host cores instead
(rank 0 only).  Prints one JSON line on rank 0.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time
from datetime import datetime

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s; grouped-GEMM % of bf16 TC peak; decode weight GB/s % HBM"
DEFAULT_WORKLOAD = "mixtral_prefill"
# the metric's other layers: decode-size weight streaming, the skewed
# 128-expert layer and the int8 layer
EXTRA_WORKLOADS = ("mixtral_decode", "skewed", "int8")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
GEMM_SOURCES = [os.path.join(ROOT, "mixture_experts_router_gb300", "csrc", n)
                for n in ("grouped_gemm.cu", "grouped_gemm_pair.cu")]
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--workload", default=DEFAULT_WORKLOAD)
    p.add_argument("--shape", default=None, help="T,d,f,E,k of a custom layer (profiling cases)")
    p.add_argument("--wdtype", default="bf16", choices=["bf16", "int8", "int4", "fp8"],
                   help="expert weights of a --shape layer")
    p.add_argument("--bias", action="store_true", help="skewed router bias on a --shape layer")
    p.add_argument("--router", default="softmax", choices=["softmax", "raw", "hash"],
                   help="router variant: softmax top-k (default), raw-logit weights, or the hash router (k = 1)")
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--l2-flush-mb", type=int, default=512)
    p.add_argument("--e2e-steps", type=int, default=50)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=15.0, help="target CPU work of the oracle baseline")
    p.add_argument("--workloads", default=",".join(EXTRA_WORKLOADS),
                   help="further workloads timed after the headline one ('none' for the headline only)")
    p.add_argument("--sub-cpu-seconds", type=float, default=4.0,
                   help="target CPU work of each further workload's oracle sample")
    return p.parse_args(argv)


# ------------------------------------------------------------------ helpers
def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def algorithmic_work(shape, counts):
    """Algorithmic bytes / flops of each stage for one forward.  Expert FLOPs
    count routed rows only (padding rows of the 128-row tiles are waste)."""
    T, d, f, E, k = shape.T, shape.d, shape.f, shape.E, shape.k
    M = T * k
    eb = {"bf16": 2.0, "int8": 1.0, "int4": 0.5, "fp8": 1.0}[shape.wdtype]   # bytes per expert weight
    active = sum(1 for c in counts if c > 0)
    # + per-channel scales (int8, int4, fp8) and zero points (int4)
    side = (4 if shape.wdtype != "bf16" else 0) + (1 if shape.wdtype == "int4" else 0)
    wbytes = int(active * 3 * d * f * eb) + active * (2 * f + d) * side
    return {
        "router_bytes": T * d * 2 + (shape.hash_dims if shape.router == "hash" else E) * d * 2 + T * k * 8,
        "dispatch_bytes": T * d * 2 + M * d * 2 + 16 * M,
        # router and dispatch in one launch: x crosses HBM once
        "route_dispatch_fused_bytes": T * d * 2 + E * d * 2 + T * k * 8 + M * d * 2 + 16 * M,
        "gateup_flops": 4 * d * f * M,
        "down_flops": 2 * d * f * M,
        "combine_bytes": M * d * 4 + 8 * M + T * d * 2,
        "active_expert_weight_bytes": wbytes,
        "gateup_weight_bytes": int(active * 2 * d * f * eb),
        "down_weight_bytes": int(active * d * f * eb),
    }


class ClockSampler:
    """nvidia-smi samples (every 20 ms) of SM clock and throttle reasons."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device):
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "20", "-i", str(device)], stdout=self.file,
                                         stderr=subprocess.DEVNULL)
        except (FileNotFoundError, OSError):
            self.proc = None

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        self.file.flush()

    def summary(self, t0, t1):
        rows = []
        with open(self.file.name) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    ts = datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    rows.append((ts, float(parts[1]), float(parts[2]), parts[5:9]))
                except ValueError:
                    continue
        os.unlink(self.file.name)
        inside = [r for r in rows if t0 - 0.02 <= r[0] <= t1 + 0.02]
        nearest = not inside
        if nearest:  # a timed region shorter than the sampling interval: the samples closest to it
            inside = sorted(rows, key=lambda r: abs(r[0] - 0.5 * (t0 + t1)))[:2]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in inside for n, v in zip(names, r[3]) if v.lower().startswith("active")})
        out = {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": max(r[2] for r in inside),
               "reasons": reasons, "samples": len(inside)}
        if nearest:
            out["nearest"] = True
        return out


def gemm_source_digest(sources=None) -> str:
    """First 16 hex digits of the sha256 over grouped-GEMM sources (default: the
    bf16 kernels'; a traffic entry may name its own, relative to the package's
    csrc/)."""
    h = hashlib.sha256()
    paths = GEMM_SOURCES if sources is None else [os.path.join(ROOT, "mixture_experts_router_gb300", "csrc", s)
                                                  for s in sources]
    for path in paths:
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_traffic(kernel_key):
    """DRAM bytes per launch of a kernel from the committed ncu summary, or None
    when the kernel's source changed since the counters were taken."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    with open(TRAFFIC_FILE) as f:
        data = json.load(f)
    entry = data.get(kernel_key)
    if not entry:
        return None
    digest = gemm_source_digest(entry.get("sources"))
    if entry.get("source_sha256_16") != digest:
        return None
    return entry.get("dram_bytes_per_launch")


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value: float, world: int) -> float:
    """Max of a float over all ranks (a measurement collective, not part of the layer)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def config_block(shape, l2_mb):
    return {"workload": shape.name, "T": shape.T, "d_model": shape.d, "d_ff": shape.f, "n_experts": shape.E,
            "top_k": shape.k, "expert_weights": shape.wdtype, "router_bias": shape.bias,
            "router": shape.router + (f" ({shape.hash_dims} hash dims)" if shape.router == "hash" else ""),
            "l2": f"flushed between timed steps ({l2_mb} MB write, outside the timed events)",
            "parallelism": "replicas (token-sharded, no collective)"}


# ------------------------------------------------------- CPU oracle baseline
def oracle_baseline(shape, layer, target_seconds=15.0, threads=None):
    """Time the fp64 oracle (as it stands) on a bounded sample of tokens."""
    import numpy as np
    import oracle
    lib = oracle.load()
    threads = threads or host_cores()
    oracle.set_threads(threads)
    orc = oracle.Oracle(layer, lib)
    rng = np.random.default_rng(0)
    n = threads
    t0 = time.perf_counter()
    orc.forward(tokens=rng.choice(shape.T, n, replace=False).astype(np.int32))
    first = time.perf_counter() - t0
    more = max(0, int(n * (target_seconds - first) / max(first, 1e-6)))
    more = min(more, shape.T - n)
    total_tokens, total_time = n, first
    if more > 0:
        toks = rng.choice(shape.T, more, replace=False).astype(np.int32)
        t0 = time.perf_counter()
        orc.forward(tokens=toks)
        total_time += time.perf_counter() - t0
        total_tokens += more
    return {"value": total_tokens / total_time, "unit": "tokens/s", "cores": oracle.get_threads(lib),
            "kind": "oracle",
            "sample": f"{total_tokens} of the {shape.T} tokens (routing + k experts + combine per token, fp64, "
                      f"OpenMP over tokens), {total_time:.1f} s"}


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    import numpy as np
    import oracle
    import synth
    shape = workload_shape(args)
    layer = synth.make_layer(shape)
    threads = host_cores()
    lib = oracle.load()
    oracle.set_threads(threads)
    orc = oracle.Oracle(layer, lib)
    rng = np.random.default_rng(1)
    per_step = threads        # one token per thread: a bounded sample of the batch
    for _ in range(min(args.warmup, 3)):
        orc.forward(tokens=rng.choice(shape.T, per_step, replace=False).astype(np.int32))
    times = []
    for _ in range(args.steps):
        toks = rng.choice(shape.T, per_step, replace=False).astype(np.int32)
        t0 = time.perf_counter()
        orc.forward(tokens=toks)
        times.append(time.perf_counter() - t0)
    total = sum(times)
    value = per_step * args.steps / total
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded SplitMix64/Box-Muller, bf16 inputs)",
            "config": config_block(shape, args.l2_flush_mb),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": oracle.get_threads(lib), "kind": "oracle",
                             "sample": f"{per_step} tokens per step of the {shape.T}-token batch"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- our arm
def stage_report(shape, work, mean, names, pk, fused_rd=False):
    """Per-stage times with their algorithmic rates and roofline fractions.
    With fused_rd the router's launch also dispatches: the router stage holds
    both and the dispatch stage is empty."""
    hbm, tc_burst, tc_sus = pk["hbm_gbs"], pk["bf16_tflops"], pk.get("bf16_tflops_sustained", pk["bf16_tflops"])
    stages = {}
    for i, n in enumerate(names):
        s = mean[i] / 1e3
        if fused_rd and n == "router":
            b = work["route_dispatch_fused_bytes"]
            stages[n] = {"ms": mean[i], "gbs": b / s / 1e9, "frac_hbm": b / s / 1e9 / hbm,
                         "about": "router and dispatch in one launch (x read from HBM once)"}
        elif fused_rd and n == "dispatch":
            stages[n] = {"ms": mean[i], "about": "in the router's launch"}
        elif n in ("gateup_gemm", "down_gemm"):
            fl = work["gateup_flops" if n == "gateup_gemm" else "down_flops"]
            wb = work["gateup_weight_bytes" if n == "gateup_gemm" else "down_weight_bytes"]
            stages[n] = {"ms": mean[i], "tflops": fl / s / 1e12, "frac_tc": fl / s / 1e12 / tc_burst,
                         "frac_tc_sustained": fl / s / 1e12 / tc_sus,
                         "weight_gbs": wb / s / 1e9, "frac_hbm_weights": wb / s / 1e9 / hbm}
        else:
            b = work[n + "_bytes"]
            stages[n] = {"ms": mean[i], "gbs": b / s / 1e9, "frac_hbm": b / s / 1e9 / hbm}
    gemm_s = (mean[2] + mean[3]) / 1e3
    fl = work["gateup_flops"] + work["down_flops"]
    stages["grouped_gemms"] = {"ms": mean[2] + mean[3], "tflops": fl / gemm_s / 1e12,
                               "frac_tc": fl / gemm_s / 1e12 / tc_burst,
                               "frac_tc_sustained": fl / gemm_s / 1e12 / tc_sus,
                               "weight_gbs": work["active_expert_weight_bytes"] / gemm_s / 1e9,
                               "frac_hbm_weights": work["active_expert_weight_bytes"] / gemm_s / 1e9 / hbm}
    rd_s = (mean[0] + mean[1]) / 1e3
    rd_b = work["route_dispatch_fused_bytes"] if fused_rd else work["router_bytes"] + work["dispatch_bytes"]
    stages["router_dispatch"] = {"ms": mean[0] + mean[1], "gbs": rd_b / rd_s / 1e9, "frac_hbm": rd_b / rd_s / 1e9 / hbm,
                                 "bytes": rd_b}
    return stages


def roofline_of(shape, work, mean, names, pk, pk_kind, fused_rd=False):
    """The dominant (longest) stage against its roofline.  A GEMM whose FLOPs
    per weight byte exceed the ridge point is tensor-bound and is compared with
    the burst bf16 peak (it runs inside a millisecond-scale step); below the
    ridge (decode sizes) it streams weights and is compared with HBM."""
    hbm, tc_burst, tc_sus = pk["hbm_gbs"], pk["bf16_tflops"], pk.get("bf16_tflops_sustained", pk["bf16_tflops"])
    dom = max(range(len(names)), key=lambda i: mean[i])
    dname = names[dom]
    intensity = (work["gateup_flops"] + work["down_flops"]) / max(1, work["active_expert_weight_bytes"])
    ridge = tc_burst * 1e12 / (hbm * 1e9)
    if dname in ("gateup_gemm", "down_gemm") and intensity >= ridge:
        fl = work["gateup_flops" if dname == "gateup_gemm" else "down_flops"]
        achieved = fl / (mean[dom] / 1e3) / 1e12
        roof = {"kernel": dname, "bound": "tensor", "achieved": achieved, "peak": tc_burst, "unit": "TFLOP/s",
                "frac": achieved / tc_burst, "peak_kind": f"{pk_kind} bf16 dense burst",
                "peak_sustained": tc_sus, "frac_of_sustained": achieved / tc_sus}
        alg = fl
    elif dname in ("gateup_gemm", "down_gemm"):
        wb = work["gateup_weight_bytes" if dname == "gateup_gemm" else "down_weight_bytes"]
        achieved = wb / (mean[dom] / 1e3) / 1e9
        roof = {"kernel": dname, "bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                "frac": achieved / hbm, "peak_kind": f"{pk_kind} HBM copy"}
        alg = wb
    else:
        alg = work["route_dispatch_fused_bytes"] if (fused_rd and dname == "router") else work[dname + "_bytes"]
        achieved = alg / (mean[dom] / 1e3) / 1e9
        roof = {"kernel": dname, "bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                "frac": achieved / hbm, "peak_kind": f"{pk_kind} HBM copy"}
    roof["traffic"] = measured_traffic(f"{dname}:{shape.name}")
    roof["algorithmic_per_launch"] = alg
    return roof


def run_workload(shape, args, device, world, cpu_seconds):
    """Time one workload: the timed steps (no stage events), a stage-timed pass,
    host-buffer forwards end to end, and optionally the oracle on a sample.
    Returns the record (rank 0) or None."""
    import numpy as np
    import torch
    import mixture_experts_router_gb300 as cb
    import synth

    local = device.index
    layer = synth.make_layer(shape)

    def dev(a):
        if a is None:
            return None
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
        return torch.from_numpy(a).to(device)

    w = {n: dev(getattr(layer, n)) for n in ("wr", "bias", "wg", "wu", "wd", "sg", "su", "sd", "wh", "zg", "zu", "zd")}
    m = cb.MoELayer(shape.T, shape.d, shape.f, shape.E, shape.k, w["wr"], w["wg"], w["wu"], w["wd"],
                    router_bias=w["bias"], s_gate=w["sg"], s_up=w["su"], s_down=w["sd"], device=local,
                    stage_timing=True, router=shape.router, w_hash=w["wh"], z_gate=w["zg"], z_up=w["zu"],
                    z_down=w["zd"], wdtype=shape.wdtype)
    launches_per_forward = m.kernels_per_forward()
    del w
    torch.cuda.empty_cache()
    x = dev(layer.x)
    out = torch.empty((shape.T, shape.d), dtype=torch.bfloat16, device=device)
    flush = torch.empty(args.l2_flush_mb << 20, dtype=torch.uint8, device=device)
    stream = torch.cuda.Stream(device)

    with torch.cuda.stream(stream):
        # the timed steps run without the stage events (nodes between the
        # kernels that cost a few microseconds each); a second pass of the same
        # steps with them on gives the per-stage times
        m.set_stage_timing(False)
        for _ in range(max(args.warmup, 3)):
            flush.zero_()
            m.forward(x, out, stream=stream)
        stream.synchronize()
        st = m.last_error()
        if st != cb.CB_OK:
            raise cb.CbMoeError(st, "warm-up forward")

        sampler = ClockSampler(local)
        time.sleep(0.3)
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        t_wall0 = time.time()
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        for i in range(args.steps):
            flush.zero_()
            starts[i].record(stream)
            m.forward(x, out, stream=stream)
            ends[i].record(stream)
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        t_wall1 = time.time()
        time.sleep(0.2)
        sampler.stop()
        clocks = sampler.summary(t_wall0, t_wall1)
        st = m.last_error()
        if st != cb.CB_OK:
            raise cb.CbMoeError(st, "timed forward")
        step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
        total_ms = max_over_ranks(sum(step_ms), world)

        # stage pass: the same steps with CUDA events between the stages
        m.set_stage_timing(True)
        for _ in range(3):
            flush.zero_()
            m.forward(x, out, stream=stream)
        stage_ms = []
        stage_step_ms = 0.0
        for i in range(args.steps):
            flush.zero_()
            starts[i].record(stream)
            m.forward(x, out, stream=stream)
            ends[i].record(stream)
            stage_ms.append(m.stage_times())   # waits for this step's last stage event
            stage_step_ms += starts[i].elapsed_time(ends[i])
        m.set_stage_timing(False)
        st = m.last_error()
        if st != cb.CB_OK:
            raise cb.CbMoeError(st, "stage-timed forward")

        # end to end through the host-buffer entry point (pinned host memory): k2
        # back-to-back calls, each copying its x in and its out back, timed by the
        # host clock between two device synchronisations (no L2 flush: per step
        # every workload but decode moves more than L2, and decode streams 2.8 GB
        # of weights)
        xh = torch.from_numpy(layer.x.view(np.int16)).pin_memory()
        oh = torch.empty_like(xh).pin_memory()
        k2 = max(1, min(args.e2e_steps, args.steps))
        for _ in range(3):
            m.forward_host(xh, oh, stream=stream)
        torch.cuda.synchronize()
        e2e_sampler = ClockSampler(local)
        time.sleep(0.3)
        if world > 1:
            torch.distributed.barrier()
        t_e0 = time.time()
        t0 = time.perf_counter()
        for i in range(k2):
            m.forward_host(xh, oh, stream=stream)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks((time.perf_counter() - t0) * 1e3, world)
        t_e1 = time.time()
        time.sleep(0.2)
        e2e_sampler.stop()
        e2e_clocks = e2e_sampler.summary(t_e0, t_e1)
        st = m.last_error()
        if st != cb.CB_OK:
            raise cb.CbMoeError(st, "host forward")
        routing = m.routing()
        counts = torch.empty(shape.E, dtype=torch.int32, device=device)
        cb.copy_from_device(counts, routing.counts, 4 * shape.E)
        counts = counts.cpu().tolist()

    m.close()
    del x, out, flush, xh, oh
    torch.cuda.empty_cache()
    if int(os.environ.get("RANK", "0")) != 0:
        return None

    pk, pk_kind = peaks()
    work = algorithmic_work(shape, counts)
    mean = [statistics.mean(s[i] for s in stage_ms) for i in range(5)]
    # router (1 launch) + dispatch + two GEMMs + combine: 4 launches means the
    # router's launch also dispatched
    fused_rd = shape.router != "hash" and launches_per_forward == 4
    names = cb.STAGE_NAMES
    value = shape.T * world * args.steps / (total_ms / 1e3)
    ms = total_ms / args.steps
    rec = {
        "value": value, "unit": "tokens/s", "ms_per_step": ms, "steps": args.steps, "warmup": args.warmup,
        "dtype": shape.wdtype, "config": config_block(shape, args.l2_flush_mb),
        "e2e": {"value": shape.T * world * k2 / (e2e_ms / 1e3), "unit": "tokens/s",
                "h2d_bytes_per_step": shape.T * shape.d * 2, "d2h_bytes_per_step": shape.T * shape.d * 2,
                "steps": k2, "timing": "host clock over back-to-back calls", "clocks": e2e_clocks,
                "api": "cb_moe_forward_host (pinned host x and out; input copy, layer and output copy on the "
                       "handle's three streams, successive calls overlapping)"},
        "gpu_launches": launches_per_forward * args.steps,
        "roofline": roofline_of(shape, work, mean, names, pk, pk_kind, fused_rd),
        "stages": stage_report(shape, work, mean, names, pk, fused_rd),
        "stage_pass": {"ms_per_step": stage_step_ms / args.steps,
                       "about": "the stage times and the roofline come from a second pass of the same steps "
                                "with CUDA events between the stages; ms_per_step and value from the first, "
                                "without them"},
        "layer_weight_streaming": {"active_expert_weight_bytes": work["active_expert_weight_bytes"],
                                   "gbs": work["active_expert_weight_bytes"] / (ms / 1e3) / 1e9,
                                   "frac_hbm": work["active_expert_weight_bytes"] / (ms / 1e3) / 1e9 / pk["hbm_gbs"],
                                   "about": "activated-expert weight bytes over the whole layer's step time"},
        "expert_rows": {"active_experts": sum(1 for c in counts if c > 0), "max_rows": max(counts),
                        "min_rows": min(counts)},
        "clocks": clocks,
    }
    if world == 1 and cpu_seconds > 0:
        rec["cpu_baseline"] = oracle_baseline(shape, layer, cpu_seconds)
    return rec


def run_ours(args):
    import torch
    import synth

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    device = torch.device("cuda", local)
    shape = workload_shape(args)
    head = run_workload(shape, args, device, world, 0.0 if args.no_cpu_baseline else args.cpu_seconds)
    extra = {}
    names = [] if args.shape or args.workloads in ("", "none") else \
        [n for n in args.workloads.split(",") if n != shape.name]
    for name in names:
        sub = synth.with_router(synth.WORKLOADS[name], args.router)
        rec = run_workload(sub, args, device, world, 0.0 if args.no_cpu_baseline else args.sub_cpu_seconds)
        if rec is not None:
            extra[name] = rec
    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return 0

    pk, pk_kind = peaks()
    line = {
        "metric": METRIC, "value": head["value"], "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": shape.wdtype,
        "data": "synthetic (seeded SplitMix64/Box-Muller; x ~ N(0,1), weights ~ N(0, 0.02^2), bf16)",
        "config": head["config"],
    }
    for key in ("e2e", "gpu_launches", "roofline", "stages", "stage_pass", "layer_weight_streaming",
                "expert_rows", "clocks", "cpu_baseline"):
        if key in head:
            line[key] = head[key]
    line["peaks"] = {"hbm_gbs": pk["hbm_gbs"], "bf16_tflops": pk["bf16_tflops"],
                     "bf16_tflops_sustained": pk.get("bf16_tflops_sustained"), "kind": pk_kind}
    if extra:
        line["workloads"] = extra
        line["workloads_about"] = ("the other layers of the metric, each timed the same way after the headline "
                                   "one (its own steps, stages, roofline, clocks, end-to-end leg and oracle "
                                   "sample); value and e2e above are the headline layer's")
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def workload_shape(args):
    import synth
    if args.shape:
        T, d, f, E, k = (int(v) for v in args.shape.split(","))
        name = f"custom_T{T}_d{d}_f{f}_E{E}_k{k}" + (f"_{args.wdtype}" if args.wdtype != "bf16" else "") + \
            ("_bias" if args.bias else "")
        return synth.with_router(synth.custom_shape(name, T=T, d=d, f=f, E=E, k=k, wdtype=args.wdtype,
                                                    bias=args.bias, seed=1100), args.router)
    return synth.with_router(synth.WORKLOADS[args.workload], args.router)


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
