#!/usr/bin/env python
"""Benchmark of the fused conv2d + BatchNorm + SiLU layer on GB300.

One *step* is one pass of the whole hot path over the five YOLO-shaped
layers (tiny, stem, downsample, pointwise, deep), each on its own synthetic
input: the BN fold of every layer (one batched launch), then each layer's
fused forward.  ``value`` is the step's
algorithmic work (2*M*C_out*C*R*S summed over the layers, padding not
counted) divided by the device time of the timed steps, in TFLOP/s, summed
over ranks (each rank runs its own replica: weak scaling, no collective on
the data path).

Timing: W warm-up steps, then K steps between two CUDA events on the
launching stream, bracketed by a barrier and torch.cuda.synchronize() on
both sides; max over ranks.  Inputs rotate over 3 buffer sets (about 426 MB
touched per rotation, more than three times the 129 MB L2), so each step
reads its data from HBM.  The step is replayed from one CUDA graph captured
from the API calls (six launches through Python per step would make the host
the bottleneck).  The dominant layer's launch duration (the ``roofline``
object) comes from a second timed run of the same steps whose graphs carry
event-record nodes around that forward: the nodes cut the programmatic-launch
overlap into it, so they stay out of the run that gives ``value``.  Per-layer
times in ``per_layer`` come from two separate passes: each call alone with the
L2 flushed before it, and each layer's forward back to back in a CUDA graph
over enough buffer sets that their rotation exceeds the L2.  SM clocks and throttle reasons are sampled with nvidia-smi during
the timed region.

``--impl reference`` times the fp64 CPU oracle on the host cores instead
(the reference arm; a bounded sample of the same workload per step).

Prints exactly one JSON line on rank 0.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from conv2d_batchnorm_silu_gb300.synthetic import (LAYERS, LAYER_ORDER,  # noqa: E402
                                                   bits_to_torch_bf16, make_layer_inputs)

METRIC = "fused conv+BN+SiLU TFLOP/s and % of conv roofline on 1 GB300"
UNIT = "TFLOP/s"
WORKLOAD = ("five YOLO-shaped fused conv+BN+SiLU layers per step: one batched BN fold of all "
            "layers, then each fused forward once: tiny 1x32x32x16->32 3x3s1p1, "
            "stem 1x640x640x3->16 3x3s2p1, "
            "down 16x160x160x64->128 3x3s2p1, pointwise 16x40x40x256->256 1x1, "
            "deep 32x20x20x512->512 3x3s1p1; NHWC bf16 x, KRSC bf16 W, fp32 BN")
DOMINANT = "deep"
ROTATION = 3
CLOCK_WINDOW_S = 1.0
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
CLOCK_FIELDS = ("timestamp,uuid,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-baseline-seconds", type=float, default=12.0)
    ap.add_argument("--reference-budget-seconds", type=float, default=120.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--layers", default=",".join(LAYER_ORDER),
                    help="comma-separated subset of layers in the step (default: all five)")
    ap.add_argument("--iso-iters", type=int, default=30,
                    help="calls per layer for the per-layer (L2-flushed) timings")
    ap.add_argument("--no-unfused", action="store_true",
                    help="skip the fused-vs-unfused comparison (conv, BN and SiLU as three kernels)")
    ap.add_argument("--no-epilogues", action="store_true",
                    help="skip the per-layer timing of the other epilogues (identity, ReLU, residual add)")
    ap.add_argument("--b2b-replays", type=int, default=20,
                    help="graph replays for the back-to-back per-layer times (0: skip)")
    ap.add_argument("--no-gemm-context", action="store_true",
                    help="skip timing cuBLAS on plain GEMMs of the pointwise and deep layers' sizes")
    ap.add_argument("--clock-window-s", type=float, default=CLOCK_WINDOW_S,
                    help="seconds of the same step replayed right after the timed steps, inside the "
                         "clock record (0: the timed steps alone)")
    ap.add_argument("--no-graphs", action="store_true",
                    help="launch through the API each step instead of replaying CUDA graphs")
    args = ap.parse_args(argv)
    args.layers = tuple(n for n in LAYER_ORDER if n in args.layers.split(","))
    if not args.layers:
        ap.error("--layers selects no known layer")
    return args


# ------------------------------------------------------------------ distributed helpers
def dist_env() -> tuple[int, int, int]:
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def dist_init(world: int, use_cuda: bool):
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend="nccl" if use_cuda else "gloo",
                                             init_method="env://")


def barrier(world: int):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(value: float, world: int, device=None) -> float:
    """The largest `value` across ranks (every rank receives it)."""
    if world <= 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def aggregate_throughput(units_per_rank: float, world: int, seconds_max: float) -> float:
    """Whole-job throughput: the units all ranks processed over the slowest rank's time."""
    return units_per_rank * world / seconds_max


# ------------------------------------------------------------------ peaks, clocks
def load_peaks() -> tuple[dict, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons while the timed region runs."""

    def __init__(self, uuid: str | None, interval_ms: int = 50):
        self.uuid = uuid
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(interval_ms)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                text=True)
        except OSError:
            self.proc = None

    def stop(self, t0: float | None = None, t1: float | None = None) -> dict | None:
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=10)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        return summarize_clocks(out, self.uuid, t0, t1)


def summarize_clocks(csv_text: str, uuid: str | None, t0: float | None = None,
                     t1: float | None = None) -> dict | None:
    """Median SM clock, max clock and throttle reasons from nvidia-smi CSV samples.

    Only samples whose timestamp falls in [t0, t1] (host wall time) count, when given.
    """
    import datetime
    sm, sm_max, power, reasons = [], [], [], set()
    names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
    for line in csv_text.splitlines():
        parts = [p.strip() for p in line.split(",")]
        if len(parts) < 11:
            continue
        if uuid and uuid not in parts[1]:
            continue
        if t0 is not None and t1 is not None:
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                continue
            if ts < t0 or ts > t1:
                continue
        try:
            sm.append(float(parts[3]))
            sm_max.append(float(parts[4]))
            power.append(float(parts[5]))
        except ValueError:
            continue
        for name, val in zip(names, parts[7:11]):
            if val.lower() == "active":
                reasons.add(name)
    if not sm:
        return None
    return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(sm_max),
            "power_w_max": max(power) if power else None, "samples": len(sm),
            "reasons": sorted(reasons)}


def device_uuid(dev_index: int) -> str | None:
    try:
        u = torch.cuda.get_device_properties(dev_index).uuid
        return str(u)
    except Exception:
        return None


# The sources of the tensor-core kernels (the dominant layer's and the others' whose DRAM
# counters profiles/dram_traffic.json records).
TC_KERNEL_SOURCES = ("tc_conv.cu", "tc_cmajor.cu", "tc_gather.cu", "ptx.cuh", "epilogue.cuh", "cbs_internal.h")


def kernel_source_sha(names=TC_KERNEL_SOURCES) -> str:
    """Hash of the tensor-core kernels' sources: DRAM counters recorded for them in
    profiles/dram_traffic.json are used only while the hash still matches."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "conv2d_batchnorm_silu_gb300", "csrc")
    for name in sorted(names):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(layer: str) -> float | None:
    """DRAM bytes per launch from the committed ncu summary, if taken on the current kernels."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    if d.get("kernel_source_sha") != kernel_source_sha():
        return None
    ent = d.get("layers", {}).get(layer)
    return float(ent["dram_bytes_per_launch"]) if ent else None


# ------------------------------------------------------------------ the GPU arm
class LayerBuffers:
    """Device tensors of one layer instance (inputs, folded BN, output)."""

    def __init__(self, inp, dev):
        sh = inp.shape
        self.shape = sh
        self.x = bits_to_torch_bf16(inp.x_bits).to(dev)
        self.w = bits_to_torch_bf16(inp.w_bits).to(dev)
        self.g, self.b, self.m, self.v = (torch.from_numpy(a).to(dev)
                                          for a in (inp.gamma, inp.beta, inp.mean, inp.var))
        self.eps = inp.eps
        self.scale = torch.empty(sh.k, dtype=torch.float32, device=dev)
        self.bias = torch.empty(sh.k, dtype=torch.float32, device=dev)
        self.y = torch.empty((sh.n, sh.ho, sh.wo, sh.k), dtype=torch.bfloat16, device=dev)


def run_ours(args, rank, world, local_rank):
    from conv2d_batchnorm_silu_gb300 import _build
    _build.build()
    from conv2d_batchnorm_silu_gb300 import capi

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    dist_init(world, True)
    layers = args.layers
    dominant = DOMINANT if DOMINANT in layers else max(layers, key=lambda n: LAYERS[n].flops)
    stream = torch.cuda.Stream(dev)
    inputs = {name: make_layer_inputs(LAYERS[name]) for name in layers}
    sets = [{name: LayerBuffers(inputs[name], dev) for name in layers} for _ in range(ROTATION)]
    flops_step = sum(LAYERS[n].flops for n in layers)
    launches_per_step = 1 + len(layers)
    # One batched BN fold per buffer set: every layer's scale and bias in one launch.
    fold_batches = [capi.FoldBatch([(lb.g, lb.b, lb.m, lb.v, lb.eps, lb.scale, lb.bias)
                                    for lb in (bufs[n] for n in layers)]) for bufs in sets]

    def forward_call(lb, strm):
        sh = lb.shape
        capi.forward(lb.x, lb.w, lb.scale, lb.bias, sh.stride, sh.pad, y=lb.y, stream=strm)

    # The step in launch order, split around the dominant layer's forward so that
    # CUDA events on the stream can bracket exactly that kernel.
    def segments(i):
        bufs = sets[i]
        pre, post, dom, seen = [lambda s, fb=fold_batches[i]: fb(s)], [], None, False
        for name in layers:
            if name == dominant:
                seen = True
                dom = (lambda s, lb=bufs[name]: forward_call(lb, s))
            else:
                (post if seen else pre).append(lambda s, lb=bufs[name]: forward_call(lb, s))
        return pre, dom, post

    # Warm up through the API (first calls encode tensor maps and set kernel attributes).
    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 3)):
            pre, dom, post = segments(i % ROTATION)
            for f in pre + [dom] + post:
                f(stream)
    torch.cuda.synchronize()
    capi.check(stream)

    # The timed steps: one CUDA graph per buffer set holding the whole step (or, with
    # --no-graphs, the API calls themselves, with events recorded around the dominant
    # layer's forward).
    def capture(calls):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for f in calls:
                f(None)
        return g

    if args.no_graphs:
        plan = [segments(i) for i in range(ROTATION)]
    else:
        plan = [capture(pre + [dom] + post) for pre, dom, post in (segments(i) for i in range(ROTATION))]
    torch.cuda.synchronize()

    def step(i, ev=None):
        if not args.no_graphs:
            plan[i % ROTATION].replay()
            return
        pre, dom, post = plan[i % ROTATION]
        for f in pre:
            f(stream)
        if ev is not None:
            ev[0].record(stream)
        dom(stream)
        if ev is not None:
            ev[1].record(stream)
        for f in post:
            f(stream)

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            step(i)
    torch.cuda.synchronize()
    capi.check(stream)

    K = args.steps
    dom_ev = ([torch.cuda.Event(enable_timing=True) for _ in range(K)],
              [torch.cuda.Event(enable_timing=True) for _ in range(K)]) if args.no_graphs else None
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(device_uuid(local_rank))
    time.sleep(0.5)  # let the sampler start
    barrier(world)
    torch.cuda.synchronize()
    t_wall0 = time.time()
    torch.cuda.nvtx.range_push("timed steps")
    with torch.cuda.stream(stream):
        start.record(stream)
        for i in range(K):
            step(i, None if dom_ev is None else (dom_ev[0][i], dom_ev[1][i]))
        end.record(stream)
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()
    # The clock record covers the timed steps and the same step replayed for
    # CLOCK_WINDOW_S more seconds right after them, so that a short timed region
    # (--steps 20 lasts about 2 ms) still has nvidia-smi samples under the same load.
    torch.cuda.nvtx.range_push("clock window")
    with torch.cuda.stream(stream):
        i = 0
        while time.time() - t_wall0 < args.clock_window_s:
            for _ in range(200):
                step(i)
                i += 1
            torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()
    t_wall1 = time.time()
    barrier(world)
    clocks = sampler.stop(t_wall0, t_wall1)
    if clocks is not None:
        clocks["window"] = (f"the timed steps plus the same step replayed right after them, "
                            f"{t_wall1 - t_wall0:.2f} s in all, sampled every 50 ms")
    capi.check(stream)
    elapsed_s = start.elapsed_time(end) / 1e3
    elapsed_max = max_over_ranks(elapsed_s, world, dev)
    if dom_ev is not None:
        dom_us, dom_how = 1e3 * float(np.mean([a.elapsed_time(b) for a, b in zip(*dom_ev)])), \
            f"events around the forward in each of the {K} timed steps"
    else:
        dom_us, dom_how = dominant_in_step(segments, capture, stream, args.warmup, min(K, 600))
    capi.check(stream)

    peaks, peak_src = load_peaks()
    b2b = layer_times_back_to_back(capi, sets, inputs, layers, stream, dev,
                                   args.b2b_replays) if args.b2b_replays > 0 else None
    torch.cuda.nvtx.range_push("per-layer timings")
    iso = isolated_layer_times(capi, sets, layers, stream, dev, args.iso_iters)
    iso_clean = isolated_layer_times(capi, sets, layers, stream, dev, args.iso_iters, clean=True)
    torch.cuda.nvtx.range_pop()
    per_layer = {}
    for n in layers:
        sh = LAYERS[n]
        t = iso[n] * 1e-6
        t_flop = sh.flops / (peaks["bf16_tflops"] * 1e12)
        t_byte = sh.compulsory_bytes / (peaks["hbm_gbs"] * 1e9)
        pl = capi.plan(sh.n, sh.h, sh.w, sh.c, sh.k, sh.r, sh.s, sh.stride, sh.pad)
        per_layer[n] = {"us_per_call": round(iso[n], 3),
                        "us_per_call_clean_l2": round(iso_clean[n], 3),
                        "roofline_frac_clean_l2": round(max(t_flop, t_byte) / (iso_clean[n] * 1e-6), 4),
                        "tflops": round(sh.flops / t / 1e12, 2),
                        "gbs": round(sh.compulsory_bytes / t / 1e9, 1),
                        "roofline_us": round(max(t_flop, t_byte) * 1e6, 3),
                        "roofline_frac": round(max(t_flop, t_byte) / t, 4),
                        "bound": "tensor" if t_flop >= t_byte else "hbm",
                        "kernel": pl["algo"], "tile": [pl["block_m"], pl["block_n"], pl["block_k"]],
                        "grid": pl["grid"]}
        if b2b is not None:
            tb = b2b[n]["us"] * 1e-6
            per_layer[n]["us_back_to_back"] = round(b2b[n]["us"], 3)
            per_layer[n]["roofline_frac_back_to_back"] = round(max(t_flop, t_byte) / tb, 4)
            if b2b[n]["l2_resident"]:
                per_layer[n]["back_to_back_l2_resident"] = True
    dom = LAYERS[dominant]
    dom_t = dom_us * 1e-6
    if per_layer[dominant]["bound"] == "tensor":
        achieved, peak, unit, bound = dom.flops / dom_t / 1e12, peaks["bf16_tflops"], "TFLOP/s", "tensor"
        per_launch = {"algorithmic_flops_per_launch": dom.flops}
    else:
        achieved, peak, unit, bound = dom.compulsory_bytes / dom_t / 1e9, peaks["hbm_gbs"], "GB/s", "hbm"
        per_launch = {"algorithmic_bytes_per_launch": dom.compulsory_bytes}
    roofline = {"bound": bound, "achieved": round(achieved, 2), "peak": peak, "unit": unit,
                "frac": round(achieved / peak, 4), "traffic": recorded_traffic(dominant),
                "kernel": f"{dominant} layer forward ({per_layer[dominant]['kernel']})",
                "launch_us": round(dom_us, 3),
                "launch_timing": dom_how,
                "peak_source": f"{peak_src} ({'bf16 dense burst' if bound == 'tensor' else 'HBM copy'})",
                **per_launch}

    fusion = None if args.no_unfused else \
        fusion_comparison(capi, sets, layers, stream, dev, args.iso_iters, iso)

    epilogues = None if args.no_epilogues else \
        epilogue_variants(capi, sets, layers, stream, dev, args.iso_iters, iso)

    gemm = None if args.no_gemm_context else gemm_context(dev, layers, iso, args.iso_iters)

    e2e = run_e2e(args, capi, inputs, dev, stream, world) if args.e2e_steps > 0 else None
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args.cpu_baseline_seconds, layers)

    value = aggregate_throughput(flops_step * K, world, elapsed_max) / 1e12
    workload = WORKLOAD if layers == LAYER_ORDER else \
        "subset of the five-layer step: " + ", ".join(LAYERS[n].description for n in layers)
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(elapsed_max / K * 1e3, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded PCG64: x~N(0,1), W~N(0,2/fan_in), BN gamma~U(.5,1.5), "
                "beta,mean~N(0,.1), var~U(.5,2), eps=1e-3)",
        "config": {"workload": workload, "flops_per_step": flops_step,
                   "l2": f"{ROTATION} rotating buffer sets (~426 MB per rotation > 129 MB L2); "
                         "per_layer times: L2 flushed (512 MB write) before each call",
                   "launch": ("direct API calls" if args.no_graphs else
                              "one CUDA graph per step captured from the API calls, replayed"),
                   "parallelism": f"replicas x{world} (each rank runs the full step)"},
        "roofline": roofline,
        "layers_roofline_frac": {n: {"isolated": per_layer[n]["roofline_frac"],
                                     "isolated_clean_l2": per_layer[n].get("roofline_frac_clean_l2"),
                                     "back_to_back": per_layer[n].get("roofline_frac_back_to_back")}
                                 for n in layers},
        "per_layer": per_layer,
        "per_layer_timing": {
            "us_per_call": "median of isolated calls, a 512 MB L2-flushing write before each; "
                           "includes the launch gap of a lone call",
            "us_per_call_clean_l2": "as us_per_call, with a 512 MB read after the flushing write, so the "
                                    "flush's dirty lines are written back before the call, not during it",
            "us_back_to_back": (None if b2b is None else
                                "one CUDA graph of G forwards of the layer back to back, each on its own "
                                "buffer set (rotation > 160 MB unless marked l2_resident), replayed "
                                f"{args.b2b_replays} times; graph time / (replays x G)"),
            "back_to_back_sets": None if b2b is None else {n: b2b[n]["calls_per_graph"] for n in b2b}},
        "gemm_context": gemm,
        "fusion": fusion,
        "epilogues": epilogues,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches_per_step * K,
        "clocks": clocks,
        "peaks": {**peaks, "source": peak_src},
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    barrier(world)


def _cu_event_record_external():
    """cuEventRecordWithFlags from the CUDA driver, or None."""
    import ctypes
    try:
        lib = ctypes.CDLL("libcuda.so.1")
        fn = lib.cuEventRecordWithFlags
    except (OSError, AttributeError):
        return None
    fn.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_uint]
    fn.restype = ctypes.c_int
    return fn


def dominant_in_step(segments, capture, stream, warmup, steps):
    """Launch duration of the dominant layer's forward inside the step: a second timed
    run of `steps` steps whose graphs carry event-record nodes around that forward.  The
    nodes cut the programmatic-launch edge into the forward, so they stay out of the run
    that gives the step's throughput.  Where the driver refuses the nodes, the step is
    split into three graphs with events recorded between their launches."""
    events = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(ROTATION)]
    graphs = capture_steps_with_events(segments, events, stream)
    with torch.cuda.stream(stream):
        if graphs is not None:
            for i in range(warmup + steps):
                graphs[i % ROTATION].replay()
            torch.cuda.synchronize()
            us = 1e3 * float(np.mean([a.elapsed_time(b) for a, b in events]))
            return us, (f"event-record nodes around the forward inside the step's graph; {steps} timed "
                        f"steps, the last replay of each of the {ROTATION} buffer sets' graphs")
        split = []
        for i in range(ROTATION):
            pre, dom, post = segments(i)
            split.append((capture(pre) if pre else None, capture([dom]), capture(post) if post else None))
        evs = []
        for i in range(warmup + steps):
            pre, dom, post = split[i % ROTATION]
            if pre is not None:
                pre.replay()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            dom.replay()
            b.record(stream)
            if post is not None:
                post.replay()
            if i >= warmup:
                evs.append((a, b))
        torch.cuda.synchronize()
    us = 1e3 * float(np.mean([a.elapsed_time(b) for a, b in evs]))
    return us, f"events between graph launches around the forward; {steps} timed steps"


def capture_steps_with_events(segments, events, stream):
    """One CUDA graph per buffer set holding the whole step, with an event-record node
    (CU_EVENT_RECORD_EXTERNAL) on each side of the dominant layer's forward, so that
    CUDA events on the launching stream bracket that kernel in every replay without
    splitting the step into several graphs.  None if the driver refuses the nodes."""
    record = _cu_event_record_external()
    if record is None:
        return None
    for a, b in events:          # torch creates the CUDA events on first use
        a.record(stream)
        b.record(stream)
    torch.cuda.synchronize()
    graphs = []
    try:
        for i, (a, b) in enumerate(events):
            pre, dom, post = segments(i)
            g = torch.cuda.CUDAGraph()
            rc = 0
            with torch.cuda.graph(g, stream=stream):
                for f in pre:
                    f(None)
                rc |= record(a.cuda_event, stream.cuda_stream, 1)
                dom(None)
                rc |= record(b.cuda_event, stream.cuda_stream, 1)
                for f in post:
                    f(None)
            if rc != 0:
                return None
            graphs.append(g)
    except RuntimeError:
        torch.cuda.synchronize()
        return None
    return graphs


def layer_times_back_to_back(capi, sets, inputs, layers, stream, dev, replays) -> dict:
    """Steady-state time per call of each layer: one CUDA graph of G forwards of the layer
    back to back, each on its own buffer set, replayed; time per call = graph time / G.
    Consecutive forwards overlap their launch and prologue with the previous one's tail
    (programmatic dependent launch), as layers do inside a network.  G is chosen so that
    the sets rotate through more than 160 MB (more than the 129 MB L2); a layer too small
    for that within 64 sets is reported with "l2_resident": true."""
    out = {}
    for n in layers:
        sh = LAYERS[n]
        g_sets = max(ROTATION, -(-160_000_000 // sh.compulsory_bytes))
        resident = g_sets > 64
        g_sets = min(g_sets, 64)
        bufs = [sets[i][n] for i in range(ROTATION)] + \
               [LayerBuffers(inputs[n], dev) for _ in range(g_sets - ROTATION)]
        with torch.cuda.stream(stream):
            for lb in bufs[ROTATION:]:
                capi.fold(lb.g, lb.b, lb.m, lb.v, lb.eps, scale=lb.scale, bias=lb.bias, stream=stream)
                capi.forward(lb.x, lb.w, lb.scale, lb.bias, sh.stride, sh.pad, y=lb.y, stream=stream)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for lb in bufs:
                capi.forward(lb.x, lb.w, lb.scale, lb.bias, sh.stride, sh.pad, y=lb.y)
        with torch.cuda.stream(stream):
            for _ in range(3):
                g.replay()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(replays):
                g.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        capi.check(stream)
        out[n] = {"us": 1e3 * e0.elapsed_time(e1) / (replays * g_sets), "calls_per_graph": g_sets,
                  "rotation_mb": round(g_sets * sh.compulsory_bytes / 1e6, 1), "l2_resident": resident}
        del g, bufs
    return out


def gemm_context(dev, layers, fused_us, iters) -> dict:
    """Context, not part of the step: cuBLAS (torch.matmul, bf16) on a plain GEMM of the
    same M, N and K as a layer -- the pointwise layer is exactly that GEMM plus the
    epilogue; for a 3x3 layer the GEMM skips the implicit im2col.  Timed like the
    per-layer forwards (L2 flushed before each call, median)."""
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
    out = {}
    for n in ("pointwise", "deep"):
        if n not in layers:
            continue
        sh = LAYERS[n]
        m, k, c = sh.m, sh.k, sh.c * sh.r * sh.s
        a = torch.randn(m, c, device=dev).to(torch.bfloat16)
        b = torch.randn(c, k, device=dev).to(torch.bfloat16)
        for _ in range(3):
            a @ b
        evs = []
        for _ in range(iters):
            flush.zero_()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            a @ b
            e1.record()
            evs.append((e0, e1))
        torch.cuda.synchronize()
        us = 1e3 * statistics.median(x.elapsed_time(y) for x, y in evs)
        out[n] = {"gemm": f"{m}x{k}x{c} (M x N x K)", "cublas_us": round(us, 3),
                  "cublas_tflops": round(2 * m * k * c / us / 1e6, 1),
                  "fused_conv_us": round(fused_us[n], 3),
                  "fused_over_cublas": round(fused_us[n] / us, 3)}
        del a, b
    del flush
    return {"layers": out, "note": "cuBLAS on the same-size plain GEMM without BN/SiLU; context only"}


def isolated_layer_times(capi, sets, layers, stream, dev, iters, clean=False) -> dict:
    """Median forward time of each layer alone: the L2 is flushed (a 512 MB write) before
    every call and CUDA events on the stream bracket the forward kernel only.

    clean=True: the write is followed by a read of another 512 MB buffer, so that the
    flush's own dirty lines are written back before the call instead of during it (the L2
    the call starts with then holds only clean lines of an unrelated buffer)."""
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
    flush_r = torch.ones(128 * 1024 * 1024, dtype=torch.float32, device=dev) if clean else None
    out = {}
    with torch.cuda.stream(stream):
        for n in layers:
            evs = []
            for i in range(iters):
                lb = sets[i % ROTATION][n]
                sh = lb.shape
                flush.zero_()
                if clean:
                    flush_r.sum()
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                a.record(stream)
                capi.forward(lb.x, lb.w, lb.scale, lb.bias, sh.stride, sh.pad, y=lb.y, stream=stream)
                b.record(stream)
                evs.append((a, b))
            torch.cuda.synchronize()
            out[n] = 1e3 * statistics.median(a.elapsed_time(b) for a, b in evs)
    del flush, flush_r
    return out


def fusion_comparison(capi, sets, layers, stream, dev, iters, fused_us) -> dict:
    """The fused forward against the three-kernel sequence it replaces (conv -> t1,
    BN -> t2, SiLU -> y), each layer timed alone like the fused one: L2 flushed
    before every call, CUDA events around the whole sequence.  The unfused
    sequence moves four extra copies of the output through HBM (t1 written and
    read, t2 written and read)."""
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
    out = {}
    with torch.cuda.stream(stream):
        for n in layers:
            sh = LAYERS[n]
            t1 = torch.empty((sh.n, sh.ho, sh.wo, sh.k), dtype=torch.bfloat16, device=dev)
            t2 = torch.empty_like(t1)
            evs = []
            for i in range(iters):
                lb = sets[i % ROTATION][n]
                flush.zero_()
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                a.record(stream)
                capi.forward_unfused(lb.x, lb.w, lb.scale, lb.bias, sh.stride, sh.pad, y=lb.y,
                                     t1=t1, t2=t2, stream=stream)
                b.record(stream)
                evs.append((a, b))
            torch.cuda.synchronize()
            capi.check(stream)
            un_us = 1e3 * statistics.median(a.elapsed_time(b) for a, b in evs)
            y_bytes = 2 * sh.m * sh.k
            out[n] = {"fused_us": round(fused_us[n], 3), "unfused_us": round(un_us, 3),
                      "speedup": round(un_us / fused_us[n], 3),
                      "hbm_bytes_fused": sh.compulsory_bytes,
                      "hbm_bytes_unfused": sh.compulsory_bytes + 4 * y_bytes}
            del t1, t2
    del flush
    tot_f = sum(v["fused_us"] for v in out.values())
    tot_u = sum(v["unfused_us"] for v in out.values())
    return {"layers": out, "fused_us_total": round(tot_f, 3), "unfused_us_total": round(tot_u, 3),
            "speedup_total": round(tot_u / tot_f, 3),
            "timing": "median of isolated calls, L2 flushed before each; unfused = 3 launches"}


def epilogue_variants(capi, sets, layers, stream, dev, iters, silu_us) -> dict:
    """Each layer timed alone (L2 flushed before every call) with the other epilogues of
    conv_bn_act_forward: BN only, BN + ReLU, BN + SiLU + a residual add (which reads a second
    output-sized tensor) and BN + SiLU with an fp8 e4m3 output (conv_bn_act_forward_fp8), next
    to the fused SiLU layer itself."""
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
    out = {}
    with torch.cuda.stream(stream):
        for n in layers:
            sh = LAYERS[n]
            res = torch.randn((sh.n, sh.ho, sh.wo, sh.k), device=dev).to(torch.bfloat16)
            row = {"silu_us": round(silu_us[n], 3)}
            y8 = torch.empty((sh.n, sh.ho, sh.wo, sh.k), dtype=torch.uint8, device=dev)
            for label, act, r in (("identity_us", "identity", None), ("relu_us", "relu", None),
                                  ("silu_residual_us", "silu", res), ("silu_fp8_out_us", "silu", "fp8")):
                evs = []
                for i in range(iters):
                    lb = sets[i % ROTATION][n]
                    flush.zero_()
                    a = torch.cuda.Event(enable_timing=True)
                    b = torch.cuda.Event(enable_timing=True)
                    a.record(stream)
                    if isinstance(r, str):
                        capi.forward_act_fp8(lb.x, lb.w, lb.scale, lb.bias, sh.stride, sh.pad, activation=act,
                                             y=y8, stream=stream)
                    else:
                        capi.forward_act(lb.x, lb.w, lb.scale, lb.bias, sh.stride, sh.pad, activation=act,
                                         residual=r, y=lb.y, stream=stream)
                    b.record(stream)
                    evs.append((a, b))
                torch.cuda.synchronize()
                capi.check(stream)
                row[label] = round(1e3 * statistics.median(a.elapsed_time(b) for a, b in evs), 3)
            out[n] = row
            del res, y8
    del flush
    return {"layers": out, "timing": "median of isolated calls, L2 flushed before each",
            "residual_bytes_note": "the residual add reads one more bf16 tensor the size of y"}


def run_e2e(args, capi, inputs, dev, stream, world):
    """Same metric through the public API with host buffers: per step, every layer's x goes
    host->device from pinned memory, the batched fold and the fused forwards run, and y comes
    back device->host into pinned memory.  Weights and BN statistics stay resident on the device.

    The copies run on their own streams (one per direction) so that layer i+1's upload and
    layer i-1's download overlap layer i's forward; events order each buffer's upload, forward
    and download, across steps too (a step's upload of x waits for the previous step's forward
    on that buffer, a forward waits for the previous download of its y).  The serial form (all
    on one stream) is reported beside it."""
    layers = args.layers
    host_x = {n: bits_to_torch_bf16(inputs[n].x_bits).pin_memory() for n in layers}
    bufs = {n: LayerBuffers(inputs[n], dev) for n in layers}
    host_y = {n: torch.empty(bufs[n].y.shape, dtype=torch.bfloat16).pin_memory() for n in layers}
    h2d = sum(t.numel() * 2 for t in host_x.values())
    d2h = sum(t.numel() * 2 for t in host_y.values())
    flops_step = sum(LAYERS[n].flops for n in layers)
    fold = capi.FoldBatch([(b.g, b.b, b.m, b.v, b.eps, b.scale, b.bias) for b in (bufs[n] for n in layers)])
    s_in = torch.cuda.Stream(dev)
    s_out = torch.cuda.Stream(dev)
    uploaded = {n: torch.cuda.Event() for n in layers}
    computed = {n: torch.cuda.Event() for n in layers}
    downloaded = {n: torch.cuda.Event() for n in layers}

    def forward(n):
        b = bufs[n]
        sh = b.shape
        capi.forward(b.x, b.w, b.scale, b.bias, sh.stride, sh.pad, y=b.y, stream=stream)

    def step_serial():
        with torch.cuda.stream(stream):
            fold(stream)
            for n in layers:
                bufs[n].x.copy_(host_x[n], non_blocking=True)
                forward(n)
                host_y[n].copy_(bufs[n].y, non_blocking=True)

    def step_pipelined():
        for n in layers:
            s_in.wait_event(computed[n])          # the previous step's forward has read x
            with torch.cuda.stream(s_in):
                bufs[n].x.copy_(host_x[n], non_blocking=True)
            uploaded[n].record(s_in)
        with torch.cuda.stream(stream):
            fold(stream)
            for n in layers:
                stream.wait_event(uploaded[n])
                stream.wait_event(downloaded[n])  # the previous step's download of y is done
                forward(n)
                computed[n].record(stream)
        for n in layers:
            s_out.wait_event(computed[n])
            with torch.cuda.stream(s_out):
                host_y[n].copy_(bufs[n].y, non_blocking=True)
            downloaded[n].record(s_out)

    def timed(step):
        for _ in range(3):
            step()
        torch.cuda.synchronize()
        s = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize()
        s.record(stream)
        s_in.wait_event(s)
        for _ in range(args.e2e_steps):
            step()
        for st in (s_in, s_out):                   # join every stream before the end event
            ev = torch.cuda.Event()
            ev.record(st)
            stream.wait_event(ev)
        e.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        return max_over_ranks(s.elapsed_time(e) / 1e3, world, dev)

    t_serial = timed(step_serial)
    t = timed(step_pipelined)
    # The last step's results are in host memory: check one layer against the device copy.
    last = layers[-1]
    assert torch.equal(host_y[last], bufs[last].y.cpu()), "e2e: downloaded y differs from the device's"
    return {"value": round(aggregate_throughput(flops_step * args.e2e_steps, world, t) / 1e12, 3),
            "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": round(t / args.e2e_steps * 1e3, 4), "steps": args.e2e_steps,
            "serial_value": round(aggregate_throughput(flops_step * args.e2e_steps, world, t_serial) / 1e12, 3),
            "serial_ms_per_step": round(t_serial / args.e2e_steps * 1e3, 4),
            "api": "conv2d_batchnorm_silu_gb300.capi.FoldBatch/forward on the C ABI, pinned host buffers; "
                   "uploads and downloads on their own streams, overlapping the forwards"}


# ------------------------------------------------------------------ the oracle (CPU) legs
def oracle_sample_step(pixels_per_layer: dict, inputs) -> int:
    """One oracle pass over a sample of output pixels of every layer; returns its flops."""
    import oracle
    flops = 0
    for n in pixels_per_layer:
        inp = inputs[n]
        sh = inp.shape
        pix = pixels_per_layer[n]
        oracle.conv_bn_silu_at(inp.x_bits, inp.w_bits, inp.gamma, inp.beta, inp.mean, inp.var,
                               inp.eps, pix, sh.stride, sh.pad)
        flops += 2 * pix.size * sh.k * sh.kdim
    return flops


def sample_pixels(fraction: float, inputs, seed: int = 0) -> dict:
    """The same fraction of every layer's output pixels (at least one), chosen evenly."""
    out = {}
    for n in inputs:
        m = inputs[n].shape.m
        cnt = max(1, int(round(m * fraction)))
        out[n] = np.linspace(0, m - 1, cnt).astype(np.int64)
    return out


def cpu_model() -> str:
    """The host CPU's model name: lscpu's "Model name" (Arm hosts have no "model name" line in
    /proc/cpuinfo), else /proc/cpuinfo's, else its implementer/part codes."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        names = [ln.split(":", 1)[1].strip() for ln in out.splitlines() if ln.startswith("Model name:")]
        vendor = [ln.split(":", 1)[1].strip() for ln in out.splitlines() if ln.startswith("Vendor ID:")]
        if names:
            return " ".join(vendor[:1] + names[:1])
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        fields = {}
        with open("/proc/cpuinfo") as f:
            for ln in f:
                if ":" in ln:
                    k, v = ln.split(":", 1)
                    fields.setdefault(k.strip(), v.strip())
        if "model name" in fields:
            return fields["model name"]
        return f"CPU implementer {fields.get('CPU implementer', '?')} part {fields.get('CPU part', '?')}"
    except OSError:
        return "unknown"


def cpu_baseline(seconds: float, layers=LAYER_ORDER) -> dict:
    """The oracle as it stands, on this host's cores, over a bounded sample of the workload.

    The sample is the same fraction of every layer's output pixels; the fraction grows
    until one pass takes about `seconds` (each pass also decodes the layer's whole input,
    so the time is not proportional to the fraction)."""
    import oracle
    inputs = {n: make_layer_inputs(LAYERS[n]) for n in layers}
    frac = 1e-4
    while True:
        pix = sample_pixels(frac, inputs)
        t0 = time.perf_counter()
        flops = oracle_sample_step(pix, inputs)
        dt = time.perf_counter() - t0
        if dt >= seconds / 2 or frac >= 1.0:
            break
        frac = min(1.0, frac * max(2.0, min(8.0, seconds / max(dt, 1e-3) / 2)))
    return {"value": round(flops / dt / 1e12, 6), "unit": UNIT, "cores": oracle.default_threads(),
            "kind": "oracle", "cpu_model": cpu_model(),
            "sample": f"{frac:.3g} of every layer's output pixels (evenly spaced, all channels), "
                      f"{sum(p.size for p in pix.values())} pixels, {flops / 1e9:.2f} GFLOP in {dt:.1f} s"}


def run_reference(args, rank, world):
    """The reference arm: the fp64 CPU oracle, timed on the host cores, per step a sample."""
    if rank != 0:
        return
    import oracle
    oracle.build()
    inputs = {n: make_layer_inputs(LAYERS[n]) for n in args.layers}
    total_steps = max(1, args.steps + args.warmup)
    target_step_s = max(1e-3, args.reference_budget_seconds / total_steps)
    frac = 1e-5
    t0 = time.perf_counter()
    oracle_sample_step(sample_pixels(frac, inputs), inputs)
    dt = time.perf_counter() - t0
    frac = min(1.0, frac * max(1.0, target_step_s / max(dt, 1e-4)))
    pix = sample_pixels(frac, inputs)
    for _ in range(args.warmup):
        oracle_sample_step(pix, inputs)
    t0 = time.perf_counter()
    flops = 0
    for _ in range(args.steps):
        flops += oracle_sample_step(pix, inputs)
    dt = time.perf_counter() - t0
    value = flops / dt / 1e12
    sample = (f"per step {frac:.3g} of every layer's output pixels "
              f"({sum(p.size for p in pix.values())} pixels, all channels)")
    line = {
        "metric": METRIC, "value": round(value, 6), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (same seeded inputs as the GPU arm)",
        "config": {"workload": WORKLOAD, "l2": "n/a (CPU)", "parallelism": "host threads"},
        "impl": "reference",
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": oracle.default_threads(),
                         "kind": "oracle", "cpu_model": cpu_model(), "sample": sample},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    args = parse_args(argv)
    rank, world, local_rank = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    run_ours(args, rank, world, local_rank)
    if world > 1 and torch.distributed.is_initialized():
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
