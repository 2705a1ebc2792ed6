#!/usr/bin/env python3
"""Benchmark of the fused MoE layer (forward + backward) on GB300.

One step = mm_moe_forward + mm_moe_backward of the 16,384-token Qwen3-30B-A3B
shaped layer (T=16384, H=2048, I=768, E=128, top-8, Zipf(1.2) routing), bf16
with fp32 accumulation.  `value` is the whole job's algorithmic TFLOP/s
(fwd 6*R*H*I + bwd 12*R*H*I, R = T*k, padding not counted) with inputs resident
in HBM; `e2e` is the same metric through the public API with the step's
activations copied from pinned host memory and the results copied back.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

For N > 1 run under torch.distributed.run: one independent layer replica per
GPU (the path has no exchange step), barrier + max-over-ranks timing.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MoE layer fwd/bwd ms & TFLOP/s (30B-shape, 16k tok) as % of GB300 tensor peak"
DEFAULT_CONFIG = "qwen3_30b_16k_zipf"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
GEMM_FLOP_FACTOR = {  # algorithmic FLOPs per launch, in units of R*H*I
    "gemm_gateup_swiglu": 4, "gemm_down_weighted": 2, "gemm_dgrad_down_dswiglu": 2,
    "gemm_dgrad_gateup": 4, "gemm_wgrad_down": 2, "gemm_wgrad_gateup": 4,
    "gemm_wgrad": 6}  # the last: both weight gradients in one launch
BWD_GEMMS = ("gemm_dgrad_down_dswiglu", "gemm_dgrad_gateup", "gemm_wgrad_down",
             "gemm_wgrad_gateup", "gemm_wgrad")
# the arithmetic each precision's GEMMs compute in
DTYPE = {"bf16": "bf16", "mxfp8": "mxfp8", "fp8_bwd": "bf16 fwd / mxfp8 bwd",
         "fp8_block": "fp8_block (e4m3, 128-block scales)"}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--config", default=DEFAULT_CONFIG)
    ap.add_argument("--cpu-sample-tokens", type=int, default=1024,
                    help="tokens of the workload the CPU oracle baseline runs on")
    ap.add_argument("--ref-sample-tokens", type=int, default=128,
                    help="tokens per step of the reference (oracle) arm")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--kernels", action="store_true", help="also print the per-kernel table")
    ap.add_argument("--graph", action="store_true",
                    help="also time the step recorded once in a CUDA graph and replayed")
    ap.add_argument("--recompute", action="store_true",
                    help="activation checkpointing: the backward re-runs the gate/up stage")
    ap.add_argument("--multicast", action="store_true",
                    help="bf16 grouped GEMMs on clusters of two SM pairs sharing A by TMA "
                         "multicast (MM_MOE_MULTICAST)")
    ap.add_argument("--with-router", action="store_true",
                    help="the step also runs the top-k router (forward before the layer, "
                         "backward after it); topk_idx/topk_w then come from the router")
    return ap.parse_args()


# ---------------------------------------------------------------- distributed plumbing
def dist_info():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world: int, backend: str):
    if world > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group(backend=backend)


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Largest value of all ranks (every rank gets it)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_value(flops_per_step: float, world: int, ms_per_step_max: float) -> float:
    """Whole-job TFLOP/s: the work of all ranks over the slowest rank's step time."""
    return world * flops_per_step / (ms_per_step_max * 1e-3) / 1e12


# ---------------------------------------------------------------- clocks
CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,"
                "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
                "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                "clocks_event_reasons.sw_power_cap")


class ClockSampler:
    def __init__(self, gpu_index: int):
        self.path = tempfile.mktemp(prefix="mm_moe_clocks_", suffix=".csv")
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={CLOCK_FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        with open(self.path) as fh:
            for line in fh:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    rows.append(dict(sm=float(parts[1]), smax=float(parts[2]), util=float(parts[4]),
                                     hw=parts[6], hwt=parts[7], swt=parts[8], swp=parts[9]))
                except ValueError:
                    continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        load = [r for r in rows if r["util"] >= 50] or rows
        reasons = set()
        for r in load:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("swp", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in load),
                "sm_max_mhz": max(r["smax"] for r in rows), "reasons": sorted(reasons),
                "samples_under_load": len(load)}


# ---------------------------------------------------------------- helpers
def peak_regime(clock, peaks):
    """Which measured bf16 peak matches the timed region: "burst" when the region's
    median SM clock under load held the maximum (within 3 %) with no power cap
    (the regime of the burst GEMM measurement), else "sustained" (the power-capped
    loop).  Returns (regime, reason)."""
    sm = clock.get("sm_mhz") if clock else None
    smax = (clock.get("sm_max_mhz") if clock else None) or peaks.get("sm_max_mhz")
    reasons = clock.get("reasons", []) if clock else []
    if sm is None or not smax:
        return "sustained", "no clock record"
    if "sw_power_cap" in reasons:
        return "sustained", f"power cap active, median {sm:.0f} MHz"
    if sm >= 0.97 * smax:
        return "burst", f"median {sm:.0f} of {smax:.0f} MHz, no power cap"
    return "sustained", f"median {sm:.0f} of {smax:.0f} MHz"


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as fh:
            d = json.load(fh)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# the files that make the GEMM kernels and their launch sequence: a recorded DRAM
# traffic figure of a GEMM holds while these are unchanged
GEMM_SOURCES = ("gemm.cuh", "gemm.cu", "ptx.cuh", "mx.cuh", "internal.h", "mm_moe.cu")


def source_digest(files=None) -> str:
    """sha1 prefix over the library sources (all of csrc/, or the named files)."""
    h = hashlib.sha1()
    csrc = os.path.join(ROOT, "mixture_experts_layer_16_gb300", "csrc")
    for fn in sorted(files if files is not None else os.listdir(csrc)):
        with open(os.path.join(csrc, fn), "rb") as fh:
            h.update(fn.encode())
            h.update(fh.read())
    return h.hexdigest()[:12]


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, if it was
    captured on this workload from the current sources; else None."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(p) as fh:
            d = json.load(fh)
    except (OSError, ValueError):
        return None
    ent = d.get(kernel)
    if not ent or ent.get("workload") != workload or \
            ent.get("sources") != source_digest(GEMM_SOURCES):
        return None
    return ent.get("dram_bytes_per_launch")


def config_json(cfg):
    routing = {"uniform": "uniform", "zipf": f"zipf(s={cfg.zipf_s})",
               "zipf_trunc": f"zipf(s={cfg.zipf_s}) over {cfg.zipf_ranks} experts"}[cfg.routing]
    return {"workload": cfg.name, "T": cfg.T, "H": cfg.H, "I": cfg.I, "E": cfg.E, "k": cfg.k,
            "routing": routing, "precision": cfg.prec,
            "l2": "inputs larger than L2 (expert weights %.2f GB bf16)" % (
                3 * cfg.E * cfg.H * cfg.I * 2 / 1e9),
            "parallelism": "replicas"}


def step_flops(cfg, with_router: bool) -> float:
    """Algorithmic FLOPs of one step: the layer (fwd 6RHI + bwd 12RHI), plus the
    router's three products (2TEH each) when it runs."""
    f = cfg.flops_fwd() + cfg.flops_bwd()
    return f + (6.0 * cfg.T * cfg.E * cfg.H if with_router else 0.0)


LAST_ORACLE_SPLIT = [0.0, 0.0]  # seconds of the last oracle_step's forward and backward


def oracle_step(d, tokens: int, prec: str = "bf16"):
    """One oracle forward+backward on the first `tokens` tokens; returns (seconds, flops)."""
    import oracle
    import oracle.moe as om
    sub = om.token_subset(d, range(tokens))
    t0 = time.perf_counter()
    f = oracle.forward(sub["x"], sub["topk_idx"], sub["topk_w"], d["W_gate"], d["W_up"],
                       d["W_down"], prec)
    t1 = time.perf_counter()
    oracle.backward(sub["dy"], sub["x"], sub["topk_idx"], sub["topk_w"], d["W_gate"], d["W_up"],
                    d["W_down"], prec, fwd=f)
    dt = time.perf_counter() - t0
    LAST_ORACLE_SPLIT[:] = [t1 - t0, dt - (t1 - t0)]
    k = d["topk_idx"].shape[1]
    H = d["x"].shape[1]
    I = d["W_gate"].shape[1]
    return dt, 18.0 * tokens * k * H * I


# ---------------------------------------------------------------- the reference arm
def run_reference(args):
    world, rank, _ = dist_info()
    if rank != 0:
        return 0
    from mixture_experts_layer_16_gb300.inputs import CONFIGS, make_inputs
    cfg = CONFIGS[args.config]
    d = make_inputs(cfg)
    n = min(args.ref_sample_tokens, cfg.T)
    for _ in range(args.warmup):
        oracle_step(d, n, cfg.prec)
    times = []
    flops = 0.0
    for _ in range(args.steps):
        dt, flops = oracle_step(d, n, cfg.prec)
        times.append(dt)
    total = sum(times)
    value = flops * args.steps / total / 1e12
    cores = os.cpu_count()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": config_json(cfg),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": f"first {n} of {cfg.T} tokens per step (all {cfg.k} routed "
                                   f"rows each, full expert weights), numpy fp64"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- our arm
def run_ours(args):
    import numpy as np
    import torch

    world, rank, local = dist_info()
    torch.cuda.set_device(local)      # each rank's GPU before its NCCL group forms
    init_dist(world, "nccl")
    dev = torch.device("cuda", local)

    from mixture_experts_layer_16_gb300 import binding as B
    from mixture_experts_layer_16_gb300 import build as build_mod
    if rank == 0:
        build_mod.build()
    barrier(world)
    from mixture_experts_layer_16_gb300 import MoELayer
    from mixture_experts_layer_16_gb300.inputs import CONFIGS, make_inputs

    cfg = CONFIGS[args.config]
    d = make_inputs(cfg)

    def bf(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)

    host = {k: bf(d[k + "_bits"]) for k in ("x", "W_gate", "W_up", "W_down", "dy")}
    host["topk_idx"] = torch.from_numpy(d["topk_idx"])
    host["topk_w"] = torch.from_numpy(d["topk_w"])
    g = {k: v.to(dev) for k, v in host.items()}
    layer = MoELayer(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, cfg.prec, device=dev,
                     recompute=args.recompute, multicast=args.multicast)
    outs = (torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16, device=dev),
            torch.empty((cfg.E, cfg.I, cfg.H), dtype=torch.bfloat16, device=dev),
            torch.empty((cfg.E, cfg.I, cfg.H), dtype=torch.bfloat16, device=dev),
            torch.empty((cfg.E, cfg.H, cfg.I), dtype=torch.bfloat16, device=dev),
            torch.empty((cfg.T, cfg.k), dtype=torch.float32, device=dev))
    y = torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)
    router = None
    if args.with_router:
        from mixture_experts_layer_16_gb300 import MoERouter
        from mixture_experts_layer_16_gb300.inputs import router_weights
        router = MoERouter(cfg.T, cfg.H, cfg.E, cfg.k, device=dev)
        g["W_router"] = bf(router_weights(cfg.E, cfg.H, seed=cfg.seed)["W_router_bits"]).to(dev)
        dW_router = torch.empty_like(g["W_router"])
    rev = []  # ("fwd" | "bwd", start, end) events around the router calls

    def ev_t():
        e = torch.cuda.Event(enable_timing=True)
        e.record(stream)
        return e

    def step(x, idx, w, dy, y_out, out, after_fwd=None, timed=False):
        """One step through the public API (with the router, it chooses idx and w).
        Returns (event between forward and backward, forward launches, backward launches)."""
        if router is not None:
            e0 = ev_t() if timed else None
            idx, w = router.forward(x, g["W_router"])
            if timed:
                rev.append(("fwd", e0, ev_t()))
        layer.forward(x, idx, w, g["W_gate"], g["W_up"], g["W_down"], y=y_out)
        n_f = B.mm_moe_last_launch_count()
        mid = ev_t() if timed else None
        if after_fwd is not None:
            after_fwd()
        layer.backward(dy, g["W_gate"], g["W_up"], g["W_down"], out=out, x=x)
        n_b = B.mm_moe_last_launch_count()
        if router is not None:
            e2 = ev_t() if timed else None
            router.backward(x, g["W_router"], idx, w, out[4], out[0], dW_router)
            if timed:
                rev.append(("bwd", e2, ev_t()))
        return mid, n_f, n_b

    for _ in range(max(args.warmup, 0)):
        step(g["x"], g["topk_idx"], g["topk_w"], g["dy"], y, outs)
    torch.cuda.synchronize()
    if layer.status() != B.MM_MOE_OK:
        raise RuntimeError("device status after warm-up: " + B.STATUS[layer.status()])
    n_fwd_launch = n_bwd_launch = 0

    # ------------------------------------------------ timed region (device-resident inputs)
    K = args.steps
    marks = []
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        barrier(world)
        torch.cuda.synchronize()
        B.mm_moe_profile_start()
        start.record(stream)
        for i in range(K):
            e0 = ev_t()
            mid, n_fwd_launch, n_bwd_launch = step(g["x"], g["topk_idx"], g["topk_w"], g["dy"],
                                                   y, outs, timed=True)
            marks.append((e0, mid, ev_t()))
        stop.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        prof = B.mm_moe_profile_stop()
    clock = clocks.summary()
    ms_step = start.elapsed_time(stop) / K
    ms_step_max = max_over_ranks(ms_step, world, dev)
    fwd_ms = statistics.median(m[0].elapsed_time(m[1]) for m in marks)
    bwd_ms = statistics.median(m[1].elapsed_time(m[2]) for m in marks)
    router_ms = None
    if router is not None:
        router_ms = {kind: statistics.median(a.elapsed_time(b) for kk, a, b in rev if kk == kind)
                     for kind in ("fwd", "bwd")}
    st = layer.status()
    if st != B.MM_MOE_OK:
        raise RuntimeError("device status after timed region: " + B.STATUS[st])

    # ------------------------------------------------ e2e through host buffers
    # Every step copies its activations in from pinned host memory and its results
    # (y, dx, dtopk_w) back, as a training loop feeding the layer would.  The copies are
    # double-buffered and run on two more streams, one a direction, so that the host
    # link carries both at once: step i+1's inputs arrive while step i computes, y leaves
    # during the backward, dx and dtopk_w during the next step.  A buffer is written
    # again only after the copy that read it is done.  With the router, topk_idx and
    # topk_w are made on the device and not copied.
    e2e = None
    if not args.no_e2e:
        names = ("x", "dy") if router is not None else ("x", "topk_idx", "topk_w", "dy")
        pin = {k: host[k].pin_memory() for k in names}
        out_h = (torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16).pin_memory(),
                 torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16).pin_memory(),
                 torch.empty((cfg.T, cfg.k), dtype=torch.float32).pin_memory())
        act = [{k: torch.empty_like(g[k]) for k in pin} for _ in range(2)]
        ys = [torch.empty_like(y) for _ in range(2)]
        dxs = [torch.empty_like(outs[0]) for _ in range(2)]
        dtws = [torch.empty_like(outs[4]) for _ in range(2)]
        h2d = sum(t.numel() * t.element_size() for t in pin.values())
        d2h = sum(t.numel() * t.element_size() for t in out_h)
        cin, cout = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

        def ev():
            return torch.cuda.Event()

        def e2e_run(n_steps, start_ev=None):
            h2d_done, fwd_done, step_done, out_done = ([ev(), ev()] for _ in range(4))
            out_pending = [False, False]
            with torch.cuda.stream(cin):
                if start_ev is not None:
                    cin.wait_event(start_ev)
                for k2, t in pin.items():
                    act[0][k2].copy_(t, non_blocking=True)
                h2d_done[0].record(cin)
            if start_ev is not None:
                cout.wait_event(start_ev)
            for i in range(n_steps):
                b = i % 2
                stream.wait_event(h2d_done[b])
                if out_pending[b]:           # step i-2's results have left buffer b
                    stream.wait_event(out_done[b])
                if i + 1 < n_steps:          # prefetch the next step's activations
                    with torch.cuda.stream(cin):
                        if i >= 1:           # the step that last read buffer 1-b is done
                            cin.wait_event(step_done[1 - b])
                        for k2, t in pin.items():
                            act[1 - b][k2].copy_(t, non_blocking=True)
                        h2d_done[1 - b].record(cin)
                a = act[b]

                def y_out(b=b):
                    fwd_done[b].record(stream)
                    with torch.cuda.stream(cout):
                        cout.wait_event(fwd_done[b])
                        out_h[0].copy_(ys[b], non_blocking=True)
                step(a["x"], a.get("topk_idx"), a.get("topk_w"), a["dy"], ys[b],
                     (dxs[b], outs[1], outs[2], outs[3], dtws[b]), after_fwd=y_out)
                step_done[b].record(stream)
                with torch.cuda.stream(cout):
                    cout.wait_event(step_done[b])
                    out_h[1].copy_(dxs[b], non_blocking=True)
                    out_h[2].copy_(dtws[b], non_blocking=True)
                    out_done[b].record(cout)
                out_pending[b] = True
            done_in, done_out = ev(), ev()
            done_in.record(cin)
            done_out.record(cout)
            stream.wait_event(done_in)
            stream.wait_event(done_out)      # the last results are on the host

        e2e_run(max(args.warmup, 1))
        torch.cuda.synchronize()
        barrier(world)
        s2, t2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s2.record(stream)
        e2e_run(K, start_ev=s2)
        t2.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        e2e_ms = max_over_ranks(s2.elapsed_time(t2) / K, world, dev)
        e2e = {"value": aggregate_value(step_flops(cfg, router is not None), world, e2e_ms),
               "unit": "TFLOP/s", "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h,
               "note": "activations (" + ", ".join(names) + ") in from pinned host memory "
                       "and y, dx, dtopk_w out, every step; copies double-buffered on two "
                       "more streams, one a direction (the next step's inputs arrive "
                       "during this step); "
                       "weights and weight gradients stay on the device"}

    # ------------------------------------------------ the same step as one CUDA graph
    # (reported beside the eager number, which stays the line's value): the layer's
    # forward and backward recorded once on device-resident inputs, then replayed
    graph = None
    if args.graph and router is None:
        cs = torch.cuda.Stream(dev)
        cs.wait_stream(stream)
        with torch.cuda.stream(cs):     # one eager step on the capture stream first
            step(g["x"], g["topk_idx"], g["topk_w"], g["dy"], y, outs)
        stream.wait_stream(cs)
        torch.cuda.synchronize()
        cg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(cg):
            step(g["x"], g["topk_idx"], g["topk_w"], g["dy"], y, outs)
        for _ in range(max(args.warmup, 3)):
            cg.replay()
        torch.cuda.synchronize()
        barrier(world)
        s3, t3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s3.record(stream)
        for _ in range(K):
            cg.replay()
        t3.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        g_ms = max_over_ranks(s3.elapsed_time(t3) / K, world, dev)
        if layer.status() != B.MM_MOE_OK:
            raise RuntimeError("device status after the graph replays: " + B.STATUS[layer.status()])
        graph = {"value": aggregate_value(step_flops(cfg, False), world, g_ms), "unit": "TFLOP/s",
                 "ms_per_step": g_ms,
                 "note": "forward + backward recorded once in a CUDA graph, replayed K times"}

    if rank != 0:
        return 0

    # ------------------------------------------------ roofline of the dominant kernel
    peaks, peak_src = load_peaks()
    RHI = float(cfg.R) * cfg.H * cfg.I
    kern = {name: {"avg_ms": ms / n, "launches_per_step": n / K, "share": 0.0}
            for name, (ms, n) in prof.items() if n > 0}
    tot = sum(v["avg_ms"] * v["launches_per_step"] for v in kern.values())
    for v in kern.values():
        v["share"] = v["avg_ms"] * v["launches_per_step"] / tot if tot else 0.0
    gemms = {k: v for k, v in kern.items() if k in GEMM_FLOP_FACTOR}
    dom = max(gemms, key=lambda k: gemms[k]["avg_ms"] * gemms[k]["launches_per_step"])
    for k, v in gemms.items():
        v["tflops"] = GEMM_FLOP_FACTOR[k] * RHI / (v["avg_ms"] * 1e-3) / 1e12
    regime, regime_why = peak_regime(clock, peaks)
    pkey = "bf16_tflops" if regime == "burst" else "bf16_tflops_sustained"
    bpeak = peaks.get(pkey, FALLBACK_PEAKS[pkey])
    # a contraction takes the peak of its own dtype: FP8 = the bf16 peak x 2 (nominal
    # 4.5 / 2.25 PFLOP/s)
    dom_fp8 = cfg.prec in ("mxfp8", "fp8_block") or (cfg.prec == "fp8_bwd" and dom in BWD_GEMMS)
    peak = bpeak * (2.0 if dom_fp8 else 1.0)
    achieved = gemms[dom]["tflops"]
    roof = {"kernel": dom, "bound": "tensor", "achieved": achieved, "peak": peak,
            "unit": "TFLOP/s", "frac": achieved / peak, "traffic": recorded_traffic(dom, cfg.name),
            "peak_source": f"{peak_src} {pkey}" + (" x 2 (FP8 = 2 x bf16, nominal ratio)"
                                                   if dom_fp8 else "") + f"; {regime_why}",
            "algorithmic_flops_per_launch": GEMM_FLOP_FACTOR[dom] * RHI}

    # ------------------------------------------------ CPU oracle baseline (rank 0, N=1)
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        n = min(args.cpu_sample_tokens, cfg.T)
        dt, fl = oracle_step(d, n, cfg.prec)
        cpu = {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": os.cpu_count(),
               "kind": "oracle", "seconds": dt, "fwd_seconds": LAST_ORACLE_SPLIT[0],
               "bwd_seconds": LAST_ORACLE_SPLIT[1],
               "sample": f"first {n} of {cfg.T} tokens (all {cfg.k} routed rows each, full "
                         f"expert weights), one forward+backward, numpy fp64"}

    flops = step_flops(cfg, router is not None)
    value = aggregate_value(flops, world, ms_step_max)
    # The path's fraction of the dense tensor peak of its precision, against the
    # measured bf16 peak of the clock regime the timed region ran in (burst: the
    # region held the maximum SM clock with no power cap; else sustained).  FP8 peak =
    # that bf16 peak x 2 (nominal 4.5 / 2.25 PFLOP/s); fp8_bwd blends the two, total
    # FLOP / (fwd FLOP / P_bf16 + bwd FLOP / P_fp8).  Blockwise FP8 runs on the same
    # block-scaled FP8 tensor cores as MXFP8 (its 128-block scales repeated over the
    # 32-element scale blocks), so its peak is the FP8 one throughout.
    r_f = 2.0 * cfg.T * cfg.E * cfg.H if router is not None else 0.0  # router products
    f_fwd, f_bwd = cfg.flops_fwd() + r_f, cfg.flops_bwd() + 2.0 * r_f

    def fractions(bp):
        p_fwd = 2.0 * bp if cfg.prec in ("mxfp8", "fp8_block") else bp
        p_bwd = 2.0 * bp if cfg.prec in ("mxfp8", "fp8_bwd", "fp8_block") else bp
        p_tot = (f_fwd + f_bwd) / (f_fwd / p_fwd + f_bwd / p_bwd)
        return {"fwd": fwd_tf / p_fwd, "bwd": bwd_tf / p_bwd, "step": value / world / p_tot,
                "peak_fwd_tflops": p_fwd, "peak_bwd_tflops": p_bwd}

    fwd_tf = f_fwd / (fwd_ms * 1e-3) / 1e12
    bwd_tf = f_bwd / (bwd_ms * 1e-3) / 1e12
    peak_fractions = dict(fractions(bpeak), regime=regime,
                          note=f"bf16 peak = measured {pkey} ({regime_why}); FP8 peak = 2 x "
                               "that (nominal ratio)")
    other = "bf16_tflops_sustained" if regime == "burst" else "bf16_tflops"
    peak_fractions["other_regime"] = dict(
        fractions(peaks.get(other, FALLBACK_PEAKS[other])), peak_key=other)
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_step_max, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": DTYPE[cfg.prec], "data": "synthetic",
        "config": dict(config_json(cfg), recompute=bool(args.recompute),
                       multicast=bool(args.multicast), router=router is not None),
        "router_ms": router_ms,
        "fwd_ms": fwd_ms, "bwd_ms": bwd_ms,
        "fwd_tflops": fwd_tf,
        "bwd_tflops": bwd_tf,
        "frac_of_bf16_peak": value / world / bpeak,
        "frac_of_precision_peak": peak_fractions,
        "peak_note": f"{peak_src} {pkey} = {bpeak} ({regime_why})",
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "graph": graph,
        # this library's kernels: the layer's, and with the router its five (the logits
        # GEMM and the top-k selection; the logit gradient and the two GEMMs after it)
        "gpu_launches": (n_fwd_launch + n_bwd_launch + (5 if router is not None else 0)) * K,
        "clocks": clock,
        "kernels": kern if args.kernels else {k: round(v["share"], 4) for k, v in kern.items()},
        "sources": source_digest(),
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
