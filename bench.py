#!/usr/bin/env python
"""Benchmark of the tiled-latent hot path on one GB300 (or N replicas).

One step is one pass of every step of the path on the 4K-class workload
(bf16 latent B=1, C=128, F=16, H=68, W=120; tiles 2x4x4 with overlaps
2/8/12; 256 conditioning tokens, 64 with a negative time start):
    tdp_extract, tdp_tokens (positions and conditioning selection in one
    launch, plus the per-token count), tdp_window_sum, tdp_blend, in order
    on one stream (the blend's persistent grid fills every SM, so the short
    token kernels gain nothing from a second stream).
The per-tile op between extract and blend is the caller's (here identity,
outside the path).  Inputs are resident in HBM when the timed region starts;
L2 is flushed (a 256 MiB write) before every step and before the blend,
outside the timed spans.

Headline: algorithmic extract+blend bytes per step / step time (GB/s):
    latent read + tile write (extract) + tile read + latent write (blend).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl tdp|reference]

Under torchrun every rank runs its own replica (the tiles of the method are
independent; there is no data-path collective) and rank 0 prints one JSON
line with the max-over-ranks step time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from overlap_add_blending_gb300 import inputs  # noqa: E402
from overlap_add_blending_gb300.workloads import WORKLOADS  # noqa: E402

WORKLOAD = WORKLOADS["4k"]
METRIC = "tile extract+blend HBM GB/s (fraction of GB300 peak) and latent elems/s"
FALLBACK_HBM_GBS = 6800.0
KERNELS_PER_STEP = 5  # extract, tokens (2: per-tile kernel, per-token count), window sum, blend


def esz(dtype: str) -> int:
    return 2 if dtype == "bf16" else 4


def algorithmic_bytes(wl, tiles_numel: int) -> dict:
    lat = wl.B * wl.C * wl.dims[0] * wl.dims[1] * wl.dims[2]
    e = esz(wl.dtype)
    extract = lat * e + tiles_numel * e
    blend = tiles_numel * e + lat * e
    return {"latent_elems": lat, "tile_elems": tiles_numel, "extract": extract, "blend": blend,
            "total": extract + blend, "overlap_factor": tiles_numel / lat}


def config_dict(wl, note: str) -> dict:
    return {"workload": f"4k-class latent {wl.dtype} B={wl.B} C={wl.C} F={wl.dims[0]} H={wl.dims[1]} "
                        f"W={wl.dims[2]}, tiles (frames {wl.tiling[0][0]}/{wl.tiling[0][1]}, height "
                        f"{wl.tiling[1][0]}/{wl.tiling[1][1]}, width {wl.tiling[2][0]}/{wl.tiling[2][1]}), "
                        f"{wl.num_cond} conditioning tokens ({wl.num_cond_negative} with negative time)",
            "step": "extract, with tokens (positions + cond select) and window_sum beside it on a side "
                    "stream, then blend; per-tile op: identity, outside",
            "l2": note}


def read_peak() -> tuple:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
        for k in ("hbm_gbs", "hbm_GBps", "hbm"):
            if k in d:
                v = d[k]
                if isinstance(v, dict):
                    v = v.get("value", v.get("gbs"))
                return float(v), "measured"
    except (OSError, ValueError, TypeError):
        pass
    return FALLBACK_HBM_GBS, "fallback"


# The sources the profiled kernels (extract, blend, tokens) are built from.
PROFILED_SOURCES = ("tdp_kernels.cu", "tdp_stream.cuh", "tdp_geometry.h")


def source_digest() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "overlap_add_blending_gb300", "csrc")
    for name in PROFILED_SOURCES:
        with open(os.path.join(csrc, name), "rb") as fh:
            h.update(name.encode() + b"\0" + fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources."""
    path = os.path.join(ROOT, "profiles", "dram_traffic_4k.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
    except (OSError, ValueError):
        return None
    if d.get("source_digest") != source_digest():
        return None
    k = d.get("kernels", {}).get(kernel)
    return None if k is None else k.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 100 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: str):
        self.lines = []
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", gpu_index], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- oracle timing
def oracle_step(wl, X, gen, cond, channels: int):
    """One step of the CPU oracle on the first `channels` channels."""
    from oracle import tdp_oracle as O
    plan = O.make_plan(wl.dims, wl.tiling)
    x = X[:, :channels]
    tiles = O.extract(plan, x)
    O.positions(plan, gen)
    O.cond_select(plan, gen, cond)
    y = O.blend(plan, tiles)
    O.max_abs_deviation(plan)
    return y


def oracle_inputs(wl, channels: int):
    import torch
    Xf = inputs.latent((wl.B, wl.C) + wl.dims, seed=0)[:, :channels]
    X = torch.from_numpy(np.ascontiguousarray(Xf)).to(torch.bfloat16).double().numpy()
    gen = inputs.grid_positions(wl.B, *wl.dims)
    cond = inputs.cond_positions(wl.B, wl.num_cond, *wl.dims, n_negative=wl.num_cond_negative, seed=2)
    return X, gen, cond


def sample_bytes(wl, channels: int) -> float:
    frac = channels / wl.C
    from oracle import tdp_oracle as O
    plan = O.make_plan(wl.dims, wl.tiling)
    tiles = sum(int(np.prod(plan.shape(t))) for t in range(plan.num_tiles)) * wl.B * wl.C
    return algorithmic_bytes(wl, tiles)["total"] * frac


def cpu_baseline(wl, budget_s: float = 10.0, channels: int = 16) -> dict:
    X, gen, cond = oracle_inputs(wl, channels)
    t0 = time.perf_counter()
    n = 0
    while True:
        oracle_step(wl, X, gen, cond, channels)
        n += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    return {"value": sample_bytes(wl, channels) * n / dt / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{n} oracle steps (extract, positions, cond select, blend, window sum; float64 NumPy, "
                      f"one thread) on {channels} of {wl.C} channels of the 4k-class workload, "
                      f"{dt:.1f} s; bytes scaled to the sample"}


def run_reference(args, rank: int, world: int):
    if rank != 0:
        return 0
    wl = WORKLOAD
    channels = 16
    X, gen, cond = oracle_inputs(wl, channels)
    for _ in range(args.warmup):
        oracle_step(wl, X, gen, cond, channels)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle_step(wl, X, gen, cond, channels)
        times.append(time.perf_counter() - t0)
    ms = 1e3 * sum(times) / len(times)
    value = sample_bytes(wl, channels) / (ms * 1e-3) / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_dict(wl, "n/a (CPU)"),
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": f"each step: oracle extract, positions, cond select, blend and window sum "
                                       f"on {channels} of {wl.C} channels (float64 NumPy, one thread); "
                                       f"bytes scaled to the sample"},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- GPU arm
def run_tdp(args, rank: int, world: int):
    import torch
    import torch.distributed as dist
    from overlap_add_blending_gb300 import tdp
    from overlap_add_blending_gb300.replicas import combine

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the tdp path has no CPU fallback)")
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wl = WORKLOAD
    dt = torch.bfloat16
    p = tdp.plan(wl.dims, wl.tiling)
    ab = algorithmic_bytes(wl, p.tiles_numel(wl.B, wl.C))

    # resident inputs and outputs
    X = torch.from_numpy(inputs.latent((wl.B, wl.C) + wl.dims, seed=0)).to(dt).to(dev)
    gen_np = inputs.grid_positions(wl.B, *wl.dims)
    cond_np = inputs.cond_positions(wl.B, wl.num_cond, *wl.dims, n_negative=wl.num_cond_negative, seed=2)
    gen = torch.from_numpy(gen_np).to(dev)
    cond = torch.from_numpy(cond_np).to(dev)
    tiles = torch.empty(p.tiles_numel(wl.B, wl.C), dtype=dt, device=dev)
    out = torch.empty_like(X)
    tok_out = {}
    maxdev = torch.empty(4, dtype=torch.float32, device=dev)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    side = torch.cuda.Stream(device=dev)
    fork, join = torch.cuda.Event(), torch.cuda.Event()

    # The token kernels and the window maximum do not read the latent or the
    # tiles: they run on a side stream beside extract (they feed the per-tile
    # model, not the blend's inputs), and the main stream waits for them
    # before the blend.
    def side_work(g=gen, c=cond, m=maxdev):
        fork.record(stream)
        side.wait_event(fork)
        tdp.tokens(p, g, c, True, True, tok_out, stream=side)
        tdp.window_sum(p, m, stream=side)
        join.record(side)

    def path(x=X, g=gen, c=cond, o=out, m=maxdev):
        side_work(g, c, m)
        tdp.extract(p, x, tiles)
        stream.wait_event(join)
        tdp.blend(p, tiles, wl.B, wl.C, o)

    # One step: extract with the token and window kernels beside it on the
    # side stream, then the blend.  Events on the main stream: ev0 start,
    # ev1 extract done, ev2 side work joined, ev3 / ev4 around the blend.  L2
    # is flushed before the step and again before the blend, outside the
    # timed spans: in use, the per-tile model runs between the two phases.
    def timed_step(ev):
        ev[0].record(stream)
        side_work()
        tdp.extract(p, X, tiles)
        ev[1].record(stream)
        stream.wait_event(join)
        ev[2].record(stream)
        flush.zero_()
        ev[3].record(stream)
        tdp.blend(p, tiles, wl.B, wl.C, out)
        ev[4].record(stream)

    # host enqueue time of one step, to size the head start given to the host
    path()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(3):
        path()
    enqueue_s = (time.perf_counter() - t0) / 3
    torch.cuda.synchronize()
    sleep_cycles = int(max(200e-6, 3 * enqueue_s) * 2.0e9)

    visible = os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")
    gpu_index = visible[local].strip() if len(visible) > local and visible[local].strip() else str(local)
    sampler = ClockSampler(gpu_index)

    for _ in range(args.warmup):
        flush.zero_()
        path()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()

    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(K)]
    wall0 = time.perf_counter()
    for k in range(K):
        flush.zero_()
        torch.cuda._sleep(sleep_cycles)      # the host enqueues the whole step meanwhile
        timed_step(evs[k])
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks = sampler.stop()

    # step = (extract beside tokens + window sum) + blend
    step = np.array([evs[k][0].elapsed_time(evs[k][2]) + evs[k][3].elapsed_time(evs[k][4]) for k in range(K)])
    seg = np.array([[evs[k][0].elapsed_time(evs[k][1]), evs[k][1].elapsed_time(evs[k][2]),
                     evs[k][3].elapsed_time(evs[k][4])] for k in range(K)])  # ms
    step_ms = float(step.mean())
    per_kernel_ms = seg.mean(axis=0)
    # extract: its own span (sharing the GPU with the side kernels); the
    # token kernels' cost is what they add after extract ends
    names = ["extract", "tokens_and_window_sum_after_extract", "blend"]

    # The next row after the step (not part of it): the conditioning-token
    # combine, on the step's selection, with D = C features per token.
    comb_in = torch.randn((p.T, wl.B, wl.num_cond, wl.C), device=dev).to(dt)
    comb_out = torch.empty((wl.B, wl.num_cond, wl.C), dtype=dt, device=dev)
    for _ in range(3):
        tdp.cond_combine(p, comb_in, tok_out["slot_of"], tok_out["weight"], out=comb_out)
    cev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(20)]
    torch.cuda._sleep(20 * sleep_cycles)   # the host enqueues all 20 launches meanwhile
    for e in cev:
        e[0].record(stream)
        tdp.cond_combine(p, comb_in, tok_out["slot_of"], tok_out["weight"], out=comb_out)
        e[1].record(stream)
    torch.cuda.synchronize()
    comb_ms = float(np.median([e[0].elapsed_time(e[1]) for e in cev]))

    # The next row after that: the token-major pair (tiles as [B, N_t, C] token
    # sequences), each launch timed alone after an L2 flush outside its events.
    tm_tiles = torch.empty_like(tiles)
    tm_out = torch.empty_like(X)

    def time_alone(fn, reps: int = 20) -> float:
        for _ in range(3):
            flush.zero_()
            fn()
        ev2 = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(reps)]
        for e in ev2:
            flush.zero_()
            e[0].record(stream)
            fn()
            e[1].record(stream)
        torch.cuda.synchronize()
        return float(np.median([e[0].elapsed_time(e[1]) for e in ev2]))

    tmx_ms = time_alone(lambda: tdp.extract_tokens(p, X, tm_tiles))
    tmb_ms = time_alone(lambda: tdp.blend_tokens(p, tm_tiles, wl.B, wl.C, tm_out))

    # The host planner (the last next row): the layout search for this
    # latent at 8 ranks, frame tiling and overlaps as in the workload.
    t0 = time.perf_counter()
    for _ in range(20):
        cands = tdp.search_layouts(wl.dims, 8, wl.tiling[0], wl.tiling[1][1], wl.tiling[2][1])
    search_us = (time.perf_counter() - t0) / 20 * 1e6
    picks = {c["role"]: list(c["counts"]) for c in cands if c["role"] in ("coarse", "fine", "balanced")}

    # e2e: host buffers in, blended latent out, through the same C-ABI calls.
    # Steps are pipelined over two device buffer sets: step k's inputs go up
    # on one copy stream while step k-1 computes, and step k-1's result comes
    # down on another while step k computes.  Timed from the first upload to
    # the last download, over K steps.
    X_h = X.cpu().pin_memory()
    gen_h = gen.cpu().pin_memory()
    cond_h = cond.cpu().pin_memory()
    out_h = [torch.empty(out.shape, dtype=dt, pin_memory=True) for _ in range(2)]
    dev_h = [torch.empty(1, dtype=torch.float32, pin_memory=True) for _ in range(2)]
    h2d = X_h.numel() * X_h.element_size() + gen_h.numel() * 4 + cond_h.numel() * 4
    d2h = out_h[0].numel() * out_h[0].element_size() + 4
    ref_out = out.cpu()
    bufs = [(X, gen, cond, out, maxdev),
            (torch.empty_like(X), torch.empty_like(gen), torch.empty_like(cond), torch.empty_like(out),
             torch.empty_like(maxdev))]
    up, down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    in_ready, in_free, out_ready, out_free = ([torch.cuda.Event() for _ in range(2)] for _ in range(4))
    for i in range(2):
        in_free[i].record(stream)
        out_free[i].record(stream)

    def e2e_step(k):
        i = k % 2
        x, g, c, o, m = bufs[i]
        up.wait_event(in_free[i])
        with torch.cuda.stream(up):
            x.copy_(X_h, non_blocking=True)
            g.copy_(gen_h, non_blocking=True)
            c.copy_(cond_h, non_blocking=True)
        in_ready[i].record(up)
        stream.wait_event(in_ready[i])
        stream.wait_event(out_free[i])
        path(x, g, c, o, m)
        in_free[i].record(stream)
        out_ready[i].record(stream)
        down.wait_event(out_ready[i])
        with torch.cuda.stream(down):
            out_h[i].copy_(o, non_blocking=True)
            dev_h[i].copy_(m[:1], non_blocking=True)
        out_free[i].record(down)

    for k in range(min(3, args.warmup)):
        e2e_step(k)
    torch.cuda.synchronize()
    t_first, t_last = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    up.wait_stream(stream)
    with torch.cuda.stream(up):
        torch.cuda._sleep(sleep_cycles)   # the host enqueues ahead meanwhile
    t_first.record(up)
    for k in range(K):
        e2e_step(k)
    down.wait_stream(stream)
    t_last.record(down)
    torch.cuda.synchronize()
    for i in range(2):
        if not torch.equal(out_h[i], ref_out):
            raise SystemExit("e2e: a downloaded result differs from the device-resident step's")
    e2e_ms = t_first.elapsed_time(t_last) / K


    # replicas: slowest rank's times, every rank's work
    mx, job_bytes = combine([step_ms, e2e_ms] + [float(v) for v in per_kernel_ms], ab["total"], device=dev)
    step_ms, e2e_ms, per_kernel_ms = mx[0], mx[1], np.array(mx[2:])

    if rank != 0:
        return 0
    peak, peak_src = read_peak()
    kern = {n: {"ms": float(per_kernel_ms[i])} for i, n in enumerate(names)}
    kern["extract"]["gbs"] = ab["extract"] / (kern["extract"]["ms"] * 1e-3) / 1e9
    kern["blend"]["gbs"] = ab["blend"] / (kern["blend"]["ms"] * 1e-3) / 1e9
    dom = "blend" if kern["blend"]["ms"] >= kern["extract"]["ms"] else "extract"
    achieved = kern[dom]["gbs"]
    traffic = recorded_traffic(dom)
    value = job_bytes / (step_ms * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": config_dict(wl, "flushed (256 MiB write, outside the events) before every step and again "
                                  "before the blend"),
        "latent_elems_per_s": world * ab["latent_elems"] / (step_ms * 1e-3),
        "extract_blend_gbs": ab["total"] / ((kern["extract"]["ms"] + kern["blend"]["ms"]) * 1e-3) / 1e9,
        "algorithmic_bytes": {"extract": ab["extract"], "blend": ab["blend"],
                              "overlap_factor": round(ab["overlap_factor"], 5)},
        "kernels": kern,
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic, "peak_source": peak_src},
        "e2e": {"value": job_bytes / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "ms_per_step": e2e_ms,
                "pipelined": "two buffer sets; uploads, steps and downloads on three streams; "
                             "first upload to last download over K steps"},
        "gpu_launches": KERNELS_PER_STEP * K,
        "next_rows": {"cond_combine": {"ms": comb_ms, "workload": f"T={p.T} tiles, B={wl.B}, M={wl.num_cond} "
                                       f"conditioning tokens, D={wl.C} bf16 features; median of 20, not in the step"},
                      "token_major": {
                          "extract_tokens": {"ms": tmx_ms, "gbs": ab["extract"] / (tmx_ms * 1e-3) / 1e9},
                          "blend_tokens": {"ms": tmb_ms, "gbs": ab["blend"] / (tmb_ms * 1e-3) / 1e9},
                          "workload": "the step's latent and tiles with each tile as [B, N_t, C] tokens; "
                                      "median of 20 launches, each after an L2 flush; not in the step"},
                      "layout_search": {"us": search_us, "ranks": 8, "candidates": len(cands), "picks": picks,
                                        "workload": "host layout search for this latent, frame tiling and "
                                                    "overlaps; mean of 20 calls"}},
        "clocks": clocks,
        "timed_wall_s": wall,
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl)
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)   # about 0.5 s timed: several clock samples
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["tdp", "reference"], default="tdp")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, rank, world)     # rank 0 alone times the oracle
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        dist.init_process_group(backend=backend)
    try:
        return run_tdp(args, rank, world)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
