#!/usr/bin/env python
"""Benchmark of the quantised-weight GEMV / GEMM library on one GB300 (or N replicas).

Headline workload (the GEMV HBM-bandwidth metric): the batch-1 Q4_K decode
GEMVs of a Llama-8B-shaped model, one step = one token through 32 layers.
Per layer: the fused attn_qkv 6144x4096 (one call; q, k and v are the row
ranges 4096/1024/1024 of its output), attn_output 4096x4096, the fused ffn
gate+up 28672x4096 (one call), ffn_down 4096x14336 -- four launches, with
programmatic dependent launch on (weights are loaded once, so a call may
stream its weights while the previous call drains).  Eight distinct layer weight
sets (983 MB, far larger than L2) are rotated, so every weight byte comes
from HBM.  Activations are fixed synthetic N(0,1) vectors (the ops between
the GEMVs are not part of this library).  The step is captured once as a
CUDA graph and replayed.

Printed: one JSON line (rank 0).  `value` is whole-job GB/s of algorithmic
bytes (quant bytes + x + y of every call); see the keys below.
`--impl reference` times the CPU oracle on the host cores instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "quantised GEMV achieved HBM GB/s (% of GB300 peak) and equiv. decode tokens/sec"
LAYERS_PER_TOKEN = 32
DISTINCT_LAYER_SETS = 8
# (name, rows, K, row-range calls as (row_offset, rows))
LAYER = [
    ("attn_qkv", 6144, 4096, [(0, 6144)]),
    ("attn_output", 4096, 4096, [(0, 4096)]),
    ("ffn_gate_up", 28672, 4096, [(0, 28672)]),
    ("ffn_down", 4096, 14336, [(0, 4096)]),
]
# the same layer with attn_qkv issued as its three output row ranges (q, k, v)
QKV_RANGES = [(0, 4096), (4096, 1024), (5120, 1024)]
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def q4k_row_bytes(K: int) -> int:
    return ((K + 255) // 256) * 144


def call_bytes(fmt_row_bytes: int, rows: int, K: int, batch: int) -> int:
    """Algorithmic bytes of one GEMV call: its quant bytes, x once, y once."""
    return rows * fmt_row_bytes + batch * K * 4 + batch * rows * 4


def layer_bytes() -> int:
    tot = 0
    for _, _, K, calls in LAYER:
        for _, n in calls:
            tot += call_bytes(q4k_row_bytes(K), n, K, 1)
    return tot


def launches_per_layer() -> int:
    return sum(len(c) for _, _, _, c in LAYER)


# ---------------------------------------------------------------------- env helpers

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(ms: float, dist, device) -> float:
    """The slowest rank's time: every rank of the group gets the maximum of
    `ms` (dist None: a single process)."""
    if dist is None:
        return ms
    import torch
    tt = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    return float(tt.item())


def whole_job_gbs(world: int, step_bytes: int, ms_step: float) -> float:
    """Whole-job throughput: every rank runs one replica of the step, so the
    job moves world * step_bytes in the slowest rank's step time."""
    return world * step_bytes / (ms_step * 1e-3) / 1e9


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    return d


def peak_hbm(peaks):
    if peaks:
        for k in ("hbm_gbs", "hbm_copy_gbs", "hbm_GBs"):
            if k in peaks and peaks[k]:
                return float(peaks[k]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def peak_bf16(peaks, sustained=False):
    if peaks:
        key = "bf16_tflops_sustained" if sustained else "bf16_tflops"
        if peaks.get(key):
            return float(peaks[key]), "measured"
    return FALLBACK_BF16_TFLOPS, "fallback"


class ClockSampler:
    """nvidia-smi sampling in the background (clocks and throttle reasons)."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, period_ms: int = 50):
        self.index = index
        self.period_ms = period_ms
        self.proc = None
        self.file = None
        self._rows = None

    def __enter__(self):
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.period_ms)],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
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
        self.file.close()

    def samples(self):
        """The parsed samples (read once; the temporary file is removed then)."""
        if self._rows is None:
            try:
                with open(self.file.name) as f:
                    self._rows = parse_clock_lines(f)
            except OSError:
                self._rows = []
            finally:
                try:
                    os.unlink(self.file.name)
                except OSError:
                    pass
        return self._rows


def parse_clock_lines(lines):
    """Rows of `nvidia-smi --query-gpu=<ClockSampler.FIELDS> --format=csv,noheader,nounits`
    as {"t": seconds, "sm": MHz, "max": MHz, "reasons": [active mask, hw_slowdown,
    hw_thermal_slowdown, sw_thermal_slowdown, sw_power_cap]}; malformed lines are skipped."""
    rows = []
    for line in lines:
        parts = [p.strip() for p in line.split(",")]
        if len(parts) < 9:
            continue
        try:
            ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
            frac = float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
            rows.append({"t": ts + frac, "sm": float(parts[1]), "max": float(parts[2]),
                         "reasons": parts[4:9]})
        except (ValueError, IndexError):
            continue
    return rows


def summarise_clocks(samples, t0, t1):
    inside = [s for s in samples if t0 - 0.05 <= s["t"] <= t1 + 0.05]
    window = "timed region"
    if not inside:
        inside = samples
        window = "whole run (timed region shorter than the sampling period)"
    if not inside:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                "samples": 0}
    names = ["active_mask", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    reasons = set()
    for s in inside:
        for n, v in zip(names[1:], s["reasons"][1:]):
            if v.strip().lower() == "active":
                reasons.add(n)
    return {"sm_mhz": statistics.median(s["sm"] for s in inside),
            "sm_max_mhz": max(s["max"] for s in inside),
            "reasons": sorted(reasons), "samples": len(inside), "window": window}


# ---------------------------------------------------------------------- workload

class LayerSetWorkload:
    """Device-resident Q4_K weights of DISTINCT_LAYER_SETS Llama-8B-shaped layers."""

    def __init__(self, torch, qk, synth, device, n_sets=DISTINCT_LAYER_SETS, seed=2):
        self.torch, self.qk = torch, qk
        self.device = device
        self.sets = []
        for li in range(n_sets):
            tensors = {}
            for ti, (name, rows, K, _) in enumerate(LAYER):
                raw = synth.weights("q4_k", rows, K, seed=seed, stream0=1000 * li + 10 * ti)
                tensors[name] = torch.from_numpy(raw).to(device)
            self.sets.append(tensors)
        self.x_host = {K: synth.activations(1, K, seed=seed, stream=200 + K % 97)
                       for K in sorted({K for _, _, K, _ in LAYER})}
        self.x = {K: torch.from_numpy(v).to(device) for K, v in self.x_host.items()}
        # outputs: one buffer per tensor (row ranges of the fused qkv land in one buffer)
        self.y = {name: torch.empty((1, rows), device=device) for name, rows, _, _ in LAYER}
        self.lib = qk.load()
        self.bytes_per_layer = layer_bytes()

    def launch_layer(self, li: int, stream_handle: int, on_launch=None, qkv_ranges: bool = False):
        t = self.sets[li % len(self.sets)]
        fn = self.lib.qmatvec_q4_k
        for name, rows, K, calls in LAYER:
            if qkv_ranges and name == "attn_qkv":
                calls = QKV_RANGES
            w = t[name].data_ptr()
            x = self.x[K].data_ptr()
            ybuf = self.y[name]
            for off, n in calls:
                if on_launch:
                    on_launch(0, name, n, K)
                st = fn(w, off, n, K, x, 1, ybuf.data_ptr() + 4 * off, rows, stream_handle)
                if st != 0:
                    raise RuntimeError(f"qmatvec_q4_k({name}) returned status {st}")
                if on_launch:
                    on_launch(1, name, n, K)

    def launch_step(self, stream_handle: int, first_layer: int = 0, qkv_ranges: bool = False):
        for l in range(LAYERS_PER_TOKEN):
            self.launch_layer(first_layer + l, stream_handle, qkv_ranges=qkv_ranges)


def measure_ours(args, torch, qk, synth, device, rank, world):
    stream = torch.cuda.Stream(device=device)
    sh = stream.cuda_stream
    wl = LayerSetWorkload(torch, qk, synth, device)
    step_bytes = wl.bytes_per_layer * LAYERS_PER_TOKEN
    launches_step = launches_per_layer() * LAYERS_PER_TOKEN

    # eager warm-up (sets kernel attributes before capture)
    with torch.cuda.stream(stream):
        wl.launch_step(sh)
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        wl.launch_step(torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()

    dist = None
    if world > 1:
        import torch.distributed as dist  # noqa: F811
    sampler = ClockSampler(int(os.environ.get("CUDA_VISIBLE_DEVICES", str(device.index or 0)).split(",")[0])
                           if os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")[0].isdigit()
                           else (device.index or 0))
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with sampler:
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        t0 = time.time()
        with torch.cuda.stream(stream):
            start.record(stream)
            for _ in range(args.steps):
                graph.replay()
            end.record(stream)
        torch.cuda.synchronize()
        t1 = time.time()
        if dist:
            dist.barrier()
    ms = max_over_ranks(start.elapsed_time(end), dist, device)
    clocks = summarise_clocks(sampler.samples(), t0, t1)
    ms_step = ms / args.steps
    value = whole_job_gbs(world, step_bytes, ms_step)

    # per-launch durations of the dominant kernel: each distinct call of a
    # layer is timed on row ranges of one tensor holding enough copies of its
    # weights to fill twice the L2 (so every call's bytes come from HBM),
    # captured as a graph of one launch per copy and replayed back to back,
    # CUDA events on the launching stream
    per_call = {}
    tot_b = tot_ms = 0.0
    l2 = getattr(torch.cuda.get_device_properties(device), "L2_cache_size", 128 << 20) or (128 << 20)
    for ti, (name, rows, K, calls) in enumerate(LAYER):
        rb = q4k_row_bytes(K)
        for off, n in calls:
            copies = max(DISTINCT_LAYER_SETS, math.ceil(2 * l2 / (n * rb)) + 1)
            big = torch.from_numpy(synth.weights("q4_k", n * copies, K, seed=7, stream0=10 * ti)).to(device)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                csh = torch.cuda.current_stream().cuda_stream
                for c in range(copies):
                    st = wl.lib.qmatvec_q4_k(big.data_ptr(), c * n, n, K, wl.x[K].data_ptr(), 1,
                                             wl.y[name].data_ptr() + 4 * off, rows, csh)
                    assert st == 0
            reps = 10
            with torch.cuda.stream(stream):
                g.replay()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for _ in range(reps):
                    g.replay()
                e1.record(stream)
            torch.cuda.synchronize()
            dt = e0.elapsed_time(e1) / (reps * copies)
            b = call_bytes(rb, n, K, 1)
            key = f"{name}[{n}x{K}]"
            if key not in per_call:
                per_call[key] = {"bytes": b, "avg_us": round(dt * 1e3, 2), "GB/s": round(b / (dt * 1e-3) / 1e9, 1),
                                 "launches_per_layer": 0, "copies_rotated": copies}
            per_call[key]["launches_per_layer"] += 1
            tot_b += b
            tot_ms += dt
            del g, big
    achieved = tot_b / (tot_ms * 1e-3) / 1e9
    peaks = read_peaks()
    hbm, hbm_src = peak_hbm(peaks)
    traffic = read_traffic("gemv_q4_k_b1", avg_launch_bytes=tot_b / launches_per_layer())
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(achieved / hbm, 4), "traffic": traffic,
                "kernel": "gemv_kernel<Q4_K, batch 1>: the four launches of a layer, each timed as "
                          "back-to-back graph replays over weight copies filling twice the L2",
                "peak_source": f"{hbm_src} HBM copy bandwidth",
                "frac_of_8TBs_nominal": round(achieved / 8000.0, 4),
                "step_frac": round(value / world / hbm, 4),
                "step_frac_note": "the whole decode step's algorithmic bytes / its time (value per GPU) "
                                  "over the same peak",
                "per_call": per_call}

    # the same step with attn_qkv as three row-range calls (q, k, v): 160 launches
    g3 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g3, stream=stream):
        wl.launch_step(torch.cuda.current_stream().cuda_stream, qkv_ranges=True)
    torch.cuda.synchronize()
    n3 = max(5, min(args.steps, 100))
    with torch.cuda.stream(stream):
        for _ in range(3):
            g3.replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n3):
            g3.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    ms3 = e0.elapsed_time(e1) / n3
    step3_bytes = LAYERS_PER_TOKEN * sum(call_bytes(q4k_row_bytes(K), n, K, 1)
                                         for name, _, K, calls in LAYER
                                         for _, n in (QKV_RANGES if name == "attn_qkv" else calls))
    qkv_ranges_row = {"GB/s": round(step3_bytes / (ms3 * 1e-3) / 1e9, 1), "ms_per_step": round(ms3, 5),
                      "launches_per_step": LAYERS_PER_TOKEN * (launches_per_layer() + len(QKV_RANGES) - 1),
                      "bytes_per_step": step3_bytes, "steps": n3,
                      "computes": "the headline step with attn_qkv issued as its q/k/v output row ranges "
                                  "4096/1024/1024 (three calls) instead of one fused call"}
    del g3

    # e2e: the same step through the C ABI from pinned host buffers
    e2e = measure_e2e(args, torch, wl, stream, step_bytes, world)
    extra = {"llama8b_decode_step_qkv_as_3_range_calls": qkv_ranges_row}
    if not args.no_extra:
        extra.update(measure_extra_rows(torch, qk, synth, device, stream))
    del graph
    return {
        "value": value, "ms_per_step": ms_step, "clocks": clocks, "roofline": roofline, "e2e": e2e,
        "gpu_launches": launches_step * args.steps, "step_bytes": step_bytes, "extra": extra,
    }


def read_traffic(kernel_key: str, avg_launch_bytes: float):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    kernel source changed after the counters were taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    ent = d.get(kernel_key)
    if not ent:
        return None
    src = os.path.join(ROOT, "quantised_gguf_weight_gb300", "csrc", ent.get("source", ""))
    try:
        fp = source_fingerprint(src)
    except OSError:
        return None
    if fp != ent.get("source_fingerprint"):
        return None
    return ent.get("dram_bytes_per_launch_avg")


def source_fingerprint(path: str) -> str:
    """sha256 (16 hex digits) of a C/CUDA source with its comments removed and
    its whitespace collapsed: it changes with the code, not with the comments."""
    text = open(path, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return hashlib.sha256(" ".join(text.split()).encode()).hexdigest()[:16]


def measure_e2e(args, torch, wl, stream, step_bytes, world):
    """The step end to end through the public API: the host->device copies
    of the step's activations from pinned memory, the 128 qmatvec_q4_k
    calls and the device->host copy of the last layer's output, captured
    once as a CUDA graph and replayed with a host synchronisation per step.
    The same step issued eagerly from Python is reported beside it."""
    x_pinned = {K: torch.from_numpy(v).pin_memory() for K, v in wl.x_host.items()}
    out_pinned = torch.empty((1, 4096), dtype=torch.float32).pin_memory()
    h2d = sum(v.numel() * 4 for v in x_pinned.values())
    d2h = out_pinned.numel() * 4

    def step(sh):
        for K, v in x_pinned.items():
            wl.x[K].copy_(v, non_blocking=True)
        wl.launch_step(sh)
        out_pinned.copy_(wl.y["ffn_down"], non_blocking=True)

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        step(torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    n = max(3, min(args.steps, 200))
    for _ in range(3):
        g.replay()
        torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(n):
        g.replay()
        torch.cuda.synchronize()
    s_graph = (time.perf_counter() - t0) / n
    del g
    # eager: every call issued from Python through ctypes
    sh = stream.cuda_stream
    ne = max(3, min(args.steps, 20))
    with torch.cuda.stream(stream):
        for it in range(2 + ne):
            if it == 2:
                torch.cuda.synchronize()
                t0 = time.perf_counter()
            step(sh)
            stream.synchronize()
        s_eager = (time.perf_counter() - t0) / ne
    return {"value": round(world * step_bytes / s_graph / 1e9, 1), "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(1e3 * s_graph, 4),
            "path": "pinned H2D + 128 qmatvec_q4_k calls + D2H captured as one CUDA graph, host sync per step",
            "eager_python_ms_per_step": round(1e3 * s_eager, 4),
            "eager_python_GB/s": round(world * step_bytes / s_eager / 1e9, 1)}


def time_calls(torch, stream, fns, iters):
    """Average device time of one call of `fns` (callables taking a stream
    handle), captured as a CUDA graph of all of them and replayed."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        sh = torch.cuda.current_stream().cuda_stream
        for f in fns:
            f(sh)
    with torch.cuda.stream(stream):
        g.replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(iters):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / (iters * len(fns))
    del g
    return ms


def measure_extra_rows(torch, qk, synth, device, stream):
    """The other GEMV configurations, each timed with CUDA events.  Tensors
    larger than L2 are rotated over several copies; the small ones are
    L2-resident by nature and labelled hot."""
    lib = qk.load()
    out = {}
    l2 = getattr(torch.cuda.get_device_properties(device), "L2_cache_size", 128 << 20) or (128 << 20)

    def gemv_row(label, fmt, rows, K, batch, seed, copies, cold_too=False):
        rb = qk.row_bytes(fmt, K)
        ws = [torch.from_numpy(synth.weights(fmt, rows, K, seed=seed, stream0=50 * c)).to(device)
              for c in range(copies)]
        x = torch.from_numpy(synth.activations(batch, K, seed=seed)).to(device)
        y = torch.empty((batch, rows), device=device)
        fn = {"q8_0": lib.qmatvec_q8_0, "q4_k": lib.qmatvec_q4_k, "q6_k": lib.qmatvec_q6_k}[fmt]
        def mk(w, off=0):
            def f(sh):
                st = fn(w.data_ptr(), off, rows, K, x.data_ptr(), batch, y.data_ptr(), rows, sh)
                assert st == 0
            return f
        fns = [mk(w) for w in ws] * max(1, 8 // len(ws))
        avg_ms = time_calls(torch, stream, fns, 20)
        b = call_bytes(rb, rows, K, batch)
        out[label] = {"bytes": b, "avg_us": round(avg_ms * 1e3, 2),
                      "GB/s": round(b / (avg_ms * 1e-3) / 1e9, 1),
                      "cache": "cold (rotated copies > L2)" if copies * rows * rb > l2 else "hot (L2-resident)"}
        if cold_too:
            # the same call on row ranges of one tensor holding n copies of the
            # weights (2 x L2 in all): each call's bytes were last touched
            # n - 1 calls earlier, so they come from HBM
            n = math.ceil(2 * l2 / (rows * rb)) + 1
            big = ws[0].repeat(n)
            avg_ms = time_calls(torch, stream, [mk(big, c * rows) for c in range(n)], 5)
            out[label + "_cold"] = {"bytes": b, "avg_us": round(avg_ms * 1e3, 2),
                                    "GB/s": round(b / (avg_ms * 1e-3) / 1e9, 1),
                                    "cache": f"cold ({n} copies, row ranges of one {n * rows * rb / 1e6:.0f} MB tensor)"}
            del big
        del ws

    def gemm_row(label, M, N, K, seed, copies, mode="store", fmt="q4_k"):
        """mode store: y = x W^T; swiglu: N gate rows and N up rows, h = silu(g) * u."""
        wrows = 2 * N if mode == "swiglu" else N
        ws = [torch.from_numpy(synth.weights(fmt, wrows, K, seed=seed, stream0=50 * c)).to(device)
              for c in range(copies)]
        x = torch.from_numpy(synth.activations(M, K, seed=seed)).to(device)
        y = torch.empty((M, N), device=device)
        nbytes = qk.gemm_workspace_bytes(M, N, K)
        wsp = torch.empty(nbytes, dtype=torch.uint8, device=device)

        def mk(w):
            def f(sh):
                if mode == "swiglu":
                    fn = lib.qgemm_swiglu_q4_k if fmt == "q4_k" else lib.qgemm_swiglu_q8_0
                    st = fn(w.data_ptr(), 0, N, N, K, x.data_ptr(), M, y.data_ptr(), N, wsp.data_ptr(), nbytes, sh)
                else:
                    fn = lib.qgemm_q4_k if fmt == "q4_k" else lib.qgemm_q8_0
                    st = fn(w.data_ptr(), 0, N, K, x.data_ptr(), M, y.data_ptr(), N, wsp.data_ptr(), nbytes, sh)
                assert st == 0
            return f
        avg_ms = time_calls(torch, stream, [mk(w) for w in ws] * max(1, 4 // copies), 20)
        flops = 2.0 * M * wrows * K
        tflops = flops / (avg_ms * 1e-3) / 1e12
        peak, src = peak_bf16(read_peaks())
        out[label] = {"avg_us": round(avg_ms * 1e3, 2), "TFLOP/s": round(tflops, 1), "flops": flops,
                      "bound": "tensor", "frac_of_bf16_peak": round(tflops / peak, 4), "peak_TFLOP/s": peak,
                      "peak_source": f"{src} bf16 dense (burst)",
                      "includes": "x->bf16 pre-pass + tcgen05 GEMM"}
        del ws

    def swiglu_row(label, fmt, F, K, batch, seed, copies):
        """Fused gate+up tensor [2F][K] (gate rows 0..F-1, up rows F..2F-1)."""
        rb = qk.row_bytes(fmt, K)
        ws = [torch.from_numpy(synth.weights(fmt, 2 * F, K, seed=seed, stream0=50 * c)).to(device)
              for c in range(copies)]
        x = torch.from_numpy(synth.activations(batch, K, seed=seed)).to(device)
        h = torch.empty((batch, F), device=device)
        fn = lib.qmatvec_swiglu_q8_0 if fmt == "q8_0" else lib.qmatvec_swiglu_q4_k

        def mk(w):
            def f(sh):
                st = fn(w.data_ptr(), 0, F, F, K, x.data_ptr(), batch, h.data_ptr(), F, sh)
                assert st == 0
            return f
        fns = [mk(w) for w in ws] * max(1, 8 // len(ws))
        avg_ms = time_calls(torch, stream, fns, 20)
        b = 2 * F * rb + batch * K * 4 + batch * F * 4
        out[label] = {"bytes": b, "avg_us": round(avg_ms * 1e3, 2),
                      "GB/s": round(b / (avg_ms * 1e-3) / 1e9, 1),
                      "cache": "cold (rotated copies > L2)" if copies * 2 * F * rb > l2 else "hot (L2-resident)",
                      "computes": "h = silu(W_gate x) * (W_up x), one launch"}
        del ws

    def experts_row(label, fmt, E, rows, K, xk, n_assign, seed):
        """One token's top-n_assign experts of a fused gate+up expert tensor [E][rows][K]."""
        rb = qk.row_bytes(fmt, K)
        w = torch.from_numpy(synth.weights(fmt, E * rows, K, seed=seed)).to(device)
        x = torch.from_numpy(synth.activations((n_assign + xk - 1) // xk, K, seed=seed)).to(device)
        y = torch.empty((n_assign, rows), device=device)
        fn = lib.qmatvec_experts_q8_0 if fmt == "q8_0" else lib.qmatvec_experts_q4_k
        # distinct expert sets per call, so consecutive calls read different weights
        sets = [torch.from_numpy((np.arange(n_assign) * 7 + 13 * c) % E).to(torch.int32).to(device)
                for c in range(8)]

        def mk(ids):
            def f(sh):
                st = fn(w.data_ptr(), E, rows, K, x.data_ptr(), xk, ids.data_ptr(), n_assign, y.data_ptr(), rows, sh)
                assert st == 0
            return f
        avg_ms = time_calls(torch, stream, [mk(i) for i in sets], 20)
        b = n_assign * rows * rb + x.numel() * 4 + n_assign * rows * 4
        out[label] = {"bytes": b, "avg_us": round(avg_ms * 1e3, 2),
                      "GB/s": round(b / (avg_ms * 1e-3) / 1e9, 1),
                      "cache": "cold (expert tensor > L2, 8 expert sets)" if E * rows * rb > l2 else "hot (L2-resident)",
                      "computes": f"{n_assign} assignments x {rows} rows, expert ids from device memory"}
        del w

    gemm_row("q4_k_gemm_512x4096x14336", 512, 14336, 4096, 4, 2)
    gemm_row("q4_k_gemm_swiglu_512x4096x2x14336", 512, 14336, 4096, 4, 2, mode="swiglu")
    gemm_row("q8_0_gemm_512x4096x14336", 512, 14336, 4096, 4, 2, fmt="q8_0")
    gemm_row("q8_0_gemm_512x896x4864", 512, 4864, 896, 1, 1, fmt="q8_0")
    experts_row("q4_k_experts_moe_top8_128x1536x2048", "q4_k", 128, 1536, 2048, 8, 8, 5)
    swiglu_row("q4_k_swiglu_llama8b_ffn_14336x4096_b1", "q4_k", 14336, 4096, 1, 2, 4)
    gemv_row("q8_0_576x576_b1", "q8_0", 576, 576, 1, 0, 1, cold_too=True)
    gemv_row("q4_k_4864x896_b1", "q4_k", 4864, 896, 1, 1, 1, cold_too=True)
    gemv_row("q4_k_896x4864_b1", "q4_k", 896, 4864, 1, 1, 1, cold_too=True)
    gemv_row("q4_k_llama8b_gate_up_28672x4096_b4", "q4_k", 28672, 4096, 4, 2, 2)
    gemv_row("q8_0_lm_head_151936x896_b1", "q8_0", 151936, 896, 1, 3, 3)
    gemv_row("q8_0_lm_head_151936x896_b8", "q8_0", 151936, 896, 8, 3, 3)
    gemv_row("q6_k_lm_head_128256x4096_b1", "q6_k", 128256, 4096, 1, 6, 1)
    gemv_row("q6_k_ffn_down_4096x14336_b1", "q6_k", 4096, 14336, 1, 7, 4)
    return out


# ---------------------------------------------------------------------- reference arm (CPU oracle)

def oracle_sample_run(orc, synth, n_rows_frac: float, threads: int, seed=2):
    """One bounded sample of the layer-set workload through the oracle:
    evenly spaced rows of every tensor (the same fraction of each)."""
    done_bytes = 0
    t = 0.0
    for ti, (name, rows, K, _) in enumerate(LAYER):
        n = max(1, int(rows * n_rows_frac))
        idx = np.linspace(0, rows - 1, n).astype(np.int64)
        rb = q4k_row_bytes(K)
        raw = synth.weights("q4_k", rows, K, seed=seed, stream0=10 * ti)
        x = synth.activations(1, K, seed=seed, stream=200 + K % 97)
        t0 = time.perf_counter()
        orc.gemv_threaded("q4_k", raw, K, x, idx, threads)
        t += time.perf_counter() - t0
        done_bytes += n * rb + K * 4 + n * 4
    return done_bytes, t


def cpu_baseline(budget_s: float = 12.0):
    """The oracle on the host cores over whole layer sets, repeated until about
    `budget_s` seconds of CPU time were spent."""
    from oracle import oracle as orc
    from quantised_gguf_weight_gb300 import synth
    threads = orc.host_cores()
    tot_b = tot_t = 0.0
    passes = 0
    frac = 0.05
    while tot_t < budget_s and passes < 200:
        b, t = oracle_sample_run(orc, synth, frac, threads, seed=2 + passes)
        tot_b += b
        tot_t += t
        passes += 1
        if passes == 1:
            frac = min(1.0, frac * max(1.0, budget_s / 4 / max(t, 1e-3)))
    # the same oracle on one thread (bit-identical results), about 2 s
    b1, t1 = oracle_sample_run(orc, synth, 0.002, 1, seed=1)
    frac1 = min(1.0, 0.002 * max(1.0, 2.0 / max(t1, 1e-3)))
    b1, t1 = oracle_sample_run(orc, synth, frac1, 1, seed=1)
    return {"value": round(tot_b / tot_t / 1e9, 3), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"{passes} passes over evenly spaced rows of every Llama-8B layer tensor "
                      f"(up to {frac:.2f} of the rows per pass), f64 decode-then-dot, {threads} host "
                      f"threads over row bands, {tot_t:.1f} s of oracle time",
            "single_thread": {"value": round(b1 / t1 / 1e9, 4), "unit": "GB/s", "cores": 1,
                              "sample": f"{frac1:.3f} of the rows of every layer tensor, {t1:.1f} s"}}


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    from oracle import oracle as orc
    from quantised_gguf_weight_gb300 import synth
    orc.build()
    threads = orc.host_cores()
    # calibrate a per-step sample so that warm-up + timed steps end within ~2 minutes
    b, t = oracle_sample_run(orc, synth, 0.002, threads)
    per_byte = t / b
    step_s = max(0.02, min(5.0, 100.0 / max(1, args.steps + args.warmup)))
    frac = max(1e-4, min(1.0, step_s / (per_byte * layer_bytes())))
    for _ in range(args.warmup):
        oracle_sample_run(orc, synth, frac, threads)
    tot_b = tot_t = 0.0
    for _ in range(args.steps):
        b, t = oracle_sample_run(orc, synth, frac, threads)
        tot_b += b
        tot_t += t
    value = tot_b / tot_t / 1e9
    ms_step = 1e3 * tot_t / args.steps
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": f"each step: {frac:.4f} of the rows of every tensor of one layer set"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config():
    return {"workload": "llama8b_q4_k_decode_token_gemvs",
            "description": "batch-1 Q4_K GEMVs of 32 Llama-8B-shaped layers per step, four calls a layer: "
                           "attn_qkv 6144x4096 as one fused call (its q/k/v are the output row ranges "
                           "4096/1024/1024; the step with three range calls is timed in other_configs), "
                           "attn_output 4096x4096, fused ffn gate+up 28672x4096, ffn_down 4096x14336",
            "weights": "Q4_K (144-byte super-blocks)", "activations": "fp32 N(0,1)", "batch": 1,
            "layers_per_step": LAYERS_PER_TOKEN, "distinct_layer_weight_sets": DISTINCT_LAYER_SETS,
            "bytes_per_step": layer_bytes() * LAYERS_PER_TOKEN,
            "l2": "inputs larger than L2: 8 distinct layer weight sets (983 MB) rotated",
            "launch": "one CUDA graph per step (128 GEMV launches, programmatic dependent launch)",
            "parallelism": "replicas"}


# ---------------------------------------------------------------------- single-call mode (profiling)

def run_only(args, torch, qk, synth, device):
    """Repeat one GEMV call (rotating weight copies larger than L2 when the
    tensor is big); used for ncu captures of a single kernel."""
    fmt, rows, K, batch = args.only.split(":")
    rows, K, batch = int(rows), int(K), int(batch)
    rb = qk.row_bytes(fmt, K)
    l2 = 128 << 20
    copies = max(1, min(4, math.ceil(2 * l2 / max(1, rows * rb))))
    ws = [torch.from_numpy(synth.weights(fmt, rows, K, seed=1, stream0=50 * c)).to(device)
          for c in range(copies)]
    x = torch.from_numpy(synth.activations(batch, K, seed=1)).to(device)
    y = torch.empty((batch, rows), device=device)
    lib = qk.load()
    fns = {"q8_0": lib.qmatvec_q8_0, "q4_k": lib.qmatvec_q4_k, "q6_k": lib.qmatvec_q6_k}
    if fmt not in fns:
        raise SystemExit(f"--only: unknown format {fmt!r} (q8_0, q4_k or q6_k)")
    fn = fns[fmt]
    if args.no_tc:
        qk.debug_gemv_tc(0)            # batch 2..8: the fp32 form, for comparison
    stream = torch.cuda.Stream(device=device)

    def mk(w):
        def f(sh):
            st = fn(w.data_ptr(), 0, rows, K, x.data_ptr(), batch, y.data_ptr(), rows, sh)
            assert st == 0
        return f
    # eager warm-up launches (also the launches an ncu capture skips)
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            mk(ws[i % copies])(stream.cuda_stream)
    torch.cuda.synchronize()
    ms = time_calls(torch, stream, [mk(w) for w in ws] * max(1, 8 // copies), max(1, args.steps))
    b = call_bytes(rb, rows, K, batch)
    print(json.dumps({"only": args.only, "avg_us": round(ms * 1e3, 2), "GB/s": round(b / (ms * 1e-3) / 1e9, 1),
                      "copies": copies, "form": "fp32" if args.no_tc else "default"}), flush=True)
    return 0


# ---------------------------------------------------------------------- main

def result_line(r, ws: int, args, cpu) -> dict:
    """The JSON line of this arm from the measurements `r` of measure_ours."""
    return {
        "metric": METRIC, "value": round(r["value"], 1), "unit": "GB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(r["ms_per_step"], 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic", "config": workload_config(),
        "tok_s_equiv": round(ws * 1e3 / r["ms_per_step"], 1),
        "roofline": r["roofline"], "cpu_baseline": cpu, "e2e": r["e2e"],
        "gpu_launches": r["gpu_launches"], "clocks": r["clocks"], "other_configs": r["extra"],
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-extra", action="store_true", help="skip the other GEMV configurations")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-pdl", action="store_true", help="launch without programmatic dependent launch")
    ap.add_argument("--only-gemm", default=None,
                    help="M:N:K or MODE:FMT:M:N:K (store|swiglu, q4_k|q8_0) -- time one prefill GEMM only")
    ap.add_argument("--only", default=None, help="FMT:ROWS:K:BATCH -- time one GEMV call only")
    ap.add_argument("--no-tc", action="store_true",
                    help="with --only: batch 2..8 calls take the fp32 form instead of the tensor-core form")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)

    import torch
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    from quantised_gguf_weight_gb300 import build as qbuild
    qbuild.build()
    from quantised_gguf_weight_gb300 import qk, synth
    qk.load()
    qk.set_programmatic_launch(not args.no_pdl)
    if args.only:
        return run_only(args, torch, qk, synth, device)
    if args.only_gemm:
        # M:N:K (the Q4_K store GEMM) or MODE:FMT:M:N:K (MODE store or swiglu,
        # FMT q4_k or q8_0; swiglu: N gate rows and N up rows, h = silu(g) * u)
        parts = args.only_gemm.split(":")
        mode, fmt = ("store", "q4_k") if len(parts) == 3 else (parts[0], parts[1])
        if mode not in ("store", "swiglu") or fmt not in ("q4_k", "q8_0"):
            raise SystemExit(f"--only-gemm: unknown mode or format in {args.only_gemm!r}")
        M, N, K = (int(v) for v in parts[-3:])
        wrows = 2 * N if mode == "swiglu" else N
        wq = torch.from_numpy(synth.weights(fmt, wrows, K, seed=4)).to(device)
        x = torch.from_numpy(synth.activations(M, K, seed=4)).to(device)
        y = torch.empty((M, N), device=device)
        wsp = torch.empty(qk.gemm_workspace_bytes(M, N, K), dtype=torch.uint8, device=device)
        stream = torch.cuda.Stream(device=device)
        lib = qk.load()
        fn = {("store", "q4_k"): lib.qgemm_q4_k, ("store", "q8_0"): lib.qgemm_q8_0,
              ("swiglu", "q4_k"): lib.qgemm_swiglu_q4_k, ("swiglu", "q8_0"): lib.qgemm_swiglu_q8_0}[(mode, fmt)]

        def f(sh):
            if mode == "swiglu":
                st = fn(wq.data_ptr(), 0, N, N, K, x.data_ptr(), M, y.data_ptr(), N, wsp.data_ptr(), wsp.numel(), sh)
            else:
                st = fn(wq.data_ptr(), 0, N, K, x.data_ptr(), M, y.data_ptr(), N, wsp.data_ptr(), wsp.numel(), sh)
            assert st == 0
        # eager warm-up launches (also the launches an ncu capture skips)
        with torch.cuda.stream(stream):
            for _ in range(args.warmup):
                f(stream.cuda_stream)
        torch.cuda.synchronize()
        ms = time_calls(torch, stream, [f] * 4, max(1, args.steps))
        flops = 2.0 * M * wrows * K
        print(json.dumps({"only_gemm": args.only_gemm, "avg_us": round(ms * 1e3, 2),
                          "TFLOP/s": round(flops / (ms * 1e-3) / 1e12, 1)}), flush=True)
        return 0
    r = measure_ours(args, torch, qk, synth, device, rank, ws)
    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline()
    if rank == 0:
        print(json.dumps(result_line(r, ws, args, cpu)), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
