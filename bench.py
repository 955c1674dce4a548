#!/usr/bin/env python
"""Benchmark of the fused W4A16 MoE layer on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

A step is one call of the whole layer (route handling, FC1 + activation, FC2 +
top-k combine) on one batch of synthetic inputs.  The headline workload is
the decode MoE (NVFP4, E=128, top_k=8, H=4096, I=1536, ReLU^2, m=1); the
metric is microseconds per call (lower is better).

Timed region: one replay of a CUDA graph holding exactly K back-to-back calls,
bracketed by CUDA events on the launching stream, inputs already resident in
HBM.  Consecutive calls cycle through several device copies of the prepared
weights (as consecutive MoE layers of a model read different weights) and
eight routing/activation draws, so that at least three times the L2 size of
other weights is read between two calls on the same copy: the inputs are
larger than L2 and every call streams its experts from HBM.  L2 is flushed
(512 MiB written, then read back) before the timed replay.  The single-call
figure of earlier measurements (one call per graph replay, L2 and code cold
before each) is kept beside it as "us_per_call_single".

Besides the headline it reports, in "secondary", the same measurement for
the other workloads (decode m=2, 4; small-batch m=16, 64; prefill m=2048 with
SwiGLU and ReLU^2; MXFP4 m=512; the dense W4A16 linear layer b4_linear,
N = K = 4096, m = 1, 16, 2048), each with its weight-stream TB/s and bf16
TFLOP/s; in "crossover", the decode workload at m = 4..64 with the small-m and
the grouped path each forced; "roofline" for the dominant kernel (timed per
launch with the library's timing events in a second graph of the same calls),
"cpu_baseline" (the float64 CPU oracle on a bounded sample), "e2e" (the same
calls through the Python API with host buffers: one graph of K steps, each a
host->device copy of the step's inputs from pinned memory, the call and the
device->host copy of the result; wall clock around replay and synchronize)
and the SM clocks sampled during the timed region.

Replicas only: under torchrun every rank runs the same workload on its own GPU
with no collective on the data path; rank 0 prints the max over ranks.
``--impl reference`` times the CPU oracle instead (the reference arm).
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused W4A16 MoE µs/call; weight-stream TB/s (m≤16), bf16 TFLOPS (m=2048)"
HEADLINE = ("decode", "relu2", 1)
SECONDARY = [("decode", "relu2", 2), ("decode", "relu2", 4), ("small", "silu", 16), ("small", "silu", 64),
             ("prefill", "silu", 2048), ("prefill", "relu2", 2048), ("mxfp4", "silu", 512),
             ("linear", "none", 1), ("linear", "none", 16), ("linear", "none", 2048)]
# the small-m / grouped crossover: the same workload with each path forced
CROSSOVER = [("decode", "relu2", m, path) for m in (4, 8, 16, 32, 64) for path in ("decode", "grouped")]
L2_FLUSH_BYTES = 512 << 20
DRAWS = 8  # independent routing / activation draws cycled through the steps


def torch_int32():
    import torch

    return torch.int32


def describe(wl, m):
    if wl.name == "linear":
        return (f"linear {'NVFP4' if wl.fmt.startswith('nvfp4') else 'MXFP4'} dense W4A16 linear layer: "
                f"N={wl.inter} K={wl.hidden} m={m}")
    return (f"{wl.name} {'NVFP4' if wl.fmt.startswith('nvfp4') else 'MXFP4'} MoE: E_g={wl.num_global_experts} "
            f"E_l={wl.num_local_experts} top_k={wl.top_k} H={wl.hidden} I={wl.inter} "
            f"{'SiLU-SwiGLU' if wl.act == 'silu' else 'ReLU^2'} m={m}")


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            d = json.load(fh)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "src": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "src": "fallback"}


# --------------------------------------------------------------- accounting
def tensor_bytes(wl, which):
    """Unpadded bytes of one expert's codes + scales (+ fp32 global scale)."""
    n, k = (wl.n1, wl.hidden) if which == 0 else (wl.hidden, wl.inter)
    return n * k // 2 + n * k // wl.group + (4 if wl.fmt.startswith("nvfp4") else 0)


def local_experts_np(wl, ids, em):
    ids = np.asarray(ids, dtype=np.int64)
    valid = (ids >= 0) & (ids < wl.num_global_experts)
    loc = np.where(valid, ids, 0)
    if em is not None:
        loc = np.asarray(em, dtype=np.int64)[loc]
    valid &= (loc >= 0) & (loc < wl.num_local_experts)
    return np.where(valid, loc, -1)


def call_accounting(wl, m, ids, em):
    loc = local_experts_np(wl, ids, em)
    hit = np.unique(loc[loc >= 0])
    r_valid = int((loc >= 0).sum())
    b13 = len(hit) * tensor_bytes(wl, 0)
    b2 = len(hit) * tensor_bytes(wl, 1)
    io = m * wl.hidden * 2 * 2 + m * wl.top_k * 8  # x, out, ids, router weights
    f13 = 2.0 * r_valid * wl.n1 * wl.hidden
    f2 = 2.0 * r_valid * wl.hidden * wl.inter
    return {"bytes": b13 + b2 + io, "weight_bytes": b13 + b2, "fc1_bytes": b13 + m * wl.hidden * 2,
            "fc2_bytes": b2, "flops": f13 + f2, "experts_hit": int(len(hit)), "routes": r_valid}


def weight_copies(b, dev, n=None):
    """Device copies of the prepared weights, cycled call by call so that no
    call finds its weights in L2: enough copies that three times the L2 size
    passes between two calls on the same copy (at least 2, at most 64), or
    exactly n (a profiling run that keeps the device footprint small)."""
    import math

    torch = b.torch
    if n is not None and n > 0:
        return [dev] + [{k: (None if v is None else v.clone()) for k, v in dev.items()} for _ in range(n - 1)]
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    per_call = statistics.mean(d["acct"]["weight_bytes"] for d in b.draws)
    n = int(min(64, max(2, math.ceil(3 * l2 / max(per_call, 1)))))
    return [dev] + [{k: (None if v is None else v.clone()) for k, v in dev.items()} for _ in range(n - 1)]


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        self.gpu = gpu_index
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is None:
            return
        time.sleep(0.3)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------- our arm
class Bench:
    def __init__(self, wl, m, seed=7, path=None, copies=None):
        import torch

        import w4a16_moe_gb300 as b4
        import workloads as W

        self.torch, self.b4, self.W = torch, b4, W
        self.wl, self.m = wl, m
        self.act = b4.ACTIVATIONS[wl.act]
        self.em_np = W.expert_map(wl)
        em = None if self.em_np is None else torch.from_numpy(self.em_np).cuda()
        self.path = b4.PATH_AUTO if path is None else path
        self.cfg = b4.MoEConfig(m, wl.top_k, wl.num_global_experts, wl.num_local_experts, wl.hidden, wl.inter,
                                format=b4.FORMATS[wl.fmt], path=self.path, expert_map=em)
        self.host = {}
        dev = {}
        for which, name in ((0, "13"), (1, "2")):
            c, s, g = W.random_codes(wl, seed, which)
            self.host["c" + name], self.host["s" + name], self.host["g" + name] = c, s, g
            wc, ws = b4.prepare_weights(self.cfg, which, self.act, torch.from_numpy(c).cuda(),
                                        torch.from_numpy(s).cuda())
            dev["w" + name], dev["s" + name] = wc, ws
            dev["g" + name] = None if g is None else torch.from_numpy(g).cuda()
        self.dev = dev
        self.draws = []
        for d in range(DRAWS):
            xb, x = W.activations(wl, m, seed=100 + d)
            ids, wts = W.routing(wl, m, seed=100 + d)
            self.draws.append({
                "x_bits": xb, "x": x, "ids": ids, "wts": wts,
                "xd": torch.from_numpy(xb.view(np.int16)).cuda().view(torch.bfloat16),
                "idsd": torch.from_numpy(ids).cuda(), "wtsd": torch.from_numpy(wts).cuda(),
                "acct": call_accounting(wl, m, ids, self.em_np)})
        self.devs = weight_copies(self, dev, copies)
        self.ws = torch.empty(b4.workspace_bytes(self.cfg, self.act), dtype=torch.uint8, device="cuda")
        self.out = torch.empty(m, wl.hidden, dtype=torch.bfloat16, device="cuda")
        self.flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
        self.flush_sink = torch.empty(1, dtype=torch.int32, device="cuda")
        self.stream = torch.cuda.Stream()
        # the library's AUTO rule: a small-m kernel (one cooperative launch) up to m = 16, and up
        # to m = 64 while there are at most two routes per local expert
        self.decode = self.path == b4.PATH_DECODE or (self.path == b4.PATH_AUTO and (
            m <= 16 or (m <= 64 and m * wl.top_k <= 2 * wl.num_local_experts)))
        self.n_kernels = 1 if self.decode else 4  # timed intervals: decode kernel; pack (+ x copy), FC1, FC2, finalize
        self.launches = 1 if self.decode else 4  # this library's kernels per call

    def flush_l2(self):
        """Evict L2: write a 512 MiB buffer (evicts everything) and read it back,
        so the write-backs of the now-dirty lines happen here, outside the timed
        region, and the measured call starts from a cold, clean L2."""
        self.flush.zero_()
        self.flush_sink.copy_(self.flush.view(torch_int32()).amax(dim=0, keepdim=True)[:1])

    def call(self, d, stream=None, dv=None):
        dv = dv or self.dev
        self.b4.fused_moe(self.cfg, d["xd"], dv["w13"], dv["s13"], dv["g13"], dv["w2"], dv["s2"], dv["g2"], d["idsd"],
                          d["wtsd"], self.act, self.out, self.ws, stream=stream)

    def call_i(self, i, stream):
        """Call i of a sequence: weight copy i mod copies, draw i mod DRAWS."""
        self.call(self.draws[i % DRAWS], stream, self.devs[i % len(self.devs)])

    def capture_seq(self, n, events=None):
        """One CUDA graph of n back-to-back calls (events: per call, the
        library's timing events, created beforehand; or None)."""
        torch = self.torch
        with torch.cuda.stream(self.stream):
            for i in range(min(n, 2 * len(self.devs))):  # eager warm-up (kernel attributes before capture)
                self.call_i(i, self.stream)
        self.stream.synchronize()
        self.b4.check_status(self.ws, self.stream)
        g = torch.cuda.CUDAGraph()
        try:
            with torch.cuda.graph(g, stream=self.stream):
                for i in range(n):
                    if events is not None:
                        self.b4.set_timing_events(events[i])
                    self.call_i(i, self.stream)
        finally:
            if events is not None:
                self.b4.set_timing_events(None)
        return g

    def time_seq(self, steps, warmup, barrier=None):
        """The timed region: one replay of a graph of exactly `steps` calls,
        after the L2 flush and >= `warmup` untimed calls; the per-kernel
        durations come from a second graph of the same calls with the
        library's timing events between its kernels."""
        torch = self.torch
        g = self.capture_seq(steps)
        with torch.cuda.stream(self.stream):
            for _ in range(max(1, -(-warmup // steps))):
                self.flush_l2()
                g.replay()
        torch.cuda.synchronize()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(self.stream):
            self.flush_l2()
        if barrier:
            barrier()
        torch.cuda.synchronize()
        t_wall = time.perf_counter()
        with torch.cuda.stream(self.stream):
            start.record(self.stream)
            g.replay()
            end.record(self.stream)
        torch.cuda.synchronize()
        if barrier:
            barrier()
        wall = time.perf_counter() - t_wall
        ms_total = start.elapsed_time(end)
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(self.n_kernels + 1)] for _ in range(steps)]
        side = torch.cuda.Stream()
        for ev in evs:  # create the CUDA events outside the capture
            for e in ev:
                e.record(side)
        side.synchronize()
        tg = self.capture_seq(steps, events=evs)
        with torch.cuda.stream(self.stream):
            self.flush_l2()
            tg.replay()
        torch.cuda.synchronize()
        kern = [[ev[j].elapsed_time(ev[j + 1]) for j in range(self.n_kernels)] for ev in evs]
        return ms_total, kern, wall

    def capture(self, timing_events=None):
        torch = self.torch
        graphs = []
        with torch.cuda.stream(self.stream):
            for d in self.draws:  # eager warm-up (sets kernel attributes before capture)
                self.call(d, self.stream)
        self.stream.synchronize()
        self.b4.check_status(self.ws, self.stream)
        if timing_events is not None:
            self.b4.set_timing_events(timing_events)
        try:
            for d in self.draws:
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=self.stream):
                    self.call(d, self.stream)
                graphs.append(g)
        finally:
            if timing_events is not None:
                self.b4.set_timing_events(None)
        return graphs

    def time_steps(self, graphs, steps, warmup, barrier=None, kernel_events=None):
        torch = self.torch
        for i in range(warmup):
            with torch.cuda.stream(self.stream):
                self.flush_l2()
                graphs[i % len(graphs)].replay()
        torch.cuda.synchronize()
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        kern = []
        if barrier:
            barrier()
        torch.cuda.synchronize()
        t_wall = time.perf_counter()
        with torch.cuda.stream(self.stream):
            for i in range(steps):
                self.flush_l2()
                starts[i].record(self.stream)
                graphs[i % len(graphs)].replay()
                ends[i].record(self.stream)
                if kernel_events is not None:
                    self.stream.synchronize()
                    kern.append([kernel_events[j].elapsed_time(kernel_events[j + 1])
                                 for j in range(len(kernel_events) - 1)])
        torch.cuda.synchronize()
        if barrier:
            barrier()
        wall = time.perf_counter() - t_wall
        ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
        return ms, kern, wall

    def run(self, steps, warmup, barrier=None, with_e2e=False, with_clocks=False, gpu_index=0):
        clocks = None
        if with_clocks:
            with ClockSampler(gpu_index) as cs:
                ms_total, kern, wall = self.time_seq(steps, warmup, barrier)
            clocks = cs.summary()
        else:
            ms_total, kern, wall = self.time_seq(steps, warmup, barrier)
        # the single-call measurement: a graph of one call, L2 flushed before each
        graphs = self.capture()
        ms_single, _, _ = self.time_steps(graphs, min(steps, 10), 3, None)
        accts = [self.draws[i % DRAWS]["acct"] for i in range(steps)]
        res = {"ms": [ms_total / steps], "ms_total": ms_total, "kern": kern, "accts": accts, "wall": wall,
               "clocks": clocks, "single_ms": ms_single}
        if with_e2e:
            res["e2e_s"] = self.e2e_timed(steps, warmup)
        return res

    def e2e_timed(self, steps, warmup):
        """End to end through the public call with host buffers: one graph of
        `steps` steps, each a host->device copy of that step's inputs (x, ids
        and router weights packed in one pinned buffer), the fused call (weight
        copies cycled as in the device-timed region) and a device->host copy
        of out; wall clock around the replay and the synchronize."""
        torch = self.torch
        m, H, k = self.m, self.wl.hidden, self.wl.top_k
        xb, ib, wb = m * H * 2, m * k * 4, m * k * 4
        x_off = 0
        i_off = (xb + 255) // 256 * 256
        w_off = i_off + (ib + 255) // 256 * 256
        nbytes = w_off + (wb + 255) // 256 * 256
        dstage = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        xd = dstage[x_off:x_off + xb].view(torch.bfloat16).view(m, H)
        idsd = dstage[i_off:i_off + ib].view(torch.int32).view(m, k)
        wtsd = dstage[w_off:w_off + wb].view(torch.float32).view(m, k)
        out_h = torch.empty(m, H, dtype=torch.int16).pin_memory()
        s = self.stream
        stages = []
        for d in self.draws:
            h = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
            h[x_off:x_off + xb].view(torch.int16).copy_(torch.from_numpy(d["x_bits"].view(np.int16).reshape(-1)))
            h[i_off:i_off + ib].view(torch.int32).copy_(torch.from_numpy(d["ids"].reshape(-1)))
            h[w_off:w_off + wb].view(torch.float32).copy_(torch.from_numpy(d["wts"].reshape(-1)))
            stages.append(h)

        def step(i):
            dv = self.devs[i % len(self.devs)]
            dstage.copy_(stages[i % DRAWS], non_blocking=True)
            self.b4.fused_moe(self.cfg, xd, dv["w13"], dv["s13"], dv["g13"], dv["w2"], dv["s2"], dv["g2"],
                              idsd, wtsd, self.act, self.out, self.ws, stream=s)
            out_h.copy_(self.out.view(torch.int16), non_blocking=True)

        with torch.cuda.stream(s):
            step(0)  # eager first: kernel attributes are set outside capture
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for i in range(steps):
                step(i)
        for _ in range(max(1, -(-warmup // steps))):
            with torch.cuda.stream(s):
                g.replay()
            s.synchronize()
        with torch.cuda.stream(s):
            self.flush_l2()
        torch.cuda.synchronize()
        ta = time.perf_counter()
        with torch.cuda.stream(s):  # a graph replays on the current stream
            g.replay()
        s.synchronize()
        total = time.perf_counter() - ta
        return {"seconds": total, "h2d": xb + ib + wb, "d2h": m * H * 2}


# DRAM traffic of the dominant kernel(s) per call, from one ncu capture
# (dram__bytes_read.sum + dram__bytes_write.sum; the summaries under profiles/
# give the commands).  A figure is reported only while the kernel sources still
# hash to the profiled ones; after any change it is null until re-measured.
KERNEL_SOURCES = {
    "decode": ["decode_moe.cu", "decode_stage.cuh", "dequant.cuh", "ptx.cuh", "kernels.cuh"],
    "decode_grouped": ["decode_grouped.cu", "decode_stage.cuh", "dequant.cuh", "ptx.cuh", "kernels.cuh"],
    "grouped": ["moe_gemm.cu", "dequant.cuh", "tma.cuh", "ptx.cuh", "kernels.cuh"],
    "grouped_wn": ["moe_gemm_wn.cu", "dequant.cuh", "tma.cuh", "ptx.cuh", "kernels.cuh"],
}
NCU_TRAFFIC = {  # (kernel family, workload, m): (source hash, DRAM read + write bytes per call of the GEMM kernel(s))
    ("decode", "decode:relu2", 1): ("f4762e7f1cc4ce5b", 56_734_720 + 302_080),
    ("decode", "small:silu", 16): ("f4762e7f1cc4ce5b", 170_955_008 + 4_806_400),
    ("grouped", "prefill:silu", 2048): ("8f4474bd57eddfdb", 1_040_493_056 + 81_164_032 + 600_330_496 + 81_992_704),
    ("grouped_wn", "small:silu", 64): ("f67e0adcb567f92f", 180_109_312 + 4_455_168 + 90_866_432 + 75_008),
}


class LinearBench(Bench):
    """The dense W4A16 linear layer (b4_linear) on the same timing harness:
    a step is one call, out [m, N] = x [m, K] . W^T."""

    def __init__(self, wl, m, seed=7):
        import torch

        import w4a16_moe_gb300 as b4
        import workloads as W

        self.torch, self.b4, self.W = torch, b4, W
        self.wl, self.m = wl, m
        n, k = wl.inter, wl.hidden
        self.cfg = b4.linear_config(m, n, k, format=b4.FORMATS[wl.fmt])
        c, s, g = W.random_codes(wl, seed, 0)
        wc, ws = b4.prepare_linear_weights(self.cfg, torch.from_numpy(c).cuda(), torch.from_numpy(s).cuda())
        self.dev = {"w": wc, "s": ws, "g": None if g is None else torch.from_numpy(g).cuda()}
        wbytes = n * k // 2 + n * k // wl.group + (4 if g is not None else 0)
        acct = {"bytes": wbytes + m * k * 2 + m * n * 2, "weight_bytes": wbytes, "fc1_bytes": wbytes + m * k * 2,
                "fc2_bytes": m * n * 2, "flops": 2.0 * m * n * k, "experts_hit": 1, "routes": m}
        self.draws = []
        for d in range(DRAWS):
            xb, x = W.activations(wl, m, seed=100 + d)
            self.draws.append({"x_bits": xb, "x": x, "acct": acct,
                               "xd": torch.from_numpy(xb.view(np.int16)).cuda().view(torch.bfloat16)})
        self.devs = weight_copies(self, self.dev)
        self.ws = torch.empty(b4.linear_workspace_bytes(self.cfg), dtype=torch.uint8, device="cuda")
        self.out = torch.empty(m, n, dtype=torch.bfloat16, device="cuda")
        self.flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
        self.flush_sink = torch.empty(1, dtype=torch.int32, device="cuda")
        self.stream = torch.cuda.Stream()
        # the fused small-m kernels (one launch) for m <= 16; above, the grouped
        # GEMM: with fewer (chunk, tile pair) units than SMs it splits K and adds
        # fp32 partials (events: memset + route pack, GEMM, rounding pass),
        # otherwise it stores bf16 (route pack, GEMM)
        self.decode = m <= 16  # AUTO: the small-m kernels (per-route m <= 4, route-grouped above)
        sms = torch.cuda.get_device_properties(0).multi_processor_count
        k_split = m < 96 and -(-m // 128) * ((-(-n // 128) + 1) // 2) < sms
        self.n_kernels = 1 if self.decode else (3 if k_split else 2)
        self.launches = 1 if self.decode else (3 if k_split else 2)  # pack, GEMM (, rounding pass)

    def call(self, d, stream=None, dv=None):
        dv = dv or self.dev
        self.b4.linear(self.cfg, d["xd"], dv["w"], dv["s"], dv["g"], self.out, self.ws, stream=stream)


def source_hash(texts):
    """Hash of source texts with comments and blank lines removed: a comment
    edit does not change the kernels the counters were taken on."""
    import hashlib
    import re

    h = hashlib.sha256()
    for src in texts:
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        h.update("\n".join(line.rstrip() for line in src.splitlines() if line.strip()).encode())
    return h.hexdigest()[:16]


def kernel_source_hash(path):
    csrc = os.path.join(os.path.dirname(os.path.abspath(__file__)), "w4a16_moe_gb300", "csrc")
    texts = []
    for f in KERNEL_SOURCES[path]:
        with open(os.path.join(csrc, f)) as fh:
            texts.append(fh.read())
    return source_hash(texts)


def kernel_family(b):
    """Which GEMM kernels serve the call: the per-route small-m kernel
    (m <= 4, m top_k <= E_local, or up to 2 E_local and 256 routes), the
    route-grouped small-m kernel, or the
    grouped weights-on-N / weights-on-M kernels (api.cu's dispatch rule)."""
    if b.decode:
        wl = b.wl
        if isinstance(b, LinearBench):
            per_route = b.m <= 4
        else:
            r = b.m * wl.top_k
            e_l = wl.num_local_experts
            per_route = b.m <= 4 or r <= e_l or (r <= 2 * e_l and r <= 256)
        return "decode" if per_route else "decode_grouped"
    wl = b.wl
    return "grouped_wn" if b.m * wl.top_k < 96 * wl.num_local_experts else "grouped"


def measured_traffic(b):
    path = kernel_family(b)
    rec = NCU_TRAFFIC.get((path, f"{b.wl.name}:{b.wl.act}", b.m))
    if rec is None or rec[0] != kernel_source_hash(path):
        return None
    return rec[1]


def summarize(b: Bench, res, peaks):
    wl, m = b.wl, b.m
    ms = res["ms"]
    us = 1e3 * statistics.mean(ms)
    acct_bytes = statistics.mean(a["bytes"] for a in res["accts"])
    acct_flops = statistics.mean(a["flops"] for a in res["accts"])
    wbytes = statistics.mean(a["weight_bytes"] for a in res["accts"])
    # GEMM kernels: the fused decode kernel (0); grouped FC1 (1) and FC2 (2);
    # the linear layer's grouped GEMM (1)
    gi = (0,) if b.decode else ((1,) if isinstance(b, LinearBench) else (1, 2))
    kern = res["kern"]
    gemm_ms = [sum(k[j] for j in gi) for k in kern]
    gemm_s = 1e-3 * statistics.mean(gemm_ms)
    g_bytes = statistics.mean(a["fc1_bytes"] + a["fc2_bytes"] for a in res["accts"])
    single = res.get("single_ms") or ms
    out = {
        "workload": describe(wl, m),
        "us_per_call": round(us, 3),
        "us_per_call_single": round(1e3 * statistics.mean(single), 3),
        "tokens_per_s": round(m / (us * 1e-6), 1),
        "weight_stream_TBps": round(wbytes / (us * 1e-6) / 1e12, 4),
        "algorithmic_TBps": round(acct_bytes / (us * 1e-6) / 1e12, 4),
        "bf16_TFLOPs": round(acct_flops / (us * 1e-6) / 1e12, 2),
        "experts_hit_mean": round(statistics.mean(a["experts_hit"] for a in res["accts"]), 2),
        "kernel_us_mean": [round(1e3 * statistics.mean(k[j] for k in kern), 3) for j in range(len(kern[0]))],
        "gemm_us": round(gemm_s * 1e6, 3),
    }
    # frac: the dominant kernel(s) alone (per-launch duration from the timing
    # events); frac_per_call: the same algorithmic figure over the whole call
    if b.decode or m <= 64:
        ach = g_bytes / gemm_s / 1e9
        per_call = acct_bytes / (us * 1e-6) / 1e9
        out["roofline"] = {"bound": "hbm", "achieved": round(ach, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                           "frac": round(ach / peaks["hbm_gbs"], 4),
                           "frac_per_call": round(per_call / peaks["hbm_gbs"], 4), "traffic": measured_traffic(b),
                           "peak_src": peaks["src"]}
    else:
        ach = acct_flops / gemm_s / 1e12
        per_call = acct_flops / (us * 1e-6) / 1e12
        out["roofline"] = {"bound": "tensor", "achieved": round(ach, 1), "peak": peaks["bf16_tflops"],
                           "unit": "TFLOP/s", "frac": round(ach / peaks["bf16_tflops"], 4),
                           "frac_per_call": round(per_call / peaks["bf16_tflops"], 4),
                           "traffic": measured_traffic(b), "peak_src": peaks["src"]}
    return out


def cpu_baseline(b: Bench, budget_s=15.0, max_calls=20):
    """The float64 oracle as it stands on the host cores, on a bounded sample of the headline workload."""
    from oracle import moe as M

    h, wl = b.host, b.wl
    t0 = time.perf_counter()
    n = 0
    while n < max_calls and (time.perf_counter() - t0) < budget_s:
        d = b.draws[n % DRAWS]
        M.fused_moe(d["x"], h["c13"], h["s13"], h["g13"], h["c2"], h["s2"], h["g2"], d["ids"], d["wts"], wl.act,
                    wl.fmt, wl.num_global_experts, expert_map=b.em_np)
        n += 1
    dt = time.perf_counter() - t0
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return {"value": round(dt / n * 1e6, 1), "unit": "us/call", "cores": cores, "kind": "oracle",
            "sample": f"{n} full calls of the headline workload ({describe(wl, b.m)}), float64 numpy, "
                      f"{dt:.1f} s; numpy/BLAS default threading on {cores} host cores"}


def run_reference(args):
    """Reference arm: the CPU oracle, as it stands, on a bounded sample of the headline workload."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import workloads as W
    from oracle import moe as M

    name, act, m = HEADLINE
    wl = W.WORKLOADS[name].with_act(act)
    c13, s13, g13 = W.random_codes(wl, 7, 0)
    c2, s2, g2 = W.random_codes(wl, 7, 1)
    em = W.expert_map(wl)
    draws = [(W.activations(wl, m, 100 + d)[1],) + W.routing(wl, m, 100 + d) for d in range(DRAWS)]

    def step(i):
        x, ids, wts = draws[i % DRAWS]
        M.fused_moe(x, c13, s13, g13, c2, s2, g2, ids, wts, wl.act, wl.fmt, wl.num_global_experts, expert_map=em)

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(i)
    dt = time.perf_counter() - t0
    us = dt / args.steps * 1e6
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    line = {
        "impl": "reference", "metric": METRIC, "value": round(us, 1), "unit": "us/call", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(us / 1e3, 3), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": describe(wl, m), "weights": "random E2M1 codes, plausible block scales"},
        "cpu_baseline": {"value": round(us, 1), "unit": "us/call", "cores": cores, "kind": "oracle",
                         "sample": f"{args.steps} full calls of the headline workload after {args.warmup} warm-up"},
        "e2e": {"value": round(us, 1), "unit": "us/call", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def max_over_ranks(value, dist, device):
    """The slowest rank's value (replicas: the job's time per step is the
    longest rank's); every rank gets it."""
    import torch

    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--no-crossover", action="store_true")
    ap.add_argument("--weight-copies", type=int, default=0,
                    help="device copies of the weights cycled by the timed calls (0: enough to keep them L2-cold)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", default="decode:relu2:1",
                    help="name:act:m of the timed workload (default: the decode headline)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
        return
    if args.workload.split(":")[0] == "linear":
        ap.error("the linear layer is reported in the secondary lines, not as the headline")

    import torch

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    barrier = None
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        barrier = dist.barrier

    import w4a16_moe_gb300 as b4
    import workloads as W

    peaks = load_peaks()
    name, act, m = args.workload.split(":")
    m = int(m)
    b = Bench(W.WORKLOADS[name].with_act(act), m, copies=args.weight_copies or None)
    res = b.run(args.steps, args.warmup, barrier, with_e2e=True, with_clocks=True, gpu_index=local)
    head = summarize(b, res, peaks)
    us = head["us_per_call"]
    if dist is not None:
        us = max_over_ranks(us, dist, "cuda")
    e2e = res["e2e_s"]
    e2e_us = e2e["seconds"] / args.steps * 1e6
    line = {
        "metric": METRIC, "value": us, "unit": "us/call", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(us / 1e3, 5), "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded; random FP4 codes, softmax top-k routing)",
        "config": {"workload": head["workload"], "parallelism": f"replicas x{world}",
                   "l2": (f"inputs larger than L2: consecutive calls cycle {len(b.devs)} device copies of the "
                          f"prepared weights and {DRAWS} routing/activation draws, so >= 3x the L2 size of other "
                          "weights is read between two calls on the same copy; L2 flushed (512 MiB written, then "
                          "read back) before the timed region") if not args.weight_copies else
                         (f"profiling run: {args.weight_copies} weight copies set by --weight-copies (calls may "
                          "find weights in L2); L2 flushed before the timed region"),
                   "launch": f"one CUDA graph of the {args.steps} timed calls, replayed once",
                   "us_per_call_single": head["us_per_call_single"],
                   "single_note": "one call per graph replay, L2 flushed before each (cold L2 and cold code)",
                   "tokens_per_s": round(head["tokens_per_s"] * world, 1),
                   "weight_stream_TBps": head["weight_stream_TBps"], "bf16_TFLOPs": head["bf16_TFLOPs"]},
        "roofline": {k: v for k, v in head["roofline"].items() if k != "peak_src"},
        "roofline_note": (("dominant kernel: the fused decode kernel (FC1, FC2 and combine in one launch)"
                           if b.decode else "dominant kernels: the grouped FC1 and FC2 GEMM launches")
                          + "; frac over those kernels' event-timed duration, frac_per_call over the whole call"
                          + f"; peak of {head['roofline']['peak_src']} MEASURED_PEAKS.json; traffic = ncu DRAM "
                          "bytes per call of those launches (null if their sources changed since the capture)"),
        "e2e": {"value": round(e2e_us, 2), "unit": "us/call", "h2d_bytes_per_step": e2e["h2d"],
                "d2h_bytes_per_step": e2e["d2h"]},
        "gpu_launches": b.launches * args.steps,
        "gpu_launches_note": "kernels of this library per call x steps; memset nodes are not counted",
        "clocks": res["clocks"],
        "kernel_us_mean": head["kernel_us_mean"],
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(b)
    if not args.no_secondary:
        sec = []
        for nm, ac, mm in SECONDARY:
            bb = LinearBench(W.WORKLOADS[nm], mm) if nm == "linear" else Bench(W.WORKLOADS[nm].with_act(ac), mm)
            r = bb.run(min(args.steps, 10), 3, barrier)
            sec.append(summarize(bb, r, peaks))
            del bb
            torch.cuda.empty_cache()
        line["secondary"] = sec
    if not args.no_crossover:
        cross = []
        for nm, ac, mm, pth in CROSSOVER:
            path = {"decode": b4.PATH_DECODE, "grouped": b4.PATH_GROUPED}[pth]
            bb = Bench(W.WORKLOADS[nm].with_act(ac), mm, path=path)
            r = bb.run(min(args.steps, 10), 3, barrier)
            sm_ = summarize(bb, r, peaks)
            cross.append({"m": mm, "path": pth, "us_per_call": sm_["us_per_call"],
                          "us_per_call_single": sm_["us_per_call_single"],
                          "weight_stream_TBps": sm_["weight_stream_TBps"]})
            del bb
            torch.cuda.empty_cache()
        line["crossover"] = {"workload": describe(W.WORKLOADS["decode"].with_act("relu2"), 0).replace(" m=0", ""),
                             "lines": cross}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
