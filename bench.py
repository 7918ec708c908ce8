#!/usr/bin/env python3
"""Throughput benchmark of the fake-quant hot path on GB300.

One step runs every operation of the path once, each on its own synthetic
workload at full size (all resident in HBM):

  w1  per-tensor symmetric int8 fake quant + STE backward, fp32 [1,048,576]
  w2  per-row affine int8 and per-row symmetric int4 fake quant, fp32 [4096, 4096]
  w3  per-tensor amax-scaled FP8 fake quant, E4M3 and E5M2, bf16 [8192, 8192]
  w4  per-group (128) symmetric int4 fake quant + STE backward, bf16 [14336, 4096]
  w5  two-level 4-bit quantize + dequantize round trip, fp32 [268,435,456]

The metric is algorithmic bytes moved per second (each input read once per
dependent pass, each output written once; per-tensor calibration of a tensor
larger than on-chip storage needs two reads of x), i.e. GB/s, with Gelem/s and the fraction of the measured HBM
copy bandwidth beside it.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs the same suite on its own GPU (the
path shards into independent units, so there is no data-path collective);
value = bytes of all ranks / max time over ranks.  --impl reference times
the CPU oracle on a bounded sample of the same workloads (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fake-quant fwd+STE-bwd GB/s and Gelem/s per format, % of GB300 HBM peak"
WORKLOAD = ("qat fake-quant suite: w1 int8 per-tensor fwd+STE fp32[1048576]; "
            "w2 per-row affine-int8 + sym-int4 fp32[4096x4096]; "
            "w3 fp8 e4m3+e5m2 per-tensor amax bf16[8192x8192]; "
            "w4 per-group-128 sym-int4 fwd+STE bf16[14336x4096]; "
            "w5 QLoRA double-quant round trip fp32[268435456]")
FALLBACK_HBM_GBS = 6800.0


# ---------------------------------------------------------------------------
# algorithmic bytes (per element unless stated)
# ---------------------------------------------------------------------------
def workload_bytes(n1=1 << 20, r2=4096, c2=4096, n3=8192 * 8192, r4=14336, c4=4096,
                   n5=268_435_456):
    """(name, elements, algorithmic bytes, launches) of every call of one step.

    Per element: per-tensor calibration of a tensor larger than on-chip
    storage reads x twice (statistics, then the map: w3); a tensor that fits
    in the registers of the resident blocks (w1, 4 MiB) is read once, its
    statistics and map in one launch; y has the dtype of x; masks are 1 bit; int8 codes 1 byte, int4 codes
    half a byte; per-unit scales (and zero points) 4 bytes each; the 4-bit
    format stores half a byte per element, one byte per 64-element block and
    4 bytes per 256 blocks."""
    n2, n4 = r2 * c2, r4 * c4
    nb5 = (n5 + 63) // 64
    ns5 = (nb5 + 255) // 256
    m = lambda n: (n + 31) // 32 * 4  # noqa: E731
    return [
        ("w1_int8_tensor_fwd", n1, n1 * (4 + 4) + m(n1) + 4, 1),
        ("w1_ste_bwd", n1, n1 * (4 + 4) + m(n1), 1),
        ("w2_affine_int8_row", n2, n2 * (4 + 1 + 4) + m(n2) + r2 * 8, 1),
        ("w2_sym_int4_row", n2, n2 * 4 + (n2 + 1) // 2 + n2 * 4 + m(n2) + r2 * 4, 1),
        ("w3_fp8_e4m3_tensor", n3, n3 * (2 + 2 + 2) + m(n3) + 4, 2),
        ("w3_fp8_e5m2_tensor", n3, n3 * (2 + 2 + 2) + m(n3) + 4, 2),
        ("w4_int4_group_fwd", n4, n4 * 2 + (n4 + 1) // 2 + n4 * 2 + m(n4) + (n4 // 128) * 4, 1),
        ("w4_ste_bwd", n4, n4 * (2 + 2) + m(n4), 1),
        ("w5_quant4_double", n5, n5 * 4 + (n5 + 1) // 2 + nb5 + ns5 * 4, 1),
        ("w5_dequant4_double", n5, (n5 + 1) // 2 + nb5 + ns5 * 4 + n5 * 4, 1),
    ]


# ---------------------------------------------------------------------------
# distributed helpers (torchrun), kept free of CUDA so they run on gloo
# ---------------------------------------------------------------------------
def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def reduce_max_sum(seconds: float, units: float):
    """(max seconds over ranks, sum of units over ranks); identity without a process group."""
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()):
        return seconds, units
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([seconds], dtype=torch.float64, device=dev)
    u = torch.tensor([units], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def barrier():
    import torch.distributed as dist

    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.rows = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.index), "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [c.strip() for c in line.split(",")]))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float):
        def parse(rows):
            sm, mx, reasons = [], [], set()
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            for _, r in rows:
                try:
                    sm.append(float(r[2]))
                    mx.append(float(r[3]))
                except (ValueError, IndexError):
                    continue
                for k, name in enumerate(names):
                    if len(r) > 6 + k and r[6 + k].lower().startswith("active"):
                        reasons.add(name)
            return sm, mx, reasons

        inside = [r for r in self.rows if t0 <= r[0] <= t1]
        window = "timed"
        if len(inside) < 3:
            inside, window = self.rows, "run"
        sm, mx, reasons = parse(inside)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "window": "unavailable"}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(mx)),
                "reasons": sorted(reasons), "samples": len(sm), "window": window}


# ---------------------------------------------------------------------------
# the GPU suite
# ---------------------------------------------------------------------------
class Suite:
    """All workloads resident on one GPU, outputs preallocated; step() issues
    every call of the path once through the C ABI binding."""

    def __init__(self, dev, fq, inputs):
        self.fq = fq
        f = torch.float32
        x1, g1, w2, a3, w4, g4, x5 = inputs
        self.inputs = [t.to(dev) for t in inputs]
        self.x1, self.g1, self.w2, self.a3, self.w4, self.g4, self.x5 = self.inputs
        e = lambda n, dt=torch.uint8: torch.empty(n, dtype=dt, device=dev)  # noqa: E731
        n1, n2, n3, n4, n5 = x1.numel(), w2.numel(), a3.numel(), w4.numel(), x5.numel()
        self.r2, self.c2 = w2.shape
        self.r4, self.c4 = w4.shape
        r2 = self.r2
        self.ws = e(16 * 1024 * 2)
        self.flags = torch.zeros(1, dtype=torch.int32, device=dev)
        self.o = dict(
            s1=e(1, f), y1=e(n1, f), m1=e((n1 + 31) // 32, torch.int32), dx1=e(n1, f),
            s2a=e(r2, f), z2a=e(r2, torch.int32), y2a=e(n2, f), c2a=e(n2, torch.int8),
            m2a=e(n2 // 32, torch.int32),
            s2b=e(r2, f), y2b=e(n2, f), c2b=e(n2 // 2), m2b=e(n2 // 32, torch.int32),
            s3=e(2, f), y3a=e(n3, torch.bfloat16), m3a=e(n3 // 32, torch.int32),
            y3b=e(n3, torch.bfloat16), m3b=e(n3 // 32, torch.int32),
            s4=e(n4 // 128, f), y4=e(n4, torch.bfloat16), c4=e(n4 // 2), m4=e(n4 // 32, torch.int32),
            dx4=e(n4, torch.bfloat16),
            d5=e(n5 // 2), q5=e((n5 + 63) // 64), u5=e(((n5 + 63) // 64 + 255) // 256, f),
            y5=e(n5, f),
        )
        self.n = (n1, n2, n3, n4, n5)

    def calls(self):
        fq, o, ws, fl = self.fq, self.o, self.ws, self.flags
        n1, n2, n3, n4, n5 = self.n
        r2, c2, r4, c4 = self.r2, self.c2, self.r4, self.c4
        return [
            lambda: fq.qat_fake_quant_int(self.x1, 1, n1, 8, 0, 0, 0, False, o["s1"], None, o["y1"],
                                          None, o["m1"], fl, ws),
            lambda: fq.qat_ste_backward(self.g1, n1, o["m1"], o["dx1"]),
            lambda: fq.qat_fake_quant_int(self.w2, r2, c2, 8, 1, 1, 0, False, o["s2a"], o["z2a"],
                                          o["y2a"], o["c2a"], o["m2a"], fl, ws),
            lambda: fq.qat_fake_quant_int(self.w2, r2, c2, 4, 0, 1, 0, False, o["s2b"], None,
                                          o["y2b"], o["c2b"], o["m2b"], fl, ws),
            lambda: fq.qat_fake_quant_fp8(self.a3, n3, 0, False, o["s3"][0:1], o["y3a"], None,
                                          o["m3a"], fl, ws),
            lambda: fq.qat_fake_quant_fp8(self.a3, n3, 1, False, o["s3"][1:2], o["y3b"], None,
                                          o["m3b"], fl, ws),
            lambda: fq.qat_fake_quant_int(self.w4, r4, c4, 4, 0, 2, 128, False, o["s4"], None,
                                          o["y4"], o["c4"], o["m4"], fl, ws),
            lambda: fq.qat_ste_backward(self.g4, n4, o["m4"], o["dx4"]),
            lambda: fq.qat_quant4_double(self.x5, n5, o["d5"], o["q5"], o["u5"], None),
            lambda: fq.qat_dequant4_double(o["d5"], o["q5"], o["u5"], n5, o["y5"]),
        ]

    def outputs_for_host(self):
        o = self.o
        return [o[k] for k in ("y1", "m1", "dx1", "s1", "s2a", "z2a", "y2a", "c2a", "m2a", "s2b", "y2b",
                               "c2b", "m2b", "s3", "y3a", "m3a", "y3b", "m3b", "s4", "y4", "c4", "m4",
                               "dx4", "d5", "q5", "u5", "y5")]


class L2Flush:
    """Between timed calls: write 256 MiB (twice the L2), then read another
    256 MiB, so that L2 holds only clean lines of unrelated data and the timed
    call pays neither for cached inputs nor for writing back the flush."""

    def __init__(self, dev):
        self.w = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        self.r = torch.ones(64 << 20, dtype=torch.float32, device=dev)

    def __call__(self):
        self.w.zero_()
        self.r.sum()


def isolated_call_ms(calls, stream, iters=30, warm=3):
    """Each call of the step alone: an L2 flush (L2Flush) before every timed
    iteration, CUDA events around the call on its stream; the mean in ms.
    Back to back, a call also pays for writing back the dirty L2 lines that
    the call before it left (w2 follows the 1 GiB written by w5's dequant);
    alone, it pays only for its own traffic."""
    flush = L2Flush(torch.device("cuda", torch.cuda.current_device()))
    out = []
    for c in calls:
        for _ in range(warm):
            flush()
            c()
        ev = []
        for _ in range(iters):
            flush()
            a = torch.cuda.Event(enable_timing=True)
            z = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            c()
            z.record(stream)
            ev.append((a, z))
        torch.cuda.synchronize()
        out.append(sum(a.elapsed_time(z) for a, z in ev) / iters)
    del flush
    return out


def run_next_rows(args, suite, wb, peak, only=None):
    """Rows past the headline path, timed like it (CUDA events per call on the
    launching stream, after warm-up) but reported outside `value`:
    - stochastic rounding (the *_sr entry points) of the w2, w3 and w4 maps,
      same inputs, outputs and algorithmic bytes as their nearest-rounding
      calls (only: name prefixes, profiling runs of these rows alone);
    - config 1 (w1 int8 per-tensor fwd + STE) replayed as one CUDA graph
      against the same two calls issued directly, with an L2 flush (L2Flush)
      before every timed iteration."""
    fq, o, ws, fl = suite.fq, suite.o, suite.ws, suite.flags
    n1, n2, n3, n4, n5 = suite.n
    r2, c2, r4, c4 = suite.r2, suite.c2, suite.r4, suite.c4
    seed = 0x5EED
    bytes_of = {name: b for name, _, b, _ in wb}
    sr = [
        ("w2_affine_int8_row_sr", "w2_affine_int8_row",
         lambda: fq.qat_fake_quant_int_sr(suite.w2, r2, c2, 8, 1, 1, 0, False, o["s2a"], o["z2a"],
                                          seed, 0, o["y2a"], o["c2a"], o["m2a"], fl, ws)),
        ("w2_sym_int4_row_sr", "w2_sym_int4_row",
         lambda: fq.qat_fake_quant_int_sr(suite.w2, r2, c2, 4, 0, 1, 0, False, o["s2b"], None, seed,
                                          0, o["y2b"], o["c2b"], o["m2b"], fl, ws)),
        ("w3_fp8_e4m3_tensor_sr", "w3_fp8_e4m3_tensor",
         lambda: fq.qat_fake_quant_fp8_sr(suite.a3, n3, 0, False, o["s3"][0:1], seed, 0, o["y3a"],
                                          None, o["m3a"], fl, ws)),
        ("w4_int4_group_fwd_sr", "w4_int4_group_fwd",
         lambda: fq.qat_fake_quant_int_sr(suite.w4, r4, c4, 4, 0, 2, 128, False, o["s4"], None,
                                          seed, 0, o["y4"], o["c4"], o["m4"], fl, ws)),
    ]
    if only:
        sr = [r for r in sr if any(r[0].startswith(p) for p in only)]
    stream = torch.cuda.current_stream()
    steps = max(3, min(args.steps, 200))
    for _ in range(3):
        for _, _, c in sr:
            c()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(sr) + 1)] for _ in range(steps)]
    torch.cuda.synchronize()
    for k in range(steps):
        for i, (_, _, c) in enumerate(sr):
            ev[k][i].record(stream)
            c()
        ev[k][len(sr)].record(stream)
    torch.cuda.synchronize()
    out = {}
    for i, (name, base, _) in enumerate(sr):
        ms = sum(ev[k][i].elapsed_time(ev[k][i + 1]) for k in range(steps)) / steps
        b = bytes_of[base]
        out[name] = {"us": round(ms * 1e3, 2), "GB_s": round(b / (ms * 1e-3) / 1e9, 1),
                     "frac_of_measured_hbm": round(b / (ms * 1e-3) / 1e9 / peak, 4),
                     "bytes": b, "launches": 2 if base.startswith("w3") else 1}
    if only:
        res = {"stochastic_rounding": out} if out else {}
        cols = run_column_rows(args, suite, peak, only)
        if cols:
            res["per_column"] = cols
        return res

    # config 1: direct calls and one CUDA graph of the same calls
    calls = suite.calls()[:2]
    b1 = bytes_of["w1_int8_tensor_fwd"] + bytes_of["w1_ste_bwd"]
    flush = L2Flush(suite.x1.device)
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        for _ in range(3):
            for c in calls:
                c()
    stream.wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for c in calls:
            c()

    def timed(run):
        t = []
        for _ in range(3):
            run()
        for _ in range(steps):
            flush()
            a = torch.cuda.Event(enable_timing=True)
            z = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            run()
            z.record(stream)
            t.append((a, z))
        torch.cuda.synchronize()
        return sum(a.elapsed_time(z) for a, z in t) / len(t)

    direct_ms = timed(lambda: [c() for c in calls])
    graph_ms = timed(g.replay)
    w1 = {}
    for key, ms in (("direct", direct_ms), ("cuda_graph", graph_ms)):
        w1[key] = {"us": round(ms * 1e3, 2), "GB_s": round(b1 / (ms * 1e-3) / 1e9, 1),
                   "frac_of_measured_hbm": round(b1 / (ms * 1e-3) / 1e9 / peak, 4)}
    w1["bytes"] = b1
    w1["l2"] = "256 MiB write then 256 MiB read before every timed iteration"
    del flush
    return {"stochastic_rounding": out, "w1_int8_tensor_fwd_ste": w1,
            "qat_optimizer_step": run_optimizer_rows(args, suite, peak),
            "per_column": run_column_rows(args, suite, peak),
            "calibration_options": run_calib_option_rows(args, suite, wb, peak),
            "block_formats": run_block_rows(args, suite, peak)}


def run_block_rows(args, suite, peak):
    """Block-scaled floating-point fake quant of the w4 weights bf16[14336,
    4096] (an L2 flush before every call): NVFP4 (E2M1 elements, blocks of 16,
    E4M3 scales under the FP32 tensor scale: a statistics pass, then the map),
    MXFP4 (E2M1, 32, E8M0) and MXFP8 (E4M3, 32, E8M0).  Algorithmic bytes per
    element: x read (2; twice for NVFP4), y written (2), the element code (1/2
    or 1), the block scale (1/16 or 1/32), the mask (1/8)."""
    fq, fl = suite.fq, suite.flags
    r4, c4 = suite.r4, suite.c4
    n = r4 * c4
    dev = suite.x1.device
    o = suite.o
    m = (n + 31) // 32 * 4
    ws = torch.empty(fq.qat_workspace_bytes(1, n, 0, 0), dtype=torch.uint8, device=dev)
    codes = torch.empty(n, dtype=torch.uint8, device=dev)
    bs = torch.empty(n // 16, dtype=torch.uint8, device=dev)
    g = torch.empty(1, dtype=torch.float32, device=dev)
    rows = [
        ("w4_nvfp4", n * (2 + 2 + 2) + n // 2 + n // 16 + m, 2, (4, 16, 1)),
        ("w4_mxfp4", n * (2 + 2) + n // 2 + n // 32 + m, 1, (4, 32, 0)),
        ("w4_mxfp8_e4m3", n * (2 + 2) + n + n // 32 + m, 1, (0, 32, 0)),
    ]
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream()
    steps = max(3, min(args.steps, 100))
    out = {}
    for name, b, launches, (fmt, block, kind) in rows:
        def call():
            fq.qat_fake_quant_block(suite.w4, n, fmt, block, kind, g, o["y4"], codes, bs,
                                    o["m4"], fl, ws)
        for _ in range(3):
            call()
        t = []
        for _ in range(steps):
            flush()
            a = torch.cuda.Event(enable_timing=True)
            z = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            call()
            z.record(stream)
            t.append((a, z))
        torch.cuda.synchronize()
        ms = sum(a.elapsed_time(z) for a, z in t) / len(t)
        out[name] = {"us": round(ms * 1e3, 2), "GB_s": round(b / (ms * 1e-3) / 1e9, 1),
                     "frac_of_measured_hbm": round(b / (ms * 1e-3) / 1e9 / peak, 4),
                     "bytes": b, "launches": launches}
    del flush
    return out


def run_calib_option_rows(args, suite, wb, peak):
    """Calibration options and percentile calibration, timed like the
    per-column rows (an L2 flush before every call):
    - w4 weights bf16[14336, 4096], symmetric int4 per group of 128 with the
      scales rounded to binary16 (same bytes as the w4 call);
    - w2 weights fp32[4096, 4096], symmetric int4 per row with the range
      clipped to 0.7 * absmax (same bytes as the w2 int4 call);
    - w2 weights, symmetric int8 per tensor calibrated by the nearest-rank
      quantiles at 0.001 / 0.999 (per_tensor_percentile); algorithmic bytes
      count x read twice (the selection, then the map), y, codes and mask
      written; the radix select reads x three times (five launches: a reset,
      three passes, the map)."""
    fq, o, fl = suite.fq, suite.o, suite.flags
    n1, n2, n3, n4, n5 = suite.n
    r2, c2, r4, c4 = suite.r2, suite.c2, suite.r4, suite.c4
    dev = suite.x1.device
    m = lambda n: (n + 31) // 32 * 4  # noqa: E731
    wsg = torch.empty(max(fq.qat_workspace_bytes(r4, c4, 2, 128), 16), dtype=torch.uint8,
                      device=dev)
    wsr = torch.empty(max(fq.qat_workspace_bytes(r2, c2, 1, 0), 16), dtype=torch.uint8, device=dev)
    wsp = torch.empty(fq.qat_percentile_workspace_bytes(), dtype=torch.uint8, device=dev)
    s1 = torch.empty(1, dtype=torch.float32, device=dev)
    c8 = torch.empty(n2, dtype=torch.int8, device=dev)
    bytes_of = {name: b for name, _, b, _ in wb}
    rows = [
        ("w4_int4_group_fp16_scales", bytes_of["w4_int4_group_fwd"],
         lambda: fq.qat_fake_quant_int_opts(suite.w4, r4, c4, 4, 0, 2, 128,
                                            fq.calib_options(1.0, True), False, 0, 0, o["s4"],
                                            None, o["y4"], o["c4"], o["m4"], fl, wsg)),
        ("w2_sym_int4_row_clip0.7", bytes_of["w2_sym_int4_row"],
         lambda: fq.qat_fake_quant_int_opts(suite.w2, r2, c2, 4, 0, 1, 0, fq.calib_options(0.7),
                                            False, 0, 0, o["s2b"], None, o["y2b"], o["c2b"],
                                            o["m2b"], fl, wsr)),
        ("w2_sym_int8_tensor_percentile", n2 * (4 + 4 + 4 + 1) + m(n2) + 4,
         lambda: fq.qat_fake_quant_int_percentile(suite.w2, n2, 8, 0, 0.001, False, 0, 0, s1,
                                                  None, o["y2a"], c8, o["m2a"], fl, wsp)),
    ]
    launches = {"w4_int4_group_fp16_scales": 1, "w2_sym_int4_row_clip0.7": 1,
                "w2_sym_int8_tensor_percentile": 5}
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream()
    steps = max(3, min(args.steps, 100))
    out = {}
    for name, b, call in rows:
        for _ in range(3):
            call()
        t = []
        for _ in range(steps):
            flush()
            a = torch.cuda.Event(enable_timing=True)
            z = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            call()
            z.record(stream)
            t.append((a, z))
        torch.cuda.synchronize()
        ms = sum(a.elapsed_time(z) for a, z in t) / len(t)
        out[name] = {"us": round(ms * 1e3, 2), "GB_s": round(b / (ms * 1e-3) / 1e9, 1),
                     "frac_of_measured_hbm": round(b / (ms * 1e-3) / 1e9 / peak, 4),
                     "bytes": b, "launches": launches[name]}
    del flush
    return out


def run_column_rows(args, suite, peak, only=None):
    """Per-column (channel axis 1) calibrated fake quant: affine int8 and
    symmetric int4 of the w2 weights fp32[4096, 4096] (the per-row calls'
    shape, one scale per column instead of per row), the int8 affine call
    with stochastic rounding, and symmetric int8 per channel of activations
    bf16[8192, 8192] drawn like w3 but without its special values (channels
    = the last dimension).  The
    column statistics must see every row before the first element is mapped,
    so x is read twice (statistics, then the map), as for per-tensor
    calibration; algorithmic bytes count both reads.  An L2 flush (L2Flush)
    precedes every timed call (CUDA events on the launching stream).  only:
    name prefixes (profiling runs of some rows alone)."""
    fq, o, fl = suite.fq, suite.o, suite.flags
    r2, c2 = suite.r2, suite.c2
    dev = suite.x1.device
    n2, n3 = r2 * c2, suite.n[2]
    side3 = int(round(n3 ** 0.5))
    m = lambda n: (n + 31) // 32 * 4  # noqa: E731
    ws = torch.empty(max(fq.qat_workspace_bytes(r2, c2, 3, 0),
                         fq.qat_workspace_bytes(side3, side3, 3, 0)), dtype=torch.uint8,
                     device=dev)
    c3 = torch.empty(n3, dtype=torch.int8, device=dev)
    s3 = torch.empty(side3, dtype=torch.float32, device=dev)
    sc = torch.empty(c2, dtype=torch.float32, device=dev)  # one scale / zero point per column
    zc = torch.empty(c2, dtype=torch.int32, device=dev)
    rows = [
        ("w2_affine_int8_col", n2 * (4 + 4 + 4 + 1) + m(n2) + c2 * 8,
         lambda: fq.qat_fake_quant_int(suite.w2, r2, c2, 8, 1, 3, 0, False, sc, zc,
                                       o["y2a"], o["c2a"], o["m2a"], fl, ws)),
        ("w2_sym_int4_col", n2 * (4 + 4 + 4) + (n2 + 1) // 2 + m(n2) + c2 * 4,
         lambda: fq.qat_fake_quant_int(suite.w2, r2, c2, 4, 0, 3, 0, False, sc, None,
                                       o["y2b"], o["c2b"], o["m2b"], fl, ws)),
        ("w2_affine_int8_col_sr", n2 * (4 + 4 + 4 + 1) + m(n2) + c2 * 8,
         lambda: fq.qat_fake_quant_int_sr(suite.w2, r2, c2, 8, 1, 3, 0, False, sc, zc, 0x5EED,
                                          0, o["y2a"], o["c2a"], o["m2a"], fl, ws)),
    ]
    if side3 * side3 == n3:  # not on a reduced profiling workload that is not square
        # per-channel activations: the w3 recipe (t(3) values, 1% outlier
        # channels) without its special values, which would poison almost
        # every channel with a NaN or Inf and leave it dead
        from fake_quant_numerics_gb300 import workloads as W

        a3c = W.cfg3(side3, side3, special_frac=0.0).to(dev)
        rows.append(
            ("w3_sym_int8_col_bf16", n3 * (2 + 2 + 2 + 1) + m(n3) + side3 * 4,
             lambda: fq.qat_fake_quant_int(a3c, side3, side3, 8, 0, 3, 0, False, s3, None,
                                           o["y3a"], c3, o["m3a"], fl, ws)))
    if only:
        rows = [r for r in rows if any(r[0].startswith(p) for p in only)]
        if not rows:
            return {}
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream()
    steps = max(3, min(args.steps, 100))
    out = {}
    for name, b, call in rows:
        for _ in range(3):
            call()
        t = []
        for _ in range(steps):
            flush()
            a = torch.cuda.Event(enable_timing=True)
            z = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            call()
            z.record(stream)
            t.append((a, z))
        torch.cuda.synchronize()
        ms = sum(a.elapsed_time(z) for a, z in t) / len(t)
        out[name] = {"us": round(ms * 1e3, 2), "GB_s": round(b / (ms * 1e-3) / 1e9, 1),
                     "frac_of_measured_hbm": round(b / (ms * 1e-3) / 1e9 / peak, 4),
                     "bytes": b, "launches": 3}
    del flush
    return out


def run_optimizer_rows(args, suite, peak, n=1 << 26):
    """The QAT optimizer step (AdamW update of an fp32 master with its moments,
    then the per-tensor int8 view with its mask, or the FP8 view) on a synthetic
    64M-parameter master (N(0, 0.02), gradients N(0, 1e-3), seeded on the
    device): 256 MB per array, so no array stays in L2.  Algorithmic bytes per
    element: update 16 read + 12 written, view 4 read + 4 written + 1/8 mask."""
    fq = suite.fq
    dev = suite.x1.device
    gen = torch.Generator(device=dev)
    gen.manual_seed(5)
    w = torch.randn(n, generator=gen, device=dev) * 0.02
    g = torch.randn(n, generator=gen, device=dev) * 0.001
    m = torch.zeros(n, device=dev)
    v = torch.zeros(n, device=dev)
    view = torch.empty(n, device=dev)
    mask = torch.empty((n + 31) // 32, dtype=torch.int32, device=dev)
    scale = torch.empty(1, device=dev)
    zp = torch.empty(1, dtype=torch.int32, device=dev)
    flags = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = torch.empty(fq.qat_workspace_bytes(1, n, 0, 0), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    steps = max(3, min(args.steps, 100))
    b = int(n * (28 + 8) + (n + 31) // 32 * 4)
    res = {"elements": n, "bytes": b, "launches": 2}
    for name, bits_, sr in (("int8_view", 8, False), ("int8_view_sr", 8, True), ("e4m3_view", 0, False)):
        t = 0
        def step():
            nonlocal t
            t += 1
            hp = fq.adam_hparams(1e-3, 0.9, 0.999, 1e-8, 0.01, t)
            fq.qat_optimizer_step(w, g, m, v, n, hp, bits_, "symmetric", "e4m3", sr, 7, t * n,
                                  view, None, mask, scale, zp, flags, ws)
        for _ in range(3):
            step()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        torch.cuda.synchronize()
        for a, z in ev:
            a.record(stream)
            step()
            z.record(stream)
        torch.cuda.synchronize()
        ms = sum(a.elapsed_time(z) for a, z in ev) / steps
        res[name] = {"us": round(ms * 1e3, 1), "GB_s": round(b / (ms * 1e-3) / 1e9, 1),
                     "frac_of_measured_hbm": round(b / (ms * 1e-3) / 1e9 / peak, 4)}
    return res


def make_inputs(frac: float = 1.0):
    """Inputs of the five workloads; frac < 1 keeps that fraction of the rows
    (elements) of each, with the same distributions (profiling runs only)."""
    if frac >= 1.0:
        from fake_quant_numerics_gb300 import workloads as W

        x1, g1 = W.cfg1()
        w2 = W.cfg2()
        a3 = W.cfg3()
        w4, g4 = W.cfg4()
        x5 = W.cfg5()
        return [x1, g1, w2, a3, w4, g4, x5]
    return list(oracle_sample(frac))


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def source_key(source: str) -> str:
    """sha256[:16] of a kernel's source file followed by the shared device
    header it includes (the key under which profiles/traffic.txt records it)."""
    h = hashlib.sha256()
    for f in (source, "qat_device.cuh"):
        with open(os.path.join(ROOT, "fake_quant_numerics_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, source: str):
    """DRAM bytes per launch of `kernel` at full size from the committed ncu
    summary, or None when the kernel's sources changed since the capture."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    try:
        key = source_key(source)
        with open(path) as f:
            for line in f:
                parts = line.split()
                if len(parts) >= 3 and parts[0] == kernel and parts[1] == key:
                    return float(parts[2])
    except OSError:
        pass
    return None


KERNEL_OF_CALL = {
    "w5_quant4_double": ("k_q4_quant", "kernels_misc.cu"),
    "w5_dequant4_double": ("k_q4_dequant", "kernels_misc.cu"),
    "w4_int4_group_fwd": ("k_int_groups", "kernels_fused.cu"),
    "w4_ste_bwd": ("k_ste", "kernels_misc.cu"),
    "w2_affine_int8_row": ("k_int_rows", "kernels_fused.cu"),
    "w2_sym_int4_row": ("k_int_rows", "kernels_fused.cu"),
    "w1_ste_bwd": ("k_ste", "kernels_misc.cu"),
}


def run_ours(args, rank, world, local):
    import fake_quant_numerics_gb300 as fq

    fq.load()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    inputs = make_inputs(args.fraction)
    suite = Suite(dev, fq, inputs)
    calls = suite.calls()
    n1, n2, n3, n4, n5 = suite.n
    wb = workload_bytes(n1, suite.r2, suite.c2, n3, suite.r4, suite.c4, n5)
    wb_all = list(wb)
    if args.only:
        keep = [i for i, w in enumerate(wb) if any(w[0].startswith(p) for p in args.only.split(","))]
        calls = [calls[i] for i in keep]
        wb = [wb[i] for i in keep]
    step_bytes = sum(b for _, _, b, _ in wb)
    step_elems = sum(e for _, e, _, _ in wb)
    stream = torch.cuda.current_stream()

    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    for _ in range(args.warmup):
        for c in calls:
            c()
    torch.cuda.synchronize()

    # timed region: K steps, events around every call (same stream)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(calls) + 1)]
          for _ in range(args.steps)]
    l0 = fq.qat_kernel_launch_count()
    barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for k in range(args.steps):
        ev[k][0].record(stream)
        for i, c in enumerate(calls):
            c()
            ev[k][i + 1].record(stream)
    end.record(stream)
    torch.cuda.synchronize()
    barrier()
    t_wall1 = time.time()
    launches = fq.qat_kernel_launch_count() - l0
    local_s = start.elapsed_time(end) / 1e3
    max_s, total_bytes = reduce_max_sum(local_s, step_bytes * args.steps)
    _, total_elems = reduce_max_sum(local_s, step_elems * args.steps)
    per_call_ms = np.array([[ev[k][i].elapsed_time(ev[k][i + 1]) for i in range(len(calls))]
                            for k in range(args.steps)])
    mean_ms = per_call_ms.mean(axis=0)
    sampler.stop()
    clocks = sampler.summary(t_wall0, t_wall1)

    # end to end through the public API with host buffers (pinned), copies timed
    e2e = run_e2e(args, suite, calls, step_bytes)

    peak, peak_kind = measured_peak()
    next_rows = None
    # profiling runs: --only names of stochastic-rounding or per-column rows
    row_only = ([p for p in args.only.split(",") if p.endswith("_sr") or "_col" in p]
                if args.only else [])
    if not args.only and args.fraction >= 1.0 and not args.no_next:
        next_rows = run_next_rows(args, suite, wb, peak)
    elif row_only:
        next_rows = run_next_rows(args, suite, wb_all, peak, only=row_only)
    iso_ms = isolated_call_ms(calls, stream) if not args.no_isolated else None
    per_wl = {}
    for i, ((name, elems, b, nl), ms) in enumerate(zip(wb, mean_ms)):
        per_wl[name] = {"ms": round(float(ms), 5), "GB_s": round(b / (ms * 1e-3) / 1e9, 1),
                        "Gelem_s": round(elems / (ms * 1e-3) / 1e9, 2),
                        "frac_of_measured_hbm": round(b / (ms * 1e-3) / 1e9 / peak, 4),
                        "launches": nl, "bytes": b}
        if iso_ms is not None:
            per_wl[name]["isolated_ms"] = round(float(iso_ms[i]), 5)
            per_wl[name]["isolated_frac_of_measured_hbm"] = round(
                b / (iso_ms[i] * 1e-3) / 1e9 / peak, 4)
    # dominant kernel: the single-launch call with the largest time (a subset
    # run of multi-launch calls only reports its longest call)
    single = [i for i, w in enumerate(wb) if w[3] == 1] or list(range(len(wb)))
    dom = max(single, key=lambda i: mean_ms[i])
    dname, _, dbytes, _ = wb[dom]
    achieved = dbytes / (mean_ms[dom] * 1e-3) / 1e9
    kern, src = KERNEL_OF_CALL.get(dname, (dname, ""))
    traffic = recorded_traffic(kern, src) if src else None
    value = total_bytes / max_s / 1e9
    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(max_s / args.steps * 1e3, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32/bf16 in, fp32 arithmetic",
        "data": "synthetic (seeded numpy generators, distributions of the five workloads)",
        "config": {"workload": WORKLOAD, "parallelism": f"replicas x{world} (independent units)",
                   "l2": "inputs larger than L2: a step streams ~4.1 GB, every input is evicted "
                         "before it is read again",
                   "Gelem_s": round(total_elems / max_s / 1e9, 2),
                   "frac_of_measured_hbm": round(value / peak, 4),
                   "frac_of_nominal_8TBs": round(value / 8000.0, 4),
                   "per_workload": per_wl},
        "gpu_launches": int(launches),
        "clocks": clocks,
        "e2e": e2e,
        "roofline": {"bound": "hbm", "kernel": kern, "call": dname,
                     "achieved": round(achieved, 1), "peak": peak, "peak_kind": peak_kind,
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": traffic, "algorithmic_bytes": dbytes},
    }
    if next_rows is not None:
        line["next_rows"] = next_rows
    if args.fraction < 1.0 or args.only:
        line["config"]["subset"] = {"only": args.only, "fraction": args.fraction}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(inputs, args.cpu_passes)
    # last key, compact, so that the per-format figures stay in the end of the
    # line: per call of the step, back to back (us, GB/s, Gelem/s, fraction of
    # the measured HBM bandwidth) and alone after an L2 flush (iso_us, iso_f)
    line["per_call"] = compact_per_call(per_wl)
    return line


def compact_per_call(per_wl):
    out = {}
    for name, r in per_wl.items():
        c = {"us": round(r["ms"] * 1e3, 1), "GBs": round(r["GB_s"]), "Gel": round(r["Gelem_s"], 1),
             "f": round(r["frac_of_measured_hbm"], 3)}
        if "isolated_ms" in r:
            c["iso_us"] = round(r["isolated_ms"] * 1e3, 1)
            c["iso_f"] = round(r["isolated_frac_of_measured_hbm"], 3)
        out[name] = c
    return out


def host_link_gbs(dev, nbytes=256 << 20, reps=3):
    """Pinned host <-> device copy bandwidth of this machine (GB/s), timed with
    CUDA events after one warm-up copy: host to device alone, device to host
    alone, and both at once on two streams (their bytes summed)."""
    h_in = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    h_out = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    d_in = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    d_out = torch.zeros(nbytes, dtype=torch.uint8, device=dev)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    out = {}
    for name in ("h2d", "d2h", "both"):
        best = None
        for _ in range(reps + 1):
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            s1.wait_event(e0)
            s2.wait_event(e0)
            if name in ("h2d", "both"):
                with torch.cuda.stream(s1):
                    d_in.copy_(h_in, non_blocking=True)
            if name in ("d2h", "both"):
                with torch.cuda.stream(s2):
                    h_out.copy_(d_out, non_blocking=True)
            torch.cuda.current_stream().wait_stream(s1)
            torch.cuda.current_stream().wait_stream(s2)
            e1.record()
            torch.cuda.synchronize()
            t = e0.elapsed_time(e1) / 1e3
            best = t if best is None else min(best, t)
        out[name] = round((2 if name == "both" else 1) * nbytes / best / 1e9, 1)
    return out


def run_e2e(args, suite, calls, step_bytes, keep=None):
    """The same step with host inputs: pinned H2D copies of every input, the
    calls, and D2H copies of every output, all inside the timed region; five
    windows of k steps, the median window's rate reported.

    Two device buffer sets and three streams (copies in, calls, copies out)
    pipeline the steps: step k's inputs come in while step k - 1 computes and
    step k - 2's outputs go out, so the two directions of the host link run
    at once.  Step k's copies into a set wait for the calls of step k - 2 on
    that set, its calls wait for its inputs and for the copy-out of step
    k - 2 from the set's outputs; every step still moves all its inputs in
    and all its outputs out.  `keep` receives the host outputs of the last
    step (a test compares them with the direct calls)."""
    dev = suite.x1.device
    if not args.only:
        calls = suite.calls()
    sets = [(suite, calls)]
    other = Suite(dev, suite.fq, [t.cpu() for t in suite.inputs])
    sets.append((other, other.calls() if not args.only else [other.calls()[i] for i in
                                                              _subset(args, suite)]))
    host_in = [t.cpu().pin_memory() for t in suite.inputs]
    host_out = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in suite.outputs_for_host()]
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = sum(t.numel() * t.element_size() for t in host_out)
    k = max(2, min(args.steps, args.e2e_steps))
    s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    in_done = [torch.cuda.Event() for _ in range(2)]
    cmp_done = [torch.cuda.Event() for _ in range(2)]
    out_done = [torch.cuda.Event() for _ in range(2)]

    def step(i):
        b = i % 2
        S, cs = sets[b]
        if i >= 2:
            s_in.wait_event(cmp_done[b])  # the calls of step i - 2 have read this set
        with torch.cuda.stream(s_in):
            for d, h in zip(S.inputs, host_in):
                d.copy_(h, non_blocking=True)
            in_done[b].record(s_in)
        s_cmp.wait_event(in_done[b])
        if i >= 2:
            s_cmp.wait_event(out_done[b])  # step i - 2's outputs have left this set
        with torch.cuda.stream(s_cmp):
            for c in cs:
                c()
            cmp_done[b].record(s_cmp)
        s_out.wait_event(cmp_done[b])
        with torch.cuda.stream(s_out):
            for h, d in zip(host_out, S.outputs_for_host()):
                h.copy_(d, non_blocking=True)
            out_done[b].record(s_out)

    step(0)
    step(1)
    torch.cuda.synchronize()
    # five timed windows of k steps each, the median reported: the host link
    # is shared with the machine's other jobs, and a window now and then runs
    # at 55-65% of the others
    runs = []
    for _ in range(5):
        barrier()
        t0 = time.perf_counter()
        for i in range(k):
            step(i)
        torch.cuda.synchronize()
        t1 = time.perf_counter()
        secs, tot = reduce_max_sum(t1 - t0, step_bytes * k)
        runs.append(tot / secs / 1e9)
    if keep is not None:
        keep["host_out"] = host_out
    del other
    # the host link bounds this figure: a step's copies take at least the
    # longer of its two directions alone and its total at the rate of both
    # (each rank measures its own link; the bounds are summed over the ranks,
    # as the value is)
    link = host_link_gbs(dev)
    t_copy = max(h2d / (link["h2d"] * 1e9), d2h / (link["d2h"] * 1e9),
                 (h2d + d2h) / (link["both"] * 1e9))
    value = sorted(runs)[len(runs) // 2]
    _, bound = reduce_max_sum(0.0, step_bytes / t_copy / 1e9)
    return {"value": round(value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": k, "windows": [round(r, 1) for r in runs],
            "pipeline": "2 device buffer sets; copies in, calls, copies out on 3 streams",
            "host_link_gbs": link, "link_bound": round(bound, 1),
            "frac_of_link_bound": round(value / bound, 3)}


def _subset(args, suite):
    n1, n2, n3, n4, n5 = suite.n
    wb = workload_bytes(n1, suite.r2, suite.c2, n3, suite.r4, suite.c4, n5)
    return [i for i, w in enumerate(wb) if any(w[0].startswith(p) for p in args.only.split(","))]


# ---------------------------------------------------------------------------
# CPU oracle arm
# ---------------------------------------------------------------------------
def oracle_sample(frac: float):
    """Inputs of every workload at a fraction of its rows (same distributions)."""
    from fake_quant_numerics_gb300 import workloads as W

    def rows(r):
        return max(1, int(round(r * frac)))

    n1 = max(1024, int((1 << 20) * frac))
    x1, g1 = W.cfg1(n=n1)
    w2 = W.cfg2(rows=rows(4096))
    a3 = W.cfg3(rows=rows(8192))
    w4, g4 = W.cfg4(rows=rows(14336))
    n5 = max(16384, int(268_435_456 * frac) // 16384 * 16384)
    x5 = W.cfg5(n=n5)
    return x1, g1, w2, a3, w4, g4, x5


def oracle_step(inputs):
    """One pass of the path through the oracle; returns (seconds, bytes, elems)."""
    import oracle
    from fake_quant_numerics_gb300 import workloads as W

    x1, g1, w2, a3, w4, g4, x5 = inputs
    x1n, g1n, w2n, x5n = x1.numpy(), g1.numpy(), w2.numpy(), x5.numpy()
    a3b, w4b, g4b = W.bf16_bits(a3), W.bf16_bits(w4), W.bf16_bits(g4)
    n1, n2, n3, n4, n5 = x1n.size, w2n.size, a3b.size, w4b.size, x5n.size
    r2, r4 = w2.shape[0], w4.shape[0]
    t0 = time.perf_counter()
    o1 = oracle.fake_quant_int(x1n, 1, n1, 8, 0, 0, want_codes=False)
    oracle.ste_backward(g1n, o1["mask"])
    oracle.fake_quant_int(w2n, r2, 4096, 8, 1, 1)
    oracle.fake_quant_int(w2n, r2, 4096, 4, 0, 1)
    oracle.fake_quant_fp8(a3b, 0, want_codes=False)
    oracle.fake_quant_fp8(a3b, 1, want_codes=False)
    o4 = oracle.fake_quant_int(w4b, r4, 4096, 4, 0, 2, 128)
    oracle.ste_backward(g4b, o4["mask"])
    q = oracle.quant4_double(x5n)
    oracle.dequant4_double(q["data"], q["qscales"], q["super_scales"], n5)
    secs = time.perf_counter() - t0
    wb = workload_bytes(n1, r2, 4096, n3, r4, 4096, n5)
    return secs, sum(b for _, _, b, _ in wb), sum(e for _, e, _, _ in wb)


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def _spans(n: int, parts: int, align: int):
    """[start, stop) pieces of range(n), every start a multiple of `align`."""
    per = -(-n // max(1, parts))
    step = max(align, -(-per // align) * align)
    return [(a, min(n, a + step)) for a in range(0, n, step)]


def oracle_step_parallel(inputs, pool, cores: int, keep=None):
    """One pass of the path through the same oracle functions, split over the
    host's cores by threads (ctypes releases the interpreter lock during each C
    call).  Elementwise and per-unit calls run on pieces of whole mask words
    (rows, 32-element runs, 16384-element super-blocks); per-tensor calls take
    the statistics of every piece in parallel, combine them (a max), derive the
    scale as the oracle does, then map every piece with that scale as a given
    parameter, which gives the calibrated call's outputs.  Returns (seconds,
    bytes, elems); `keep` (a dict) receives the outputs."""
    import ctypes
    import math

    import oracle
    from fake_quant_numerics_gb300 import workloads as W

    L = oracle.lib()
    P = oracle._p
    x1, g1, w2, a3, w4, g4, x5 = inputs
    x1n, g1n, w2n, x5n = x1.numpy(), g1.numpy(), w2.numpy(), x5.numpy()
    a3b, w4b, g4b = W.bf16_bits(a3), W.bf16_bits(w4), W.bf16_bits(g4)
    n1, n2, n3, n4, n5 = x1n.size, w2n.size, a3b.size, w4b.size, x5n.size
    r2, c2, r4, c4 = w2.shape[0], w2.shape[1], w4.shape[0], w4.shape[1]

    def run(fn, spans):
        for f in [pool.submit(fn, a, b) for a, b in spans]:
            f.result()

    def absmax_of(x, dt, n):
        out = [0.0]

        def piece(a, b):
            mn, mx, am, nb = ctypes.c_float(), ctypes.c_float(), ctypes.c_float(), ctypes.c_int64()
            L.or_unit_stats(P(x), dt, a, b - a, ctypes.byref(mn), ctypes.byref(mx),
                            ctypes.byref(am), ctypes.byref(nb))
            return am.value
        futs = [pool.submit(piece, a, b) for a, b in _spans(n, cores, 1024)]
        for f in futs:
            out[0] = max(out[0], f.result())
        return np.float32(out[0])

    def int_rows(x, dt, rows, cols, bits, scheme, gran, group, y, codes, mask, sc, zp):
        def piece(a, b):
            e0, e1 = a * cols, b * cols
            cb = e0 if bits == 8 else e0 // 2
            u0 = a if gran == oracle.PER_ROW else e0 // group
            fl = ctypes.c_int32(0)
            L.or_fake_quant_int(P(x[e0:e1]), dt, b - a, cols, bits, scheme, gran, group, 0,
                                P(sc[u0:]), P(zp[u0:]), P(y[e0:e1]), P(codes[cb:]),
                                P(mask[e0 // 32:]), ctypes.byref(fl), 1)
        run(piece, _spans(rows, cores, 32 // math.gcd(cols, 32)))  # whole mask words
        if keep is not None:
            keep.setdefault("rows", []).append((y, codes, mask, sc, zp))

    def ste(g, dt, n, mask, dx):
        def piece(a, b):
            L.or_ste_backward(P(g[a:b]), dt, b - a, P(mask[a // 32:]), P(dx[a:b]))
        run(piece, _spans(n, cores, 32))

    t0 = time.perf_counter()
    # w1: per-tensor symmetric int8 (statistics, scale, given-scale map), STE
    y1, m1 = np.empty(n1, np.float32), np.empty((n1 + 31) // 32, np.uint32)
    s1 = np.array([absmax_of(x1n, oracle.F32, n1) / np.float32(127)], np.float32)
    z1 = np.zeros(1, np.int32)

    def w1_piece(a, b):
        fl = ctypes.c_int32(0)
        L.or_fake_quant_int(P(x1n[a:b]), oracle.F32, 1, b - a, 8, oracle.SYM, oracle.PER_TENSOR, 0,
                            1, P(s1), P(z1), P(y1[a:b]), None, P(m1[a // 32:]), ctypes.byref(fl), 1)
    run(w1_piece, _spans(n1, cores, 1024))
    dx1 = np.empty_like(g1n)
    ste(g1n, oracle.F32, n1, m1, dx1)
    # w2: per row, affine int8 and symmetric int4
    int_rows(w2n.reshape(-1), oracle.F32, r2, c2, 8, oracle.AFFINE, oracle.PER_ROW, 0,
             np.empty(n2, np.float32), np.empty(n2, np.int8), np.empty(n2 // 32, np.uint32),
             np.empty(r2, np.float32), np.empty(r2, np.int32))
    int_rows(w2n.reshape(-1), oracle.F32, r2, c2, 4, oracle.SYM, oracle.PER_ROW, 0,
             np.empty(n2, np.float32), np.empty(n2 // 2, np.uint8), np.empty(n2 // 32, np.uint32),
             np.empty(r2, np.float32), np.empty(r2, np.int32))
    # w3: per-tensor amax FP8, both formats (the amax is the same for both)
    a3f = a3b.reshape(-1)
    amax3 = absmax_of(a3f, oracle.BF16, n3)
    for fmt in (oracle.E4M3, oracle.E5M2):
        s3 = ctypes.c_float(float(amax3 / np.float32(oracle.FP8_MAX[fmt])))
        y3, m3 = np.empty(n3, np.uint16), np.empty(n3 // 32, np.uint32)

        def w3_piece(a, b, s3=s3, y3=y3, m3=m3, fmt=fmt):
            fl = ctypes.c_int32(0)
            s = ctypes.c_float(s3.value)
            L.or_fake_quant_fp8(P(a3f[a:b]), oracle.BF16, b - a, fmt, 1, ctypes.byref(s),
                                P(y3[a:b]), None, P(m3[a // 32:]), ctypes.byref(fl))
        run(w3_piece, _spans(n3, cores, 1024))
        if keep is not None:
            keep.setdefault("fp8", []).append((y3, m3, s3.value))
    # w4: per group of 128, symmetric int4, then the STE
    m4 = np.empty(n4 // 32, np.uint32)
    int_rows(w4b.reshape(-1), oracle.BF16, r4, c4, 4, oracle.SYM, oracle.PER_GROUP, 128,
             np.empty(n4, np.uint16), np.empty(n4 // 2, np.uint8), m4,
             np.empty(n4 // 128, np.float32), np.empty(n4 // 128, np.int32))
    dx4 = np.empty(n4, np.uint16)
    ste(g4b.reshape(-1), oracle.BF16, n4, m4, dx4)
    # w5: two-level 4-bit quantize, then dequantize, per run of super-blocks
    nd, nb, ns = oracle.q4_sizes(n5)
    d5, q5, u5 = np.zeros(nd, np.uint8), np.zeros(nb, np.uint8), np.zeros(ns, np.float32)
    y5 = np.empty(n5, np.float32)
    spans5 = _spans(n5, cores, 16384)

    def q_piece(a, b):
        L.or_quant4_double(P(x5n[a:b]), b - a, P(d5[a // 2:]), P(q5[a // 64:]),
                           P(u5[a // 16384:]), None)

    def dq_piece(a, b):
        L.or_dequant4_double(P(d5[a // 2:]), P(q5[a // 64:]), P(u5[a // 16384:]), b - a,
                             P(y5[a:b]))
    run(q_piece, spans5)
    run(dq_piece, spans5)
    secs = time.perf_counter() - t0
    if keep is not None:
        keep.update(w1=(y1, m1, s1[0], dx1), dx4=dx4, w5=(d5, q5, u5, y5))
    wb = workload_bytes(n1, r2, c2, n3, r4, c4, n5)
    return secs, sum(b for _, _, b, _ in wb), sum(e for _, e, _, _ in wb)


def cpu_baseline(inputs, passes: int):
    """The oracle over the benchmark's own full-size inputs: single-threaded
    (the oracle as it stands), and beside it the same oracle functions split
    over every host core by oracle_step_parallel."""
    secs = nbytes = elems = 0.0
    for _ in range(passes):
        s, b, e = oracle_step(inputs)
        secs, nbytes, elems = secs + s, nbytes + b, elems + e
    out = {"value": round(nbytes / secs / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
           "Gelem_s": round(elems / secs / 1e9, 4), "seconds": round(secs, 2),
           "sample": f"the five workloads at full size (the GPU run's own inputs), {passes} "
                     f"pass(es) of the whole path, single-threaded C oracle"}
    import concurrent.futures as cf

    cores = host_cores()
    with cf.ThreadPoolExecutor(max_workers=cores) as pool:
        oracle_step_parallel(inputs, pool, cores)  # warm the pool and the pages
        t = [oracle_step_parallel(inputs, pool, cores) for _ in range(passes)]
    med = sorted(t, key=lambda r: r[0])[len(t) // 2]
    out["all_cores"] = {"value": round(med[1] / med[0] / 1e9, 4), "unit": "GB/s", "cores": cores,
                        "kind": "oracle", "Gelem_s": round(med[2] / med[0] / 1e9, 4),
                        "seconds": round(med[0], 3),
                        "sample": f"the same inputs, median of {passes} passes; the oracle's "
                                  f"functions on pieces of every call, one thread per core"}
    return out


def run_reference(args, rank, world):
    if rank != 0:
        return None
    frac = args.ref_fraction
    if frac <= 0:
        # size each step so the whole run stays within about two minutes
        probe = 1 / 256
        secs, _, _ = oracle_step(oracle_sample(probe))
        per_full = secs / probe
        frac = 120.0 / max(1, args.steps + args.warmup) / per_full
        frac = float(min(1 / 8, max(1 / 4096, frac)))
    inputs = oracle_sample(frac)
    for _ in range(args.warmup):
        oracle_step(inputs)
    tot_s, tot_b, tot_e = 0.0, 0.0, 0.0
    for _ in range(args.steps):
        s, b, e = oracle_step(inputs)
        tot_s += s
        tot_b += b
        tot_e += e
    value = tot_b / tot_s / 1e9
    sample = (f"every workload at {frac:g} of its rows/elements (same distributions), "
              f"single-threaded C oracle, one pass of the whole path per step")
    return {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(tot_s / args.steps * 1e3, 2), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32/bf16 in, fp32 arithmetic",
            "data": "synthetic", "config": {"workload": WORKLOAD, "sample_fraction": frac},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": sample, "Gelem_s": round(tot_e / tot_s / 1e9, 4)},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--cpu-passes", type=int, default=3,
                    help="oracle passes over the full workloads for cpu_baseline")
    ap.add_argument("--ref-fraction", type=float, default=0.0,
                    help="per-step sample of the reference arm (0: sized to ~2 min in total)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-isolated", action="store_true",
                    help="skip the per-call timings with an L2 flush before each call")
    ap.add_argument("--no-next", action="store_true",
                    help="skip the stochastic-rounding and CUDA-graph timings (next_rows)")
    ap.add_argument("--only", default="",
                    help="profiling: comma-separated call-name prefixes to run (e.g. w5,w4_int4); "
                         "names ending in _sr or holding _col select stochastic-rounding and "
                         "per-column rows (e.g. w1,w3_fp8_e4m3_tensor_sr,w2_affine_int8_col)")
    ap.add_argument("--fraction", type=float, default=1.0,
                    help="profiling: fraction of every workload's rows to generate")
    args = ap.parse_args(argv)
    args.warmup = max(args.warmup, 3)
    rank, world, local = dist_env()
    if world > 1 and args.impl == "ours":
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    else:
        line = run_ours(args, rank, world, local)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if world > 1 and args.impl == "ours":
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
