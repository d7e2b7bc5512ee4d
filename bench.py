"""Benchmark of the block-quantized GEMV on GB300.

One step is one pass of the whole product over one activation: q_matvec --
the f32 activation quantized per 256-element block under m*2^e, then the
Q4_K-like 4096x4096 matrix times it (exact block sums, once-rounded block
values, in-order row fold), in a single launch -- the workload the headline
metric is quoted on.
Weights are seeded synthetic data with the format's distributions; each step
reads a different copy of the matrix, and the copies total more than 4x the
L2, so every step streams its weights from HBM.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                  [--workload q4k_4096x4096|q8_0_512x1024|q6k_14336x4096|f16_49152x576|...]

Workloads ending in _sub32 run the ActScaling::Sub32 product (activation
scales per 32 elements, one rounding per 256-element group) through
q_matvec_sub32: one launch a step for one column (x quantized in the product
kernel's prologue), quantize_act_sub32 then q_gemv_sub32 otherwise.

Prints one JSON line.  --impl reference times the CPU oracle (test
infrastructure; a deliberately plain scalar C program) on the host cores.
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

from block_quantized_weight_quantize_gb300 import synth  # noqa: E402

L2_BYTES = 129 * 1024 * 1024
WORKLOADS = {
    # name: (fmt, rows, K, ncols, seed, outlier fraction, description)
    "q4k_4096x4096": (synth.FMT_Q4K, 4096, 4096, 1, 1, 0.001,
                      "Q4_K-like GEMV 4096x4096, batch 1, activation N(0,1) with 0.1% outliers x50"),
    "q8_0_512x1024": (synth.FMT_Q8_0, 512, 1024, 1, 0, 0.0, "Q8_0 GEMV 512x1024, batch 1"),
    "q6k_14336x4096": (synth.FMT_Q6K, 14336, 4096, 1, 2, 0.0, "Q6_K-like FFN gate 14336x4096, batch 1"),
    "f16_49152x576": (synth.FMT_F16, 49152, 576, 1, 3, 0.0, "F16 tied-embedding logits 49152x576, batch 1"),
    "q4k_4096x4096_b16": (synth.FMT_Q4K, 4096, 4096, 16, 1, 0.001, "Q4_K-like GEMV 4096x4096, 16 columns"),
    "q4k_4096x4096_b4": (synth.FMT_Q4K, 4096, 4096, 4, 1, 0.001, "Q4_K-like GEMV 4096x4096, 4 columns"),
    "q4k_28672x4096_b4": (synth.FMT_Q4K, 28672, 4096, 4, 1, 0.001,
                          "Q4_K-like FFN gate+up 28672x4096, 4 columns"),
    # ActScaling::Sub32: activation scales per 32 elements, one rounding per 256-element group
    "q4k_4096x4096_sub32": (synth.FMT_Q4K, 4096, 4096, 1, 1, 0.001,
                            "Q4_K-like GEMV 4096x4096, batch 1, activation scaled per 32 (Sub32)"),
    "q4k_4096x4096_b16_sub32": (synth.FMT_Q4K, 4096, 4096, 16, 1, 0.001,
                                "Q4_K-like GEMV 4096x4096, 16 columns, activation scaled per 32 (Sub32)"),
    "q8_0_4096x4096_sub32": (synth.FMT_Q8_0, 4096, 4096, 1, 5, 0.001,
                             "Q8_0 GEMV 4096x4096, batch 1, activation scaled per 32 (Sub32)"),
    "q6k_14336x4096_sub32": (synth.FMT_Q6K, 14336, 4096, 1, 2, 0.0,
                             "Q6_K-like FFN gate 14336x4096, batch 1, activation scaled per 32 (Sub32)"),
}
SUB32 = {k for k in WORKLOADS if k.endswith("_sub32")}


# Matrices that share one activation, run as one grouped call (q_matvec_many):
# name: (fmt, rows of each matrix, K, ncols, seed, outlier fraction, description)
GROUPED = {
    "q4k_qkv_4096": (synth.FMT_Q4K, [4096, 1024, 1024], 4096, 1, 4, 0.001,
                     "Q4_K-like Q, K, V projections (4096, 1024, 1024 rows x 4096), batch 1, one grouped launch"),
}


# A Q6_K-like FFN block at batch 1: gate and up (14336x4096) from one shared
# activation in one grouped call, then down (4096x14336) from its own
# activation (q_matvec_many + q_matvec a step):
# name: (fmt, gate/up rows, K, down rows, seed, description)
FFN = {
    "q6k_ffn_14336x4096": (synth.FMT_Q6K, 14336, 4096, 4096, 2,
                           "Q6_K-like FFN: gate + up 14336x4096 (one grouped call) and down 4096x14336, batch 1"),
}

# The int8 cache's score path: query heads quantized, then scored against the
# cached key rows (kv_quantize_heads + kv_scores a step):
# name: (scaling, query heads, key heads, head size, cached positions, seed, description)
KV = {
    "kv_scores_32k_sub32": (1, 32, 8, 128, 32768, 6,
                            "int8 key cache scores: 32 query heads on 8 key heads of 128, 32768 positions, "
                            "query scaled per 32 (Sub32)"),
    "kv_scores_32k_perblock": (0, 32, 8, 128, 32768, 6,
                               "int8 key cache scores: 32 query heads on 8 key heads of 128, 32768 positions, "
                               "query one block a head (PerBlock)"),
}


# FP8 E4M3 weights with 128x128 block scales (q_gemv_fp8, one launch a step):
# name: (rows, K, columns, seed, description)
FP8 = {
    "fp8_4096x4096": (4096, 4096, 1, 7, "FP8 E4M3 GEMV 4096x4096, 128x128 block scales, batch 1"),
    "fp8_4096x4096_b16": (4096, 4096, 16, 7, "FP8 E4M3 GEMV 4096x4096, 128x128 block scales, 16 columns"),
}


# The 8B-class decode stack: a step is every product of one decode step --
# 32 layers of QKV 6144x4096, O 4096x4096, gate+up 28672x4096, down 4096x14336
# (Q4_K-like) and the 128256x4096 Q6_K-like output -- each from its f32
# activation in one q_matvec call (name: columns)
STACK = {"stack_8b_b1": 1, "stack_8b_b4": 4, "stack_8b_b16": 16}

# Activation codes that cross in two words (16-bit codes: a signed high byte
# weighted by 256 and an unsigned low byte), q_gemv_w2 a step:
# name: (fmt, rows, K, ncols, seed, description)
W2 = {
    "q4k_4096x4096_w2": (synth.FMT_Q4K, 4096, 4096, 1, 8,
                         "Q4_K-like GEMV 4096x4096, batch 1, two-word (16-bit) activation codes"),
}
STACK_LAYERS = 32
STACK_MATS = [("qkv", synth.FMT_Q4K, 6144, 4096), ("o", synth.FMT_Q4K, 4096, 4096),
              ("gate_up", synth.FMT_Q4K, 28672, 4096), ("down", synth.FMT_Q4K, 4096, 14336)]
STACK_OUT = ("output", synth.FMT_Q6K, 128256, 4096)


def metric_for(workload):
    """The metric string of a workload, the same on both arms."""
    if workload == "q4k_4096x4096":
        return "weight GB/s at batch 1 (Q4_K-like GEMV 4096x4096, rows/s and fraction of 8 TB/s alongside)"
    if workload in STACK:
        return (f"weight GB/s (8B-class decode stack, {STACK[workload]} column(s): 32 layers of Q4_K-like QKV "
                f"6144x4096, O 4096x4096, gate+up 28672x4096, down 4096x14336 + Q6_K-like output 128256x4096)")
    if workload in KV:
        return f"key-cache GB/s ({KV[workload][-1]})"
    desc = (WORKLOADS[workload][-1] if workload in WORKLOADS else GROUPED[workload][-1] if workload in GROUPED
            else FFN[workload][-1] if workload in FFN else W2[workload][-1] if workload in W2 else FP8[workload][-1])
    return f"weight GB/s ({desc})"


def kernel_sources_sha() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "block_quantized_weight_quantize_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def barrier():
    """All ranks meet (nothing to do for one process)."""
    import torch.distributed as tdist
    if tdist.is_available() and tdist.is_initialized() and tdist.get_world_size() > 1:
        tdist.barrier()


def max_over_ranks(v, device=None) -> float:
    """The largest v over the ranks (v itself for one process): a timed region
    lasts until its slowest rank ends."""
    import torch
    import torch.distributed as tdist
    if not (tdist.is_available() and tdist.is_initialized()) or tdist.get_world_size() == 1:
        return float(v)
    dev = device if tdist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(v)], dtype=torch.float64, device=dev)
    tdist.all_reduce(t, op=tdist.ReduceOp.MAX)
    return float(t.item())


def lead_in(stream) -> None:
    """Queues ~0.1 ms of spinning on the stream right before the timed region's
    first event, so that the host has submitted the timed graph before the GPU
    reaches it: otherwise the first replay's host-side submission (tens of us)
    is counted as idle GPU time inside the region, which at a few dozen steps
    inflates the step time by tens of percent."""
    import torch
    with torch.cuda.stream(stream):
        torch.cuda._sleep(200_000)


def one_graph_timing(capture_steps, stream, warmup, steps, max_steps=1000):
    """For a run of at most `max_steps` timed steps: captures one CUDA graph of
    `warmup` untimed steps followed by the `steps` timed ones, with the start
    event recorded on a branch that waits for the last warm-up step to
    complete and the end event after the last timed step.  The launch chain
    itself is left as in a long run -- each step's launch may begin while its
    predecessor drains (programmatic dependent launch) -- so the events span
    exactly `steps` step completions of a running pipeline: an event between
    two launches would instead hold the next one back until the previous one
    finished.  Replays the graph once untimed and returns (graph, start
    event, end event), or None where this torch cannot record events as graph
    nodes, or the run is longer."""
    import torch
    if steps > max_steps:
        return None
    try:
        t0 = torch.cuda.Event(enable_timing=True, external=True)
        t1 = torch.cuda.Event(enable_timing=True, external=True)
    except TypeError:  # no event record nodes in this torch
        return None
    side = torch.cuda.Stream(stream.device)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        g.capture_begin()
        try:
            capture_steps(0, max(1, warmup))
            fork = torch.cuda.Event()
            fork.record(stream)
            side.wait_event(fork)
            t0.record(side)
            capture_steps(max(1, warmup), steps)
            t1.record(stream)
            join = torch.cuda.Event()
            join.record(side)
            stream.wait_event(join)
        finally:
            g.capture_end()
    with torch.cuda.stream(stream):
        g.replay()
    stream.synchronize()
    return g, t0, t1


def prime_graph(g, stream) -> str:
    """Readies a captured CUDA graph so that its first replay inside a timed
    region costs what every later one does: the instantiated graph is uploaded
    to the device (cuGraphUpload) ahead of the timing.  Where the executable
    graph's handle is not reachable from this torch, the graph is replayed once,
    untimed, instead.  Returns which of the two was done."""
    import ctypes
    import torch
    try:
        h = g.raw_cuda_graph_exec()
        rc = ctypes.CDLL("libcuda.so.1").cuGraphUpload(ctypes.c_void_p(h), ctypes.c_void_p(stream.cuda_stream))
        if rc == 0:
            stream.synchronize()
            return "uploaded before timing"
    except Exception:
        pass
    with torch.cuda.stream(stream):
        g.replay()
    stream.synchronize()
    return "replayed once untimed before timing"


def traffic_for(workload):
    """DRAM bytes per launch of the workload's dominant kernel from the committed
    ncu summary, or None when the kernels changed since that capture."""
    tp = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(tp):
        return None
    ent = json.load(open(tp)).get(workload)
    if ent and ent.get("src_sha") == kernel_sources_sha():
        return ent.get("dram_bytes_per_launch")
    return None


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def tensor_peak():
    """Dense f16 tensor-core TFLOP/s: the measured bf16 burst figure (f16 and
    bf16 share the nominal rate), else the stated fallback."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        if "bf16_tflops" in d:
            return float(d["bf16_tflops"]), "measured (cuBLAS bf16 GEMM, burst; f16 has the same nominal rate)"
    return 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            f = [t.strip() for t in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": ["no samples"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def algorithmic_bytes(fmt, rows, K, ncols, sub32=False):
    """Weights + activation (codes, 4-B block scales, 2-B unit sums) + outputs."""
    wb = synth.weight_bytes(fmt, rows, K)
    if fmt == synth.FMT_F16:
        return wb, wb + ncols * 2 * K + 4 * rows * ncols
    blk = 32 if sub32 else synth.BLOCK[fmt]
    return wb, wb + ncols * (K + 4 * (K // blk) + 2 * (K // 16)) + 4 * rows * ncols


# The multi-column product is bound by the integer pipeline, not by HBM: its
# roofline is the dp4a issue rate, 64 lanes a clock per SM (two warp
# instructions a clock; a throughput probe on a GB300 measured 1.885) x 8 ops
# (4 multiply-adds) x 152 SMs x 2.07 GHz (the maximum SM clock).
DP4A_PEAK_TOPS = 64 * 8 * 152 * 2.07e9 / 1e12


def one_col_gemv3(fmt, rows, K):
    """The library's rule for one column: the 256-element formats take the
    multi-column kernel's organisation when the one-column kernel would need
    more than one ring iteration per CTA (more than 2 * (512 // (K/128)) rows a
    CTA over min(152, rows) CTAs)."""
    if fmt == synth.FMT_Q8_0 or K % 256:
        return False
    g = max(1, min(152, rows))
    return ((rows + g - 1) // g + 1) // 2 > 512 // (K // 128)


def one_col_gemv6(fmt, rows, K):
    """The library's rule for the warp-ring one-column kernel: K = 4096, every
    Q6_K-like shape, Q4_K-like ones up to 48 rows a CTA over min(152, rows/2) CTAs."""
    if fmt not in (synth.FMT_Q4K, synth.FMT_Q6K) or K != 4096 or rows < 1:
        return False
    g = max(1, min(152, (rows + 1) // 2))
    return fmt == synth.FMT_Q6K or (rows + g - 1) // g <= 48


def one_col_gemv7(fmt, rows, K):
    """The library's rule for the block-per-warp one-column kernel: K = 4096,
    rows a CTA (over min(152, rows) CTAs) up to 32, or as many as fit the
    shared-memory budget of two CTAs a SM (Q4_K-like 45, Q6_K-like 31)."""
    if fmt not in (synth.FMT_Q4K, synth.FMT_Q6K) or K != 4096 or rows < 1:
        return False
    g = max(1, min(152, rows))
    per = (rows + g - 1) // g
    pitch = synth.weight_bytes(fmt, 1, K) + 16
    smem = 9088 + per * pitch   # codes, sums, the block-value table, the rows
    return (fmt == synth.FMT_Q4K and per <= 32) or smem <= (228 * 1024) // 2 - 1024 - 256


TC_MIN_COLS = 9


def tc_applies(fmt, K, ncols):
    """The library's rule for the tensor-core (tcgen05) kernel: Q4_K-like or
    Q6_K-like, K % 256 == 0, from TC_MIN_COLS columns, and some cluster split of
    the blocks (1..8 CTAs) whose shared memory fits 227 KB."""
    if fmt not in (synth.FMT_Q4K, synth.FMT_Q6K) or K % 256 or ncols < TC_MIN_COLS:
        return False
    nb = K // 256
    bb = 144 if fmt == synth.FMT_Q4K else 208
    for ks in range(1, min(8, nb) + 1):
        nbq, cpc = -(-nb // ks), -(-ncols // ks)
        if fmt == synth.FMT_Q6K and 2 * nbq + 14 > 64:
            continue
        bact = (8 * (8 + nbq) + 4 + 127) // 128 * 128
        total = (bact + nbq * 8192 + (nbq * 512 if fmt == synth.FMT_Q4K else 0) + (16 * nbq * 4 + 127) // 128 * 128 +
                 (cpc * nb * 512 + 127) // 128 * 128 + nbq * 128 * bb + (128 * 64 if fmt == synth.FMT_Q6K else 0))
        if total <= 227 * 1024:
            return True
    return False


def multi_col_kernel(fmt, rows, K, ncols):
    """The library's choice of product kernel for 2..16 columns (Q4_K-like /
    Q6_K-like): the tensor-core kernel from TC_MIN_COLS columns; at 2..4
    columns and K = 4096 the warp-per-block kernel while a CTA's rows (at
    most 64) fit its shared memory, else (Q4_K-like) its ring form, which also
    takes K = 8192 and 14336; the dp4a CTA-ring kernel otherwise."""
    if tc_applies(fmt, K, ncols):
        return f"tc_kernel<{synth.FORMAT_NAMES[fmt]}, {ncols} columns> (tcgen05 f16 MMAs, accumulators in tensor memory)"
    g = max(1, min(152, rows))
    per = (rows + g - 1) // g
    if 2 <= ncols <= 4 and K == 4096 and per <= 64:
        pitch = synth.weight_bytes(fmt, 1, K) + 16
        vs = (ncols * 17) | 1
        smem = (128 + (ncols * 64 + 127) // 128 * 128 + ncols * 4096 + ncols * 512 + (64 * vs * 4 + 127) // 128 * 128 +
                per * pitch)
        minb = 1 if ncols >= 3 and per > 32 else 2
        if smem <= (228 * 1024) // minb - 1280:
            return (f"gemv7m_kernel<{synth.FORMAT_NAMES[fmt]}, {ncols} columns, a warp per block, a lane per row, "
                    f"{minb} CTA(s) a SM>")
    if fmt == synth.FMT_Q4K and 2 <= ncols <= 4 and K in (4096, 8192, 14336) and (K != 4096 or per > 64):
        return (f"gemv7r_kernel<q4k, {ncols} columns, ring of 32-row tiles, a warp per block, a lane per row, "
                f"producer warp>")
    return f"gemv3_kernel<{synth.FORMAT_NAMES[fmt]}, {ncols} columns>"


def roofline(fmt, ncols, single, achieved, peak, peak_kind, traffic, roof_bytes, per_launch_s, prod_s, abytes,
             ops_per_step, roof_launches, sub32=False, rows=0, K=0):
    g7 = ncols == 1 and not sub32 and fmt != synth.FMT_F16 and one_col_gemv7(fmt, rows, K)
    g6 = ncols == 1 and not sub32 and fmt != synth.FMT_F16 and not g7 and one_col_gemv6(fmt, rows, K)
    g3 = ncols == 1 and not sub32 and fmt != synth.FMT_F16 and not g6 and one_col_gemv3(fmt, rows, K)
    g6name = (f"gemv6_kernel<{synth.FORMAT_NAMES[fmt]}, one column, warp rings" +
              (", single launch> (quantize + product)" if single else ">"))
    g7name = (f"gemv7_kernel<{synth.FORMAT_NAMES[fmt]}, one column, a warp per block, a lane per row" +
              (", single launch> (quantize + product)" if single else ">"))
    name = (g7name if g7 else g6name if g6 else
            f"gemv_f16w_kernel<{ncols}{', single launch (f16 rounding in the prologue)' if single else ''}>"
            if fmt == synth.FMT_F16 else
            (f"s32_kernel<{synth.FORMAT_NAMES[fmt]}, one column, single launch> (quantize + product)" if single
             else f"s32_kernel<{synth.FORMAT_NAMES[fmt]}, {min(ncols, 2)} column(s) a thread group>") if sub32 else
            f"gemv3_kernel<{synth.FORMAT_NAMES[fmt]}, one column, single launch> (quantize + product)"
            if single and g3 else
            f"gemv2_kernel<{synth.FORMAT_NAMES[fmt]}, single launch> (quantize + product)" if single and ncols == 1
            else multi_col_kernel(fmt, rows, K, ncols))
    prod = {"avg_launch_us": round(prod_s * 1e6, 4),
            "achieved_gbs": round(abytes / prod_s / 1e9, 1),
            "frac_of_hbm": round(abytes / prod_s / 1e9 / peak, 4),
            "note": "activation quantized beforehand (q_gemv)"}
    if fmt != synth.FMT_F16 and ncols > 1 and not sub32 and tc_applies(fmt, K, ncols):
        tflops = ops_per_step / prod_s / 1e12
        tpk, tkind = tensor_peak()
        return {"bound": "tensor", "kernel": name, "achieved": round(tflops, 2), "peak": round(tpk, 1),
                "peak_kind": tkind, "unit": "TFLOP/s", "frac": round(tflops / tpk, 4), "traffic": traffic,
                "algorithmic_ops_per_launch": ops_per_step, "avg_launch_us": round(prod_s * 1e6, 4),
                "launches_timed": 3 * roof_launches, "hbm_side": prod,
                "dp4a_side": {"achieved_tops": round(tflops, 2), "peak_tops": round(DP4A_PEAK_TOPS, 1),
                              "frac": round(tflops / DP4A_PEAK_TOPS, 4)}}
    if fmt != synth.FMT_F16 and ncols > 1:
        tops = ops_per_step / prod_s / 1e12
        return {"bound": "alu", "kernel": name, "achieved": round(tops, 2), "peak": round(DP4A_PEAK_TOPS, 1),
                "peak_kind": "dp4a issue rate from unit counts and the maximum clock (64 lanes/clk/SM x 8 ops x "
                             "152 SMs x 2.07 GHz)",
                "unit": "TOPS", "frac": round(tops / DP4A_PEAK_TOPS, 4), "traffic": traffic,
                "algorithmic_ops_per_launch": ops_per_step, "avg_launch_us": round(prod_s * 1e6, 4),
                "launches_timed": 3 * roof_launches, "hbm_side": prod}
    return {"bound": "hbm", "kernel": name, "achieved": round(achieved, 1), "peak": peak,
            "peak_kind": f"{peak_kind} (HBM copy, burst)", "unit": "GB/s", "frac": round(achieved / peak, 4),
            "traffic": traffic, "algorithmic_bytes_per_launch": roof_bytes,
            "avg_launch_us": round(per_launch_s * 1e6, 4), "launches_timed": 3 * roof_launches,
            "product_kernel_only": prod}


# ---------------------------------------------------------------- our arm

def _kv_inputs(scaling, nh, nkv, d, L, seed):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((nh, d)).astype(np.float32)
    k = rng.standard_normal((nkv * L, d)).astype(np.float32)
    return q, k


def run_kv(args, rank, world):
    """A step is kv_quantize_heads + kv_scores over the whole key cache; the
    cache (int8 codes + f16 scales, built by kv_cache_rows) is the streamed input."""
    import torch
    import block_quantized_weight_quantize_gb300 as qb

    scaling, nh, nkv, d, L, seed, desc = KV[args.workload]
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    q, k = _kv_inputs(scaling, nh, nkv, d, L, seed + 1000 * rank)
    kbytes = nkv * L * (d + 2)
    ncopy = max(2, -(-4 * L2_BYTES // kbytes))
    kc = torch.empty((ncopy, nkv, L, d), dtype=torch.int8, device=dev)
    ks = torch.empty((ncopy, nkv, L), dtype=torch.int16, device=dev)
    kd = torch.from_numpy(k).to(dev)
    qb.kv_cache_rows(kd, kc[0].view(nkv * L, d), ks[0].view(-1))
    for i in range(1, ncopy):
        kc[i].copy_(kc[0])
        ks[i].copy_(ks[0])
    del kd
    qd = torch.from_numpy(q).to(dev)
    dp = qb.kv_head_codes(scaling, d)
    nbq = dp // 32 if scaling == qb.SUB32 else 1
    qc = torch.empty((nh, dp), dtype=torch.int8, device=dev)
    qs = torch.empty((nh, nbq), dtype=torch.int32, device=dev)
    out = torch.empty((nh, L), dtype=torch.float32, device=dev)
    scale = float(1.0 / np.sqrt(d))
    stream = torch.cuda.Stream(dev)

    def step(i, s):
        qb.kv_quantize_heads(scaling, qd, qc, qs, stream=s)
        qb.kv_scores(scaling, qc, qs, d, kc[i % ncopy], ks[i % ncopy], L, scale, out, stream=s)

    def scores_only(i, s):
        qb.kv_scores(scaling, qc, qs, d, kc[i % ncopy], ks[i % ncopy], L, scale, out, stream=s)

    with torch.cuda.stream(stream):
        for i in range(3):
            step(i, stream)
    stream.synchronize()
    G = min(args.steps, 200)

    def capture(fn, n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            g.capture_begin()
            for i in range(n):
                fn(i, stream)
            g.capture_end()
        return g

    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    g_main = capture(step, G)
    g_w = capture(step, max(1, min(args.warmup, G)))
    with torch.cuda.stream(stream):
        for _ in range(max(1, args.warmup // max(1, min(args.warmup, G)))):
            g_w.replay()
    stream.synchronize()
    primed = prime_graph(g_main, stream)
    nrep = max(1, args.steps // G)
    with ClockSampler(dev.index) as clk:
        barrier()
        torch.cuda.synchronize()
        lead_in(stream)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(nrep):
                g_main.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        barrier()
    ms = max_over_ranks(e0.elapsed_time(e1), dev) / (nrep * G)
    clocks = clk.summary()
    g_roof = capture(scores_only, G)
    with torch.cuda.stream(stream):
        g_roof.replay()
        e0.record(stream)
        for _ in range(3):
            g_roof.replay()
        e1.record(stream)
    stream.synchronize()
    sc_s = e0.elapsed_time(e1) / 1e3 / (3 * G)
    roof_bytes = kbytes + nh * (dp + 4 * nbq) + 4 * nh * L
    peak, peak_kind = measured_peaks()
    # e2e: the query from pinned host memory, the scores back to pinned host memory
    qh = torch.from_numpy(q).pin_memory()
    oh = torch.empty((nh, L), dtype=torch.float32).pin_memory()
    n_e2e = min(args.steps, 2000)
    barrier()
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for i in range(n_e2e):
            qd.copy_(qh, non_blocking=True)
            step(i, stream)
            oh.copy_(out, non_blocking=True)
    stream.synchronize()
    e2e_s = max_over_ranks(time.perf_counter() - t0, dev)
    assert qb.q_device_status() == qb.QB_OK
    step_s = ms / 1e3
    value = world * kbytes / step_s / 1e9
    res = {
        "metric": metric_for(args.workload),
        "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": nrep * G, "warmup": args.warmup,
        "ms_per_step": round(ms, 6), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "int8 codes x int8 codes (tensor-core s8 MMA), exact int64, f32 rounding",
        "data": "synthetic (seeded PCG64; N(0,1) keys and queries); no trained weights",
        "config": {"workload": desc, "query_heads": nh, "key_heads": nkv, "head": d, "positions": L,
                   "scaling": "Sub32" if scaling == 1 else "PerBlock", "key_bytes_per_step": kbytes,
                   "l2": f"each step reads a different one of {ncopy} key caches ({ncopy * kbytes / 2**20:.0f} MiB "
                         f"> 4x L2); no flush",
                   "timing": f"CUDA graphs of {G} steps (kv_quantize_heads + kv_scores, 2 launches a step); "
                             f"CUDA events on the launching stream; the timed graph {primed}",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "scores_per_s": round(world * nh * L / step_s, 1),
        "frac_of_8tbs": round(value / 8000.0, 4), "frac_of_measured_copy": round(value / peak, 4),
        "gpu_launches": 2 * nrep * G, "clocks": clocks,
        "roofline": {"bound": "hbm", "kernel": f"kv_scores_kernel<{'Sub32' if scaling else 'PerBlock'}, {d // 32} blocks>",
                     "achieved": round(roof_bytes / sc_s / 1e9, 1), "peak": peak,
                     "peak_kind": f"{peak_kind} (HBM copy, burst)", "unit": "GB/s",
                     "frac": round(roof_bytes / sc_s / 1e9 / peak, 4), "traffic": traffic_for(args.workload),
                     "algorithmic_bytes_per_launch": roof_bytes, "avg_launch_us": round(sc_s * 1e6, 4),
                     "launches_timed": 3 * G},
        "e2e": {"value": round(world * kbytes * n_e2e / e2e_s / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": int(q.nbytes), "d2h_bytes_per_step": int(4 * nh * L), "steps": n_e2e,
                "how": "per step: pinned query -> device, kv_quantize_heads + kv_scores through the binding, "
                       "scores -> pinned host; host wall clock"},
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = kv_cpu_baseline(scaling, nh, nkv, d, L, q, k, kbytes, args.cpu_seconds)
    return res


def run_grouped(args, rank, world):
    """A step is one grouped call over the matrices of GROUPED[workload]; the
    same step as one call per matrix is timed alongside."""
    import torch
    import block_quantized_weight_quantize_gb300 as qb

    fmt, rows_list, K, ncols, seed, outl, desc = GROUPED[args.workload]
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    rng = np.random.default_rng(seed + 1000 * rank)
    Whs = [synth.pack(fmt, synth.draw(fmt, rng, r, K)) for r in rows_list]
    x = synth.draw_act(rng, ncols, K, outlier_frac=outl)
    sizes = [W.size for W in Whs]
    offs = np.concatenate([[0], np.cumsum(sizes)]).astype(int)
    wbytes = int(offs[-1])
    ncopy = max(2, -(-4 * L2_BYTES // wbytes))
    buf = torch.empty((ncopy, wbytes), dtype=torch.uint8, device=dev)
    for j, W in enumerate(Whs):
        buf[0, offs[j]:offs[j + 1]].copy_(torch.from_numpy(W))
    for i in range(1, ncopy):
        buf[i].copy_(buf[0])
    mats = [[buf[i, offs[j]:offs[j + 1]] for j in range(len(rows_list))] for i in range(ncopy)]
    xd = torch.from_numpy(x).to(dev)
    outs = [torch.empty((ncols, r), dtype=torch.float32, device=dev) for r in rows_list]
    ws = torch.empty(qb.q_matvec_workspace_bytes(fmt, K, ncols), dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(dev)

    def grouped(i, s):
        qb.q_matvec_many(fmt, mats[i % ncopy], rows_list, K, xd, outs, workspace=ws, stream=s)

    def separate(i, s):
        for j, r in enumerate(rows_list):
            qb.q_matvec(fmt, mats[i % ncopy][j], r, K, xd, outs[j], workspace=ws, stream=s)

    with torch.cuda.stream(stream):
        for i in range(3):
            grouped(i, stream)
            separate(i, stream)
    stream.synchronize()
    G = min(args.steps, 1000)

    def capture(fn, n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            g.capture_begin()
            for i in range(n):
                fn(i, stream)
            g.capture_end()
        return g

    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)

    def time_graph(fn, steps, clocks=False):
        g = capture(fn, G)
        gw = capture(fn, max(1, min(args.warmup, G)))
        with torch.cuda.stream(stream):
            for _ in range(max(1, args.warmup // max(1, min(args.warmup, G)))):
                gw.replay()
        stream.synchronize()
        prime_graph(g, stream)
        sampler = ClockSampler(dev.index) if clocks else None
        if sampler:
            sampler.__enter__()
        barrier()
        torch.cuda.synchronize()
        lead_in(stream)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(max(1, steps // G)):
                g.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        barrier()
        if sampler:
            sampler.__exit__(None, None, None)
        ms_ = max_over_ranks(e0.elapsed_time(e1), dev)
        return ms_ / (max(1, steps // G) * G), (sampler.summary() if sampler else None)

    ms, clocks = time_graph(grouped, args.steps, clocks=True)
    ms_sep, _ = time_graph(separate, min(args.steps, 20000))
    step_s = ms / 1e3
    value = world * wbytes / step_s / 1e9
    peak, peak_kind = measured_peaks()
    roof_bytes = wbytes + 4 * K * ncols + 4 * sum(rows_list) * ncols
    # e2e through the binding with host buffers
    xh = torch.from_numpy(x).pin_memory()
    ohs = [torch.empty((ncols, r), dtype=torch.float32).pin_memory() for r in rows_list]
    n_e2e = min(args.steps, 3000)
    barrier()
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for i in range(n_e2e):
            xd.copy_(xh, non_blocking=True)
            grouped(i, stream)
            for oh, o in zip(ohs, outs):
                oh.copy_(o, non_blocking=True)
    stream.synchronize()
    e2e_s = max_over_ranks(time.perf_counter() - t0, dev)
    assert qb.q_device_status() == qb.QB_OK
    res = {
        "metric": metric_for(args.workload),
        "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": max(1, args.steps // G) * G,
        "warmup": args.warmup, "ms_per_step": round(ms, 6), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int8 codes x int8 codes, exact int32/int64, f32 rounding",
        "data": "synthetic (seeded PCG64; the format's code/scale distributions); no trained weights",
        "config": {"workload": desc, "rows": rows_list, "K": K, "ncols": ncols, "format": synth.FORMAT_NAMES[fmt],
                   "weight_bytes_per_step": wbytes,
                   "l2": f"each step reads a different one of {ncopy} copies of the group "
                         f"({ncopy * wbytes / 2**20:.0f} MiB > 4x L2); no flush",
                   "timing": f"CUDA graphs of {G} steps, one q_matvec_many launch a step; CUDA events",
                   "separate_calls_ms_per_step": round(ms_sep, 6),
                   "separate_calls_gbs": round(world * wbytes / (ms_sep / 1e3) / 1e9, 2),
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "rows_per_s": round(world * sum(rows_list) / step_s, 1),
        "frac_of_8tbs": round(value / 8000.0, 4), "frac_of_measured_copy": round(value / peak, 4),
        "gpu_launches": max(1, args.steps // G) * G, "clocks": clocks,
        "roofline": {"bound": "hbm",
                     "kernel": f"{'gemv7_kernel' if one_col_gemv7(fmt, sum(rows_list), K) else 'gemv6_kernel' if one_col_gemv6(fmt, sum(rows_list), K) else 'gemv3_kernel' if one_col_gemv3(fmt, sum(rows_list), K) else 'gemv2_kernel'}"
                               f"<{synth.FORMAT_NAMES[fmt]}, one column, single launch, grouped>",
                     "achieved": round(roof_bytes / step_s / 1e9, 1), "peak": peak,
                     "peak_kind": f"{peak_kind} (HBM copy, burst)", "unit": "GB/s",
                     "frac": round(roof_bytes / step_s / 1e9 / peak, 4), "traffic": traffic_for(args.workload),
                     "algorithmic_bytes_per_launch": roof_bytes, "avg_launch_us": round(ms * 1e3, 4)},
        "e2e": {"value": round(world * wbytes * n_e2e / e2e_s / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": int(x.nbytes), "d2h_bytes_per_step": int(4 * sum(rows_list) * ncols),
                "steps": n_e2e,
                "how": "per step: pinned x -> device, q_matvec_many through the Python binding, outputs -> pinned "
                       "host; host wall clock over all steps"},
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, n, sample = sampled_oracle_rate([(fmt, r, K, W, x, 1.0) for r, W in zip(rows_list, Whs)],
                                           args.cpu_seconds)
        res["cpu_baseline"] = {"value": round(v, 4), "unit": "GB/s", "cores": n, "kind": "oracle", "sample": sample}
    return res


def run_grouped_reference(args):
    """The reference arm on a grouped workload: the oracle over the group's
    matrices (one shared activation), sampled rows a step."""
    fmt, rows_list, K, ncols, seed, outl, desc = GROUPED[args.workload]
    rng = np.random.default_rng(seed)
    Whs = [synth.pack(fmt, synth.draw(fmt, rng, r, K)) for r in rows_list]
    x = synth.draw_act(rng, ncols, K, outlier_frac=outl)
    mats = [(fmt, r, K, W, x, 1.0) for r, W in zip(rows_list, Whs)]
    n = _oracle_threads()
    t0 = time.perf_counter()
    sampled_oracle_pass(mats, n, 1.0)
    full = time.perf_counter() - t0
    frac = max(1e-3, min(1.0, (100.0 / max(1, args.steps + args.warmup)) / max(full, 1e-6)))
    for _ in range(args.warmup):
        sampled_oracle_pass(mats, n, frac)
    done, t0 = 0, time.perf_counter()
    for _ in range(args.steps):
        done += sampled_oracle_pass(mats, n, frac)
    el = time.perf_counter() - t0
    value = done / el / 1e9
    sample = (f"each step: quantize + {frac:.3g} of the rows of each of the {len(rows_list)} matrices, split over "
              f"{n} threads of the scalar C oracle")
    return {
        "impl": "reference", "metric": metric_for(args.workload),
        "value": round(value, 4), "unit": "GB/s", "n_gpus": 0, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(el * 1e3 / args.steps, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int64/int128 exact, f32 rounding (scalar C)",
        "data": "synthetic (seeded PCG64)",
        "config": {"workload": desc, "rows": rows_list, "K": K, "ncols": ncols, "format": synth.FORMAT_NAMES[fmt]},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": n, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_ours(args, rank, world):
    import torch
    import block_quantized_weight_quantize_gb300 as qb

    fmt, rows, K, ncols, seed, outl, desc = WORKLOADS[args.workload]
    sub32 = args.workload in SUB32
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    rng = np.random.default_rng(seed + 1000 * rank)
    lg = synth.draw(fmt, rng, rows, K)
    Wh = synth.pack(fmt, lg)
    x = synth.draw_act(rng, ncols, K, outlier_frac=outl)
    wbytes, abytes = algorithmic_bytes(fmt, rows, K, ncols, sub32)
    ncopy = max(2, -(-4 * L2_BYTES // wbytes))        # copies totalling >= 4x L2
    W = torch.empty((ncopy, Wh.size), dtype=torch.uint8, device=dev)
    W[0].copy_(torch.from_numpy(Wh))
    for i in range(1, ncopy):
        W[i].copy_(W[0])
    xd = torch.from_numpy(x).to(dev)
    out = torch.empty((ncols, rows), dtype=torch.float32, device=dev)
    if fmt == synth.FMT_F16:
        act = torch.empty((ncols, K), dtype=torch.int16, device=dev)
    elif sub32:
        act = qb.alloc_act(ncols, K, 32, dev)
        qb.quantize_act_sub32(xd, *act)
    else:
        act = qb.alloc_act(ncols, K, synth.BLOCK[fmt], dev)
        qb.quantize_act(synth.BLOCK[fmt], xd, *act)
    ws = torch.empty(qb.q_matvec_sub32_workspace_bytes(K, ncols) if sub32 else
                     qb.q_matvec_workspace_bytes(fmt, K, ncols), dtype=torch.uint8, device=dev)
    # one launch per step where the single-launch product applies, else two
    # (Sub32 too: its one-column kernel quantizes x in its prologue; PerBlock
    # Q4_K-like rows of K >= 12288 given a workspace take quantize + product)
    single = ((fmt != synth.FMT_F16 and ncols == 1 and K % 256 == 0 and
               (sub32 or not (fmt == synth.FMT_Q4K and K >= 12288))) or
              (fmt == synth.FMT_F16 and ncols * K * 4 <= 227 * 1024) or
              # 2..4 columns at K = 4096: the warp-per-block kernel or its ring form from x
              (not sub32 and 2 <= ncols <= 4 and K == 4096 and
               multi_col_kernel(fmt, rows, K, ncols).startswith(("gemv7m", "gemv7r"))))
    launches_per_step = 1 if single else 2
    stream = torch.cuda.Stream(dev)

    def step(i, s):
        if sub32:
            qb.q_matvec_sub32(fmt, W[i % ncopy], rows, K, xd, out, workspace=ws, stream=s)
        else:
            qb.q_matvec(fmt, W[i % ncopy], rows, K, xd, out, workspace=ws, stream=s)

    def gemv_only(i, s):
        if sub32:
            qb.q_gemv_sub32(fmt, W[i % ncopy], rows, K, act, ncols, out, s)
        elif fmt == synth.FMT_F16:
            qb.q_gemv_f16(W[i % ncopy], rows, K, act, ncols, out, s)
        else:
            qb.q_gemv(fmt, W[i % ncopy], rows, K, act, ncols, out, s)

    # eager warm-up (also loads the kernels), then graphs of G steps each
    with torch.cuda.stream(stream):
        for i in range(3):
            step(i, stream)
    stream.synchronize()
    G = min(args.steps, 1000)

    def capture(fn, n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            g.capture_begin()
            for i in range(n):
                fn(i, stream)
            g.capture_end()
        return g

    g_main = capture(step, G)
    rem = args.steps % G
    g_rem = capture(step, rem) if rem else None
    g_w = capture(step, max(1, min(args.warmup, G)))

    def replay_steps(n_full, g_tail):
        for _ in range(n_full):
            g_main.replay()
        if g_tail is not None:
            g_tail.replay()

    # warm-up: W steps
    with torch.cuda.stream(stream):
        for _ in range(max(1, args.warmup // max(1, min(args.warmup, G)))):
            g_w.replay()
    stream.synchronize()
    primed = prime_graph(g_main, stream)
    if g_rem is not None:
        prime_graph(g_rem, stream)

    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    g_one = one_graph_timing(capture_steps=lambda n0, n: [step(n0 + i, stream) for i in range(n)],
                             stream=stream, warmup=args.warmup, steps=args.steps)
    with ClockSampler(dev.index) as clk:
        barrier()
        torch.cuda.synchronize()
        if g_one is not None:
            # W warm-up steps, then the K timed steps between two event nodes,
            # all in one graph: the first timed step follows a warm pipeline
            g, t0, t1 = g_one
            with torch.cuda.stream(stream):
                g.replay()
            torch.cuda.synchronize()
            barrier()
            ms = max_over_ranks(t0.elapsed_time(t1), dev)
            primed = ("holds the W warm-up steps and the K timed ones; the start event waits on a branch for the "
                      "last warm-up step, the end event follows the last timed step (one untimed replay first)")
        else:
            lead_in(stream)
            with torch.cuda.stream(stream):
                e0.record(stream)
                replay_steps(args.steps // G, g_rem)
                e1.record(stream)
            torch.cuda.synchronize()
            barrier()
            ms = max_over_ranks(e0.elapsed_time(e1), dev)
    clocks = clk.summary()

    # ---- roofline: the step's dominant kernel, live, over rotating copies.  For a
    # single-launch step that is the step's own kernel (reading the f32
    # activation); otherwise the product kernel.  The product kernel alone (a
    # pre-quantized activation) is timed too, as context.
    def time_launches(fn):
        n_roof = args.roof_launches
        g_roof = capture(fn, n_roof)
        with torch.cuda.stream(stream):
            g_roof.replay()
            e0.record(stream)
            for _ in range(3):
                g_roof.replay()
            e1.record(stream)
        stream.synchronize()
        return e0.elapsed_time(e1) / 1e3 / (3 * n_roof)

    prod_s = time_launches(gemv_only)
    per_launch_s = time_launches(step) if single else prod_s
    roof_bytes = (wbytes + 4 * K * ncols + 4 * rows * ncols) if single else abytes
    peak, peak_kind = measured_peaks()
    achieved = roof_bytes / per_launch_s / 1e9
    ops_per_step = 2 * rows * K * ncols
    traffic = traffic_for(args.workload)

    # ---- e2e: the C-ABI call with HOST buffers (q_matvec_host: x copied in, the
    # product, the result copied out, one call a step), copies inside the timed region
    xh = torch.from_numpy(x).pin_memory()
    oh = torch.empty((ncols, rows), dtype=torch.float32).pin_memory()
    scaling = qb.SUB32 if sub32 else qb.PERBLOCK
    wsh = torch.empty(qb.q_matvec_host_workspace_bytes(scaling, fmt, rows, K, ncols), dtype=torch.uint8, device=dev)
    n_e2e = min(args.steps, 3000)

    Wv = [W[j] for j in range(ncopy)]  # the rotating copies as tensors (indexing them is the bench's, not the call's)

    def host_step(i):
        qb.q_matvec_host(fmt, Wv[i % ncopy], rows, K, xh, oh, wsh, scaling=scaling, stream=stream)

    for i in range(5):
        host_step(i)
    stream.synchronize()
    barrier()
    t0 = time.perf_counter()
    for i in range(n_e2e):
        host_step(i)
    stream.synchronize()
    e2e_s = max_over_ranks(time.perf_counter() - t0, dev)

    assert qb.q_device_status() == qb.QB_OK
    step_s = ms / 1e3 / args.steps
    value = world * wbytes / step_s / 1e9
    res = {
        "metric": metric_for(args.workload),
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms / args.steps, 6),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "int8 codes x int8 codes, exact int32/int64, f32 rounding" if fmt != synth.FMT_F16 else "f16 x f16, f32",
        "data": "synthetic (seeded PCG64; the format's code/scale distributions); no trained weights",
        "config": {
            "workload": desc,
            "rows": rows, "K": K, "ncols": ncols,
            "format": synth.FORMAT_NAMES[fmt],
            "weight_bytes_per_step": wbytes,
            "l2": f"each step reads a different one of {ncopy} weight copies ({ncopy * wbytes / 2**20:.0f} MiB "
                  f"> 4x L2); no flush",
            "timing": f"CUDA graphs of {G} steps ({'q_matvec_sub32' if sub32 else 'q_matvec'}: activation "
                      f"quantization + product, "
                      f"{launches_per_step} launch(es) a step, programmatic dependent launch) replayed; "
                      f"CUDA events on the launching stream; the timed graph {primed}",
            "parallelism": "replicas" if world > 1 else "single GPU",
        },
        "rows_per_s": round(world * rows / step_s, 1),
        "tops": round(world * ops_per_step / step_s / 1e12, 3),
        "frac_of_8tbs": round(value / 8000.0, 4),
        "frac_of_measured_copy": round(value / peak, 4),
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
        "roofline": roofline(fmt, ncols, single, achieved, peak, peak_kind, traffic, roof_bytes, per_launch_s,
                             prod_s, abytes, ops_per_step, args.roof_launches, sub32, rows, K),
        "e2e": {
            "value": round(world * wbytes * n_e2e / e2e_s / 1e9, 2),
            "unit": "GB/s",
            "h2d_bytes_per_step": int(x.nbytes),
            "d2h_bytes_per_step": int(4 * rows * ncols),
            "steps": n_e2e,
            "how": "per step one q_matvec_host call through the binding (pinned x -> device, "
                   f"{'q_matvec_sub32' if sub32 else 'q_matvec'}, out -> pinned host, all on the stream); "
                   "host wall clock over all steps",
        },
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(fmt, rows, K, ncols, Wh, x, wbytes, budget_s=args.cpu_seconds,
                                           sub32=sub32)
    return res


# ---------------------------------------------------------------- the oracle on the host

def _oracle_threads():
    return max(1, os.cpu_count() or 1)


_POOL = None


def _pool(n):
    global _POOL
    if _POOL is None:
        import concurrent.futures as cf
        _POOL = cf.ThreadPoolExecutor(n)
    return _POOL


def oracle_pass(fmt, rows, K, Wh, x, nthreads, row_limit=None, sub32=False):
    """quantize + product over (a sample of) rows, rows split across threads
    (ctypes releases the GIL; the oracle is reentrant)."""
    import oracle
    r_end = rows if row_limit is None else min(rows, row_limit)
    ex = _pool(nthreads)
    if fmt == synth.FMT_F16:
        x16 = oracle.quantize_f16(x)
        W16 = Wh.view(np.uint16).reshape(rows, K)[:r_end]
        chunks = np.array_split(np.arange(r_end), nthreads)
        list(ex.map(lambda c: oracle.gemv_f16(np.ascontiguousarray(W16[c]), len(c), K, x16)
                    if len(c) else None, chunks))
        return r_end
    codes, m, e, _ = oracle.quantize_sub32(x) if sub32 else oracle.quantize_blocks(x, synth.BLOCK[fmt])
    out = np.zeros((x.shape[0], rows), np.float32)
    bounds = np.linspace(0, r_end, nthreads + 1).astype(int)
    prod = oracle.gemv_sub32 if sub32 else oracle.gemv
    list(ex.map(lambda i: prod(fmt, Wh, rows, K, codes, m, e, int(bounds[i]), int(bounds[i + 1]), out),
                range(nthreads)))
    return r_end


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else platform)."""
    import platform
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.processor() or platform.machine()


def cpu_baseline(fmt, rows, K, ncols, Wh, x, wbytes, budget_s=10.0, sub32=False):
    n = _oracle_threads()
    oracle_pass(fmt, rows, K, Wh, x, n, sub32=sub32)          # warm (also builds the oracle if needed)
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle_pass(fmt, rows, K, Wh, x, n, sub32=sub32)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    # single thread: passes over a sample of the rows, about a quarter of the budget
    r1 = max(1, rows // 16)
    reps1, t1 = 0, time.perf_counter()
    while True:
        oracle_pass(fmt, rows, K, Wh, x, 1, row_limit=r1, sub32=sub32)
        reps1 += 1
        el1 = time.perf_counter() - t1
        if el1 >= budget_s / 4:
            break
    rec = wbytes / rows
    return {"value": round(wbytes * reps / el / 1e9, 4), "unit": "GB/s", "cores": n, "kind": "oracle",
            "sample": f"{reps} full passes (quantize + all {rows} rows) in {el:.1f} s, rows split over {n} "
                      f"threads of the scalar C oracle",
            "single_thread": {"value": round(rec * r1 * reps1 / el1 / 1e9, 4), "unit": "GB/s",
                              "sample": f"{reps1} passes of quantize + the first {r1} rows on one thread "
                                        f"in {el1:.1f} s"},
            "cpu_model": cpu_model()}


def sampled_oracle_pass(mats, n, frac):
    """The oracle (quantize + product) over a fraction of the rows of every
    (fmt, rows, K, weights, activation, weight) entry of a step, the fraction
    for an entry being frac * weight (at most 1); returns the weight bytes
    processed."""
    done = 0
    for fmt, rows, K, W, x, wt in mats:
        r = max(1, min(rows, int(rows * frac * wt)))
        oracle_pass(fmt, rows, K, W, x, n, row_limit=r)
        done += synth.record_bytes(fmt, K) * r
    return done


def sampled_oracle_rate(mats, budget_s):
    """Weight GB/s of the oracle over repeated sampled passes of a step's
    matrices, about budget_s seconds of host work in all (the sample sized
    from a timed small pass); returns (GB/s, threads, description)."""
    n = _oracle_threads()
    t0 = time.perf_counter()
    sampled_oracle_pass(mats, n, 0.002)                    # warm (and builds the oracle)
    small = time.perf_counter() - t0
    frac = max(0.002, min(1.0, 0.002 * (budget_s / 5.0) / max(small, 1e-6)))
    done, reps, t0 = 0, 0, time.perf_counter()
    while True:
        done += sampled_oracle_pass(mats, n, frac)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    return done / el / 1e9, n, (f"{reps} passes over {frac:.3g} of the rows of each of the step's {len(mats)} matrix "
                                f"shapes (quantize + product), rows split over {n} threads of the scalar C oracle, "
                                f"{el:.1f} s")


def _ffn_host(rng_seed):
    """The FFN workload's three matrices and two activations, drawn on the host."""
    fmt, rows, K, drows, seed, desc = FFN["q6k_ffn_14336x4096"]
    rng = np.random.default_rng(rng_seed)
    Ws = [synth.pack(fmt, synth.draw(fmt, rng, r, k)) for r, k in ((rows, K), (rows, K), (drows, rows))]
    x = synth.draw_act(rng, 1, K)
    h = synth.draw_act(rng, 1, rows)
    return fmt, rows, K, drows, desc, Ws, x, h


def ffn_oracle_pass(fmt, rows, K, drows, Ws, x, h, n, frac=1.0):
    """The oracle over the FFN step: gate and up from x, down from h (a
    fraction of each matrix's rows when frac < 1)."""
    for W, r, k, a in ((Ws[0], rows, K, x), (Ws[1], rows, K, x), (Ws[2], drows, rows, h)):
        oracle_pass(fmt, r, k, W, a, n, row_limit=max(1, int(r * frac)))


def run_ffn(args, rank, world):
    """A step is the FFN block: q_matvec_many over gate and up (one launch),
    then q_matvec of down (K = 14336); the two calls are also timed alone."""
    import torch
    import block_quantized_weight_quantize_gb300 as qb

    fmt, rows, K, drows, desc, Ws, x, h = _ffn_host(2 + 1000 * rank)
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    sizes = [W.size for W in Ws]
    wbytes = int(sum(sizes))
    ncopy = max(2, -(-4 * L2_BYTES // wbytes))
    bufs = [[torch.from_numpy(W).to(dev) for W in Ws]]
    for _ in range(1, ncopy):
        bufs.append([w.clone() for w in bufs[0]])
    xd = torch.from_numpy(x).to(dev)
    hd = torch.from_numpy(h).to(dev)
    og = torch.empty((1, rows), dtype=torch.float32, device=dev)
    ou = torch.empty((1, rows), dtype=torch.float32, device=dev)
    od = torch.empty((1, drows), dtype=torch.float32, device=dev)
    ws = torch.empty(max(qb.q_matvec_workspace_bytes(fmt, k, 1) for k in (K, rows)), dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(dev)

    def gate_up(i, s):
        b = bufs[i % ncopy]
        qb.q_matvec_many(fmt, [b[0], b[1]], [rows, rows], K, xd, [og, ou], workspace=ws, stream=s)

    def down(i, s):
        qb.q_matvec(fmt, bufs[i % ncopy][2], drows, rows, hd, od, workspace=ws, stream=s)

    def step(i, s):
        gate_up(i, s)
        down(i, s)

    with torch.cuda.stream(stream):
        for i in range(3):
            step(i, stream)
    stream.synchronize()
    G = min(args.steps, 500)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)

    def time_graph(fn, steps, clocks=False):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            g.capture_begin()
            for i in range(G):
                fn(i, stream)
            g.capture_end()
        with torch.cuda.stream(stream):
            for _ in range(max(1, -(-args.warmup // G))):
                g.replay()
        stream.synchronize()
        sampler = ClockSampler(dev.index) if clocks else None
        if sampler:
            sampler.__enter__()
        barrier()
        torch.cuda.synchronize()
        lead_in(stream)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(max(1, steps // G)):
                g.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        barrier()
        if sampler:
            sampler.__exit__(None, None, None)
        return max_over_ranks(e0.elapsed_time(e1), dev) / (max(1, steps // G) * G), \
            (sampler.summary() if sampler else None)

    ms, clocks = time_graph(step, args.steps, clocks=True)
    ms_gu, _ = time_graph(gate_up, min(args.steps, 20000))
    ms_dn, _ = time_graph(down, min(args.steps, 20000))
    # e2e: pinned x and h in, the three outputs back, a step's calls through the binding
    xh = torch.from_numpy(x).pin_memory()
    hh = torch.from_numpy(h).pin_memory()
    ohs = [torch.empty((1, r), dtype=torch.float32).pin_memory() for r in (rows, rows, drows)]
    n_e2e = min(args.steps, 2000)
    barrier()
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for i in range(n_e2e):
            xd.copy_(xh, non_blocking=True)
            hd.copy_(hh, non_blocking=True)
            step(i, stream)
            for oh, o in zip(ohs, (og, ou, od)):
                oh.copy_(o, non_blocking=True)
    stream.synchronize()
    e2e_s = max_over_ranks(time.perf_counter() - t0, dev)
    assert qb.q_device_status() == qb.QB_OK
    step_s = ms / 1e3
    value = world * wbytes / step_s / 1e9
    peak, peak_kind = measured_peaks()
    gu_bytes = sizes[0] + sizes[1] + 4 * K + 8 * rows
    two = False  # Q6_K-like down: the single-launch form (q_matvec's rule)
    res = {
        "metric": metric_for(args.workload),
        "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": max(1, args.steps // G) * G,
        "warmup": args.warmup, "ms_per_step": round(ms, 6), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int8 codes x int8 codes, exact int32/int64, f32 rounding",
        "data": "synthetic (seeded PCG64; the format's code/scale distributions); no trained weights",
        "config": {"workload": desc, "gate_up_rows": [rows, rows], "K": K, "down": [drows, rows], "ncols": 1,
                   "format": synth.FORMAT_NAMES[fmt], "weight_bytes_per_step": wbytes,
                   "l2": f"each step reads a different one of {ncopy} copies of the three matrices "
                         f"({ncopy * wbytes / 2**20:.0f} MiB > 4x L2); no flush",
                   "timing": f"CUDA graphs of {G} steps (two launches a step, programmatic dependent launch); "
                             f"CUDA events",
                   "gate_up_ms": round(ms_gu, 6), "down_ms": round(ms_dn, 6),
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "rows_per_s": round(world * (2 * rows + drows) / step_s, 1),
        "frac_of_8tbs": round(value / 8000.0, 4), "frac_of_measured_copy": round(value / peak, 4),
        "gpu_launches": max(1, args.steps // G) * G * (3 if two else 2), "clocks": clocks,
        "roofline": {"bound": "hbm",
                     "kernel": "gemv6_kernel<q6k, one column, single launch, grouped> (gate + up, 28672 rows)",
                     "achieved": round(gu_bytes / (ms_gu / 1e3) / 1e9, 1), "peak": peak,
                     "peak_kind": f"{peak_kind} (HBM copy, burst)", "unit": "GB/s",
                     "frac": round(gu_bytes / (ms_gu / 1e3) / 1e9 / peak, 4), "traffic": traffic_for(args.workload),
                     "algorithmic_bytes_per_launch": gu_bytes, "avg_launch_us": round(ms_gu * 1e3, 4),
                     "down_kernel": "gemv3_kernel<q6k, one column, single launch> (4096 x 14336)",
                     "down_achieved": round((sizes[2] + 4 * rows + 4 * drows) / (ms_dn / 1e3) / 1e9, 1)},
        "e2e": {"value": round(world * wbytes * n_e2e / e2e_s / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": int(x.nbytes + h.nbytes), "d2h_bytes_per_step": int(4 * (2 * rows + drows)),
                "steps": n_e2e,
                "how": "per step: pinned x and h -> device, q_matvec_many + q_matvec through the Python binding, "
                       "the three outputs -> pinned host; host wall clock over all steps"},
    }
    if rank == 0 and not args.no_cpu_baseline:
        n = _oracle_threads()
        ffn_oracle_pass(fmt, rows, K, drows, Ws, x, h, n)
        reps, t0 = 0, time.perf_counter()
        while True:
            ffn_oracle_pass(fmt, rows, K, drows, Ws, x, h, n)
            reps += 1
            el = time.perf_counter() - t0
            if el >= args.cpu_seconds:
                break
        res["cpu_baseline"] = {"value": round(wbytes * reps / el / 1e9, 4), "unit": "GB/s", "cores": n,
                               "kind": "oracle",
                               "sample": f"{reps} full FFN steps (quantize x and h, all rows of gate, up and down) "
                                         f"in {el:.1f} s, rows split over {n} threads of the scalar C oracle"}
    return res


def run_ffn_reference(args):
    """The reference arm on the FFN workload: the oracle over whole FFN steps."""
    fmt, rows, K, drows, desc, Ws, x, h = _ffn_host(2)
    wbytes = int(sum(W.size for W in Ws))
    n = _oracle_threads()
    t0 = time.perf_counter()
    ffn_oracle_pass(fmt, rows, K, drows, Ws, x, h, n)
    full = time.perf_counter() - t0
    frac = max(1e-4, min(1.0, (100.0 / max(1, args.steps + args.warmup)) / max(full, 1e-6)))
    for _ in range(args.warmup):
        ffn_oracle_pass(fmt, rows, K, drows, Ws, x, h, n, frac)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        ffn_oracle_pass(fmt, rows, K, drows, Ws, x, h, n, frac)
    el = time.perf_counter() - t0
    done = sum(synth.record_bytes(fmt, k) * max(1, int(r * frac)) for r, k in ((rows, K), (rows, K), (drows, rows)))
    value = done * args.steps / el / 1e9
    sample = (f"each step: quantize x and h + {frac:.3g} of the rows of gate, up and down, split over {n} threads "
              f"of the scalar C oracle")
    return {
        "impl": "reference", "metric": metric_for(args.workload),
        "value": round(value, 4), "unit": "GB/s", "n_gpus": 0, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(el * 1e3 / args.steps, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int64/int128 exact, f32 rounding (scalar C)",
        "data": "synthetic (seeded PCG64)",
        "config": {"workload": desc, "gate_up_rows": [rows, rows], "K": K, "down": [drows, rows], "ncols": 1,
                   "weight_bytes_per_step": wbytes},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": n, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def _stack_host(ncols, seed):
    """The stack's drawn matrices on the host (one per shape, and the first
    eighth of the output matrix, which the device tiles eight times) and its
    two activations, in the draw order the bench uses."""
    rng = np.random.default_rng(seed)
    hmats = [synth.pack(fmt, synth.draw(fmt, rng, rows, K)) for _, fmt, rows, K in STACK_MATS]
    _, ofmt, orows, oK = STACK_OUT
    Wo = synth.pack(ofmt, synth.draw(ofmt, rng, orows // 8, oK))
    xh = {k: synth.draw_act(rng, ncols, k) for k in (4096, 14336)}
    return hmats, Wo, xh


def _stack_oracle_mats(hmats, Wo, xh):
    """The stack's matrices for the sampled oracle, each weighted by how often
    a step reads it: the layer shapes 1 (32 times a step), the output
    matrix's drawn eighth 8/32 (8 times a step), so a pass has the step's mix
    of bytes."""
    _, ofmt, orows, oK = STACK_OUT
    mats = [(fmt, rows, K, W, xh[K], 1.0) for (_, fmt, rows, K), W in zip(STACK_MATS, hmats)]
    mats.append((ofmt, orows // 8, oK, Wo, xh[oK], 8.0 / STACK_LAYERS))
    return mats


def run_stack(args, rank, world):
    """One step = the 129 products of an 8B-class decode step (every layer's
    weights its own copy in HBM, 4.36 GB in all), each a q_matvec call from
    its f32 activation; the first and the last take host buffers
    (q_matvec_host), so the step runs from a host activation to host logits."""
    import torch
    import block_quantized_weight_quantize_gb300 as qb

    ncols = STACK[args.workload]
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    hmats, Wo, xhost = _stack_host(ncols, 9 + 1000 * rank)
    mats = []  # (name, fmt, rows, K, device weights per layer)
    for (name, fmt, rows, K), Wh in zip(STACK_MATS, hmats):
        w0 = torch.from_numpy(Wh).to(dev)
        layers = [w0] + [w0.clone() for _ in range(STACK_LAYERS - 1)]
        mats.append((name, fmt, rows, K, layers))
    oname, ofmt, orows, oK = STACK_OUT
    wo = torch.empty(orows * synth.record_bytes(ofmt, oK), dtype=torch.uint8, device=dev)
    for i in range(8):
        wo[i * Wo.size:(i + 1) * Wo.size].copy_(torch.from_numpy(Wo))
    wbytes = sum(synth.weight_bytes(f, r, k) for _, f, r, k in STACK_MATS) * STACK_LAYERS + \
        synth.weight_bytes(ofmt, orows, oK)
    xs = {k: torch.from_numpy(v).to(dev) for k, v in xhost.items()}
    outs = {name: torch.empty((ncols, rows), dtype=torch.float32, device=dev) for name, _, rows, _, _ in mats}
    logits = torch.empty((ncols, orows), dtype=torch.float32, device=dev)
    wsb = max(qb.q_matvec_workspace_bytes(f, k, ncols) for _, f, _, k in STACK_MATS + [STACK_OUT])
    ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(dev)
    # q_matvec launches a call: one for a single column (except Q4_K-like at
    # K >= 12288 given a workspace: quantize, then the product) and for 2..4
    # columns at K = 4096 where the warp-per-block kernels take the rows, two
    # otherwise
    calls = [(f, r, k) for _, f, r, k in STACK_MATS] * STACK_LAYERS + [(STACK_OUT[1], STACK_OUT[2], STACK_OUT[3])]

    def one_launch(f, r, k):
        if ncols == 1:
            return not (f == synth.FMT_Q4K and k >= 12288)
        return 2 <= ncols <= 4 and k == 4096 and multi_col_kernel(f, r, k, ncols).startswith(("gemv7m", "gemv7r"))

    launches_step = sum(1 if one_launch(f, r, k) else 2 for f, r, k in calls)

    def step(i, s):
        for layer in range(STACK_LAYERS):
            for name, fmt, rows, K, layers in mats:
                qb.q_matvec(fmt, layers[layer], rows, K, xs[K], outs[name], workspace=ws, stream=s)
        qb.q_matvec(ofmt, wo, orows, oK, xs[oK], logits, workspace=ws, stream=s)

    with torch.cuda.stream(stream):
        step(0, stream)
    stream.synchronize()
    G = max(1, min(args.steps, 5))

    def capture(fn, n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            g.capture_begin()
            for i in range(n):
                fn(i, stream)
            g.capture_end()
        return g

    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    g_main = capture(step, G)
    with torch.cuda.stream(stream):
        for _ in range(max(1, -(-args.warmup // G))):
            g_main.replay()
    stream.synchronize()
    nrep = max(1, args.steps // G)
    with ClockSampler(dev.index) as clk:
        barrier()
        torch.cuda.synchronize()
        lead_in(stream)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(nrep):
                g_main.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        barrier()
    ms = max_over_ranks(e0.elapsed_time(e1), dev) / (nrep * G)
    clocks = clk.summary()
    # e2e: host activation in (the first call), host logits out (the last)
    xh = torch.from_numpy(synth.draw_act(np.random.default_rng(10), ncols, 4096)).pin_memory()
    lh = torch.empty((ncols, orows), dtype=torch.float32).pin_memory()
    f0, r0, k0 = mats[0][1], mats[0][2], mats[0][3]
    wsh0 = torch.empty(qb.q_matvec_host_workspace_bytes(qb.PERBLOCK, f0, r0, k0, ncols), dtype=torch.uint8, device=dev)
    wsh1 = torch.empty(qb.q_matvec_host_workspace_bytes(qb.PERBLOCK, ofmt, orows, oK, ncols), dtype=torch.uint8,
                       device=dev)

    qkv_host = torch.empty((ncols, mats[0][2]), dtype=torch.float32).pin_memory()

    def host_step():
        for layer in range(STACK_LAYERS):
            for j, (name, fmt, rows, K, layers) in enumerate(mats):
                if layer == 0 and j == 0:  # the step's input arrives from the host
                    qb.q_matvec_host(fmt, layers[0], rows, K, xh, qkv_host, wsh0, stream=stream)
                else:
                    qb.q_matvec(fmt, layers[layer], rows, K, xs[K], outs[name], workspace=ws, stream=stream)
        qb.q_matvec_host(ofmt, wo, orows, oK, xh, lh, wsh1, stream=stream)  # logits back to the host

    host_step()
    stream.synchronize()
    n_e2e = max(3, min(args.steps, 20))
    barrier()
    t0 = time.perf_counter()
    for _ in range(n_e2e):
        host_step()
    stream.synchronize()
    e2e_s = max_over_ranks(time.perf_counter() - t0, dev)
    assert qb.q_device_status() == qb.QB_OK
    step_s = ms / 1e3
    value = world * wbytes / step_s / 1e9
    peak, peak_kind = measured_peaks()
    nrows = sum(r for _, _, r, _ in STACK_MATS) * STACK_LAYERS + orows
    ops = 2 * ncols * (sum(r * k for _, _, r, k in STACK_MATS) * STACK_LAYERS + orows * oK)
    res = {
        "metric": metric_for(args.workload),
        "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": nrep * G, "warmup": args.warmup,
        "ms_per_step": round(ms, 6), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "int8 codes x int8 codes, exact int32/int64, f32 rounding",
        "data": "synthetic (seeded PCG64; the formats' code/scale distributions; one drawn copy per matrix shape, "
                "each layer its own device copy, the output matrix drawn as 1/8 and tiled); no trained weights",
        "config": {"workload": f"8B-class decode stack, {ncols} column(s)", "layers": STACK_LAYERS,
                   "matrices": [[n, synth.FORMAT_NAMES[f], r, k] for n, f, r, k in STACK_MATS + [STACK_OUT]],
                   "ncols": ncols, "weight_bytes_per_step": wbytes,
                   "l2": "every layer reads its own weights (4.36 GB a step, 34x L2); no flush",
                   "timing": f"CUDA graphs of {G} steps ({launches_step} launches a step, "
                             f"programmatic dependent launch); CUDA events",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "rows_per_s": round(world * nrows / step_s, 1), "tokens_per_s": round(world * ncols / step_s, 1),
        "tops": round(world * ops / step_s / 1e12, 3),
        "frac_of_8tbs": round(value / 8000.0, 4), "frac_of_measured_copy": round(value / peak, 4),
        "gpu_launches": nrep * G * launches_step, "clocks": clocks,
        "roofline": {"bound": "hbm" if ncols == 1 else "alu", "kernel": "the step's 129 products (one-column "
                     "streaming kernels at 1 column; at 4 the warp-per-block kernel for QKV and O, its ring form "
                     "for gate+up and the K = 14336 down projection, the dp4a kernel for the Q6_K-like output; "
                     "the tcgen05 tensor-core kernel at 16, the dp4a kernel for the down projection)",
                     "achieved": round(value, 1) if ncols == 1 else round(ops / step_s / 1e12, 2),
                     "peak": peak if ncols == 1 else round(DP4A_PEAK_TOPS, 1),
                     "peak_kind": f"{peak_kind} (HBM copy, burst)" if ncols == 1 else
                                  "dp4a issue rate from unit counts and the maximum clock",
                     "unit": "GB/s" if ncols == 1 else "TOPS",
                     "frac": round(value / peak, 4) if ncols == 1 else round(ops / step_s / 1e12 / DP4A_PEAK_TOPS, 4),
                     "traffic": None, "algorithmic_bytes_per_step": wbytes},
        "e2e": {"value": round(world * wbytes * n_e2e / e2e_s / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": int(xh.numel() * 4), "d2h_bytes_per_step": int(lh.numel() * 4),
                "steps": n_e2e, "how": "per step the 129 calls through the binding, the first (QKV) and the last "
                "(output) q_matvec_host with pinned host buffers; host wall clock"},
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, n, sample = sampled_oracle_rate(_stack_oracle_mats(hmats, Wo, xhost), args.cpu_seconds)
        res["cpu_baseline"] = {"value": round(v, 4), "unit": "GB/s", "cores": n, "kind": "oracle", "sample": sample}
    return res


def run_stack_reference(args):
    """The reference arm on the stack: the oracle over sampled rows of the
    step's matrices (the layer shapes and the output matrix in the step's mix
    of bytes), each step's sample sized so the run stays within ~2 minutes."""
    ncols = STACK[args.workload]
    hmats, Wo, xhost = _stack_host(ncols, 9)
    mats = _stack_oracle_mats(hmats, Wo, xhost)
    n = _oracle_threads()
    t0 = time.perf_counter()
    sampled_oracle_pass(mats, n, 0.002)
    small = time.perf_counter() - t0
    frac = max(0.002, min(1.0, 0.002 * (100.0 / max(1, args.steps + args.warmup)) / max(small, 1e-6)))
    for _ in range(args.warmup):
        sampled_oracle_pass(mats, n, frac)
    done, t0 = 0, time.perf_counter()
    for _ in range(args.steps):
        done += sampled_oracle_pass(mats, n, frac)
    el = time.perf_counter() - t0
    value = done / el / 1e9
    sample = (f"each step: {frac:.3g} of the rows of every layer shape and 8/32 of that of the output matrix's "
              f"drawn eighth ({ncols} column(s), quantize + product), split over {n} threads of the scalar C oracle")
    return {
        "impl": "reference",
        "metric": metric_for(args.workload),
        "value": round(value, 4), "unit": "GB/s", "n_gpus": 0, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(el * 1e3 / args.steps, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int64/int128 exact, f32 rounding (scalar C)",
        "data": "synthetic (seeded PCG64)",
        "config": {"workload": f"8B-class decode stack, {ncols} column(s)", "layers": STACK_LAYERS,
                   "matrices": [[nm, synth.FORMAT_NAMES[f], r, k] for nm, f, r, k in STACK_MATS + [STACK_OUT]],
                   "ncols": ncols},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": n, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def _fp8_inputs(rows, K, ncols, seed):
    rng = np.random.default_rng(seed)
    W = rng.integers(0, 256, size=(rows, K), dtype=np.uint8)
    W[(W & 0x7F) == 0x7F] = 0x3C  # no NaN codes
    scales = (2.0 ** rng.uniform(-12, -4, size=((rows + 127) // 128, (K + 127) // 128))).astype(np.float32)
    x = rng.standard_normal((ncols, K)).astype(np.float32)
    return W, scales, x


def run_fp8(args, rank, world):
    """A step is one q_gemv_fp8 over the matrix (weights streamed from HBM)."""
    import torch
    import block_quantized_weight_quantize_gb300 as qb

    rows, K, ncols, seed, desc = FP8[args.workload]
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    Wh, sh, x = _fp8_inputs(rows, K, ncols, seed + 1000 * rank)
    wbytes = rows * K + sh.nbytes
    ncopy = max(2, -(-4 * L2_BYTES // wbytes))
    W = torch.empty((ncopy, rows, K), dtype=torch.uint8, device=dev)
    W[0].copy_(torch.from_numpy(Wh))
    for i in range(1, ncopy):
        W[i].copy_(W[0])
    sd = torch.from_numpy(sh).to(dev)
    xd = torch.from_numpy(x).to(dev)
    out = torch.empty((ncols, rows), dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(dev)

    def step(i, s):
        qb.q_gemv_fp8(W[i % ncopy], sd, rows, K, xd, out, stream=s)

    with torch.cuda.stream(stream):
        for i in range(3):
            step(i, stream)
    stream.synchronize()
    G = min(args.steps, 1000)

    def capture(fn, n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            g.capture_begin()
            for i in range(n):
                fn(i, stream)
            g.capture_end()
        return g

    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    g_main = capture(step, G)
    g_w = capture(step, max(1, min(args.warmup, G)))
    with torch.cuda.stream(stream):
        for _ in range(max(1, args.warmup // max(1, min(args.warmup, G)))):
            g_w.replay()
    stream.synchronize()
    primed = prime_graph(g_main, stream)
    nrep = max(1, args.steps // G)
    with ClockSampler(dev.index) as clk:
        barrier()
        torch.cuda.synchronize()
        lead_in(stream)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(nrep):
                g_main.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        barrier()
    ms = max_over_ranks(e0.elapsed_time(e1), dev) / (nrep * G)
    clocks = clk.summary()
    # e2e: x from pinned host memory, the outputs back
    xh = torch.from_numpy(x).pin_memory()
    oh = torch.empty((ncols, rows), dtype=torch.float32).pin_memory()
    n_e2e = min(args.steps, 3000)
    barrier()
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for i in range(n_e2e):
            xd.copy_(xh, non_blocking=True)
            step(i, stream)
            oh.copy_(out, non_blocking=True)
    stream.synchronize()
    e2e_s = max_over_ranks(time.perf_counter() - t0, dev)
    assert qb.q_device_status() == qb.QB_OK
    step_s = ms / 1e3
    value = world * wbytes / step_s / 1e9
    peak, peak_kind = measured_peaks()
    roof_bytes = wbytes + 4 * K * ncols + 4 * rows * ncols
    ops = 2 * rows * K * ncols
    cmax = 16  # columns a launch: the staged activation stays within 200 KB (as the library splits them)
    while cmax > 1 and cmax * ((K // 16 + 31) // 32) * 2048 > 200 * 1024:
        cmax //= 2
    launches = -(-ncols // cmax)
    res = {
        "metric": metric_for(args.workload), "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": nrep * G, "warmup": args.warmup, "ms_per_step": round(ms, 6), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3 weights decoded to f32, f32 x, f32 FMA",
        "data": "synthetic (seeded PCG64: uniform E4M3 codes without NaN, log-uniform 2^-12..2^-4 block scales, "
                "N(0,1) activations)",
        "config": {"workload": desc, "rows": rows, "K": K, "ncols": ncols, "weight_bytes_per_step": wbytes,
                   "l2": f"each step reads a different one of {ncopy} weight copies "
                         f"({ncopy * wbytes / 2**20:.0f} MiB > 4x L2); no flush",
                   "timing": f"CUDA graphs of {G} steps, one q_gemv_fp8 launch a step; CUDA events; "
                             f"the timed graph {primed}",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "rows_per_s": round(world * rows / step_s, 1), "tops": round(world * ops / step_s / 1e12, 3),
        "frac_of_8tbs": round(value / 8000.0, 4), "frac_of_measured_copy": round(value / peak, 4),
        "gpu_launches": nrep * G * launches, "clocks": clocks,
        "roofline": {"bound": "hbm", "kernel": f"gemv_fp8_kernel ({ncols} columns in {launches} launch(es))",
                     "achieved": round(roof_bytes / step_s / 1e9, 1), "peak": peak,
                     "peak_kind": f"{peak_kind} (HBM copy, burst)", "unit": "GB/s",
                     "frac": round(roof_bytes / step_s / 1e9 / peak, 4), "traffic": traffic_for(args.workload),
                     "algorithmic_bytes_per_launch": roof_bytes, "avg_launch_us": round(ms * 1e3, 4)},
        "e2e": {"value": round(world * wbytes * n_e2e / e2e_s / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": int(x.nbytes), "d2h_bytes_per_step": int(4 * rows * ncols), "steps": n_e2e,
                "how": "per step: pinned x -> device, q_gemv_fp8 through the binding, out -> pinned host"},
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = fp8_cpu_baseline(rows, K, Wh, sh, x, wbytes, args.cpu_seconds)
    return res


def fp8_oracle_pass(rows, K, Wh, sh, x, nthreads, row_limit=None):
    import oracle
    r_end = rows if row_limit is None else min(rows, row_limit)
    ex = _pool(nthreads)
    bounds = np.linspace(0, r_end, nthreads + 1).astype(int)

    def one(i):
        a, b = int(bounds[i]), int(bounds[i + 1])
        a0 = a // 128 * 128  # whole scale blocks: the oracle indexes scales from the first row it gets
        if b > a:
            oracle.gemv_fp8(Wh[a0:b], sh[a0 // 128:], b - a0, K, x)
    list(ex.map(one, range(nthreads)))
    return r_end


def fp8_cpu_baseline(rows, K, Wh, sh, x, wbytes, budget_s=10.0):
    n = _oracle_threads()
    t0 = time.perf_counter()
    fp8_oracle_pass(rows, K, Wh, sh, x, n, 256)
    per = (time.perf_counter() - t0) / 256
    R = int(max(128, min(rows, budget_s / 3 / max(per, 1e-9))))
    reps, t0 = 0, time.perf_counter()
    while True:
        fp8_oracle_pass(rows, K, Wh, sh, x, n, R)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    return {"value": round(wbytes * (R / rows) * reps / el / 1e9, 4), "unit": "GB/s", "cores": n, "kind": "oracle",
            "sample": f"{reps} passes over {R} of {rows} rows in {el:.1f} s, rows over {n} threads of the scalar C "
                      f"oracle (decode, dequantize, dot in double)"}


def kv_oracle_pass(scaling, nh, nkv, d, L, q, k, nthreads, pos_limit=None):
    """cache rows + query heads + scores of (a sample of) positions with the oracle, key heads over threads."""
    import oracle
    P = L if pos_limit is None else min(L, pos_limit)
    qc, m, e = oracle.quantize_heads(scaling, q)
    G = nh // nkv
    ex = _pool(nthreads)

    def one(h):
        kc, ks = oracle.cache_rows(k[h * L:h * L + P])
        oracle.kv_scores(scaling, qc[h * G:(h + 1) * G], m[h * G:(h + 1) * G], e[h * G:(h + 1) * G], d,
                         kc.reshape(1, P, d), ks.reshape(1, P), P, 1, 0.125)
    list(ex.map(one, range(nkv)))
    return P


def kv_cpu_baseline(scaling, nh, nkv, d, L, q, k, kbytes, budget_s=10.0):
    n = _oracle_threads()
    t0 = time.perf_counter()
    kv_oracle_pass(scaling, nh, nkv, d, L, q, k, n, 512)
    per = (time.perf_counter() - t0) / 512
    P = int(max(256, min(L, budget_s / 3 / max(per, 1e-9))))
    reps, t0 = 0, time.perf_counter()
    while True:
        kv_oracle_pass(scaling, nh, nkv, d, L, q, k, n, P)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    value = kbytes * (P / L) * reps / el / 1e9
    return {"value": round(value, 4), "unit": "GB/s", "cores": n, "kind": "oracle",
            "sample": f"{reps} passes over {P} of {L} positions of every key head (cache rows, query heads, "
                      f"scores) in {el:.1f} s, key heads over {n} threads of the scalar C oracle"}


def run_kv_reference(args):
    scaling, nh, nkv, d, L, seed, desc = KV[args.workload]
    q, k = _kv_inputs(scaling, nh, nkv, d, L, seed)
    n = _oracle_threads()
    kbytes = nkv * L * (d + 2)
    t0 = time.perf_counter()
    kv_oracle_pass(scaling, nh, nkv, d, L, q, k, n, 1024)
    per = (time.perf_counter() - t0) / 1024
    budget = 100.0 / max(1, args.steps + args.warmup)
    P = int(max(64, min(L, budget / max(per, 1e-9))))
    for _ in range(args.warmup):
        kv_oracle_pass(scaling, nh, nkv, d, L, q, k, n, P)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        kv_oracle_pass(scaling, nh, nkv, d, L, q, k, n, P)
    el = time.perf_counter() - t0
    value = kbytes * (P / L) * args.steps / el / 1e9
    sample = f"each step: cache rows, query heads and scores of {P} of {L} positions, key heads over {n} threads"
    return {
        "impl": "reference", "metric": metric_for(args.workload), "value": round(value, 4), "unit": "GB/s",
        "n_gpus": 0, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el * 1e3 / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "int64 exact, f32 rounding (scalar C)", "data": "synthetic (seeded PCG64)",
        "config": {"workload": desc, "query_heads": nh, "key_heads": nkv, "head": d, "positions": L},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": n, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_fp8_reference(args):
    rows, K, ncols, seed, desc = FP8[args.workload]
    Wh, sh, x = _fp8_inputs(rows, K, ncols, seed)
    n = _oracle_threads()
    wbytes = rows * K + sh.nbytes
    t0 = time.perf_counter()
    fp8_oracle_pass(rows, K, Wh, sh, x, n, 256)
    per = (time.perf_counter() - t0) / 256
    budget = 100.0 / max(1, args.steps + args.warmup)
    R = int(max(128, min(rows, budget / max(per, 1e-9))))
    for _ in range(args.warmup):
        fp8_oracle_pass(rows, K, Wh, sh, x, n, R)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        fp8_oracle_pass(rows, K, Wh, sh, x, n, R)
    el = time.perf_counter() - t0
    value = wbytes * (R / rows) * args.steps / el / 1e9
    sample = f"each step: {R} of {rows} rows, over {n} threads of the scalar C oracle"
    return {
        "impl": "reference", "metric": metric_for(args.workload), "value": round(value, 4), "unit": "GB/s",
        "n_gpus": 0, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el * 1e3 / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64 dot (scalar C)",
        "data": "synthetic (seeded PCG64)", "config": {"workload": desc, "rows": rows, "K": K, "ncols": ncols},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": n, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_reference(args):
    fmt, rows, K, ncols, seed, outl, desc = WORKLOADS[args.workload]
    sub32 = args.workload in SUB32
    rng = np.random.default_rng(seed)
    lg = synth.draw(fmt, rng, rows, K)
    Wh = synth.pack(fmt, lg)
    x = synth.draw_act(rng, ncols, K, outlier_frac=outl)
    n = _oracle_threads()
    # size each step's row sample so the whole run stays within ~2 minutes
    t0 = time.perf_counter()
    oracle_pass(fmt, rows, K, Wh, x, n, sub32=sub32)
    full = time.perf_counter() - t0
    budget = 100.0 / max(1, args.steps + args.warmup)
    rows_s = int(max(1, min(rows, rows * budget / max(full, 1e-6))))
    for _ in range(args.warmup):
        oracle_pass(fmt, rows, K, Wh, x, n, rows_s, sub32=sub32)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_pass(fmt, rows, K, Wh, x, n, rows_s, sub32=sub32)
    el = time.perf_counter() - t0
    rec = synth.record_bytes(fmt, K)
    value = rec * rows_s * args.steps / el / 1e9
    sample = f"each step: quantize + {rows_s} of {rows} rows, split over {n} threads of the scalar C oracle"
    return {
        "impl": "reference",
        "metric": metric_for(args.workload),
        "value": round(value, 4), "unit": "GB/s", "n_gpus": 0, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(el * 1e3 / args.steps, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int64/int128 exact, f32 rounding (scalar C)",
        "data": "synthetic (seeded PCG64)", "config": {"workload": desc, "rows": rows, "K": K, "ncols": ncols},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": n, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }

# ---------------------------------------------------------------- two-word activation codes

def _w2_inputs(fmt, rows, K, ncols, seed):
    rng = np.random.default_rng(seed)
    Wh = synth.pack(fmt, synth.draw(fmt, rng, rows, K))
    nb = K // synth.BLOCK[fmt]
    a16 = rng.integers(-32768, 32768, (ncols, K)).astype(np.int16)
    m = rng.integers(128, 256, (ncols, nb)).astype(np.uint8)
    e = rng.integers(-40, -10, (ncols, nb)).astype(np.int16)
    return Wh, a16, m, e


def _w2_packed(m, e):
    return (m.astype(np.uint32) | (e.astype(np.int32).astype(np.uint32) << 16)).view(np.int32)


def w2_oracle_pass(fmt, rows, K, Wh, a16, m, e, nthreads, row_limit=None):
    import oracle
    r_end = rows if row_limit is None else min(rows, row_limit)
    out = np.zeros((a16.shape[0], rows), np.float32)
    bounds = np.linspace(0, r_end, nthreads + 1).astype(int)
    list(_pool(nthreads).map(lambda i: oracle.gemv_w2(fmt, Wh, rows, K, a16, m, e, int(bounds[i]),
                                                       int(bounds[i + 1]), out), range(nthreads)))
    return r_end


def run_w2(args, rank, world):
    """A step is one q_gemv_w2 call: the matrix times a two-word activation."""
    import torch
    import block_quantized_weight_quantize_gb300 as qb

    fmt, rows, K, ncols, seed, desc = W2[args.workload]
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    Wh, a16, m, e = _w2_inputs(fmt, rows, K, ncols, seed + 1000 * rank)
    wbytes = synth.weight_bytes(fmt, rows, K)
    ncopy = max(2, -(-4 * L2_BYTES // wbytes))
    W = torch.empty((ncopy, Wh.size), dtype=torch.uint8, device=dev)
    W[0].copy_(torch.from_numpy(Wh))
    for i in range(1, ncopy):
        W[i].copy_(W[0])
    ad = torch.from_numpy(a16).to(dev)
    sd = torch.from_numpy(_w2_packed(m, e)).to(dev)
    out = torch.empty((ncols, rows), dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(dev)

    def step(i, s):
        qb.q_gemv_w2(fmt, W[i % ncopy], rows, K, ad, sd, ncols, out, s)

    with torch.cuda.stream(stream):
        for i in range(3):
            step(i, stream)
    stream.synchronize()
    g_one = one_graph_timing(capture_steps=lambda n0, n: [step(n0 + i, stream) for i in range(n)],
                             stream=stream, warmup=args.warmup, steps=min(args.steps, 1000))
    steps = min(args.steps, 1000)
    if g_one is None:  # no event nodes in this torch: one graph of the steps between two stream events
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            g.capture_begin()
            for i in range(steps):
                step(i, stream)
            g.capture_end()
            g.replay()
        stream.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index) as clk:
        barrier()
        torch.cuda.synchronize()
        if g_one is not None:
            g, t0, t1 = g_one
            with torch.cuda.stream(stream):
                g.replay()
        else:
            with torch.cuda.stream(stream):
                t0.record(stream)
                g.replay()
                t1.record(stream)
        torch.cuda.synchronize()
        barrier()
        ms = max_over_ranks(t0.elapsed_time(t1), dev)
    clocks = clk.summary()
    step_s = ms / 1e3 / steps
    # e2e: host codes in, the call, host result out, one step at a time on the stream
    ah = torch.from_numpy(a16).pin_memory()
    oh = torch.empty((ncols, rows), dtype=torch.float32).pin_memory()
    n_e2e = min(steps, 2000)
    barrier()
    t0h = time.perf_counter()
    with torch.cuda.stream(stream):
        for i in range(n_e2e):
            ad.copy_(ah, non_blocking=True)
            step(i, stream)
            oh.copy_(out, non_blocking=True)
    stream.synchronize()
    e2e_s = max_over_ranks(time.perf_counter() - t0h, dev)
    assert qb.q_device_status() == qb.QB_OK
    peak, peak_kind = measured_peaks()
    roof_bytes = wbytes + 2 * K * ncols + 4 * (K // synth.BLOCK[fmt]) * ncols + 4 * rows * ncols
    value = world * wbytes / step_s / 1e9
    res = {
        "metric": metric_for(args.workload), "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": steps, "warmup": args.warmup, "ms_per_step": round(ms / steps, 6), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "int8 codes x 16-bit codes (two words), exact int64/int128, "
                                                          "f32 rounding",
        "data": "synthetic (seeded PCG64; 16-bit codes uniform over their range, m in 128..255, e in -40..-11)",
        "config": {"workload": desc, "rows": rows, "K": K, "ncols": ncols, "format": synth.FORMAT_NAMES[fmt],
                   "weight_bytes_per_step": wbytes,
                   "l2": f"each step reads a different one of {ncopy} weight copies; no flush",
                   "timing": f"CUDA graph of {steps} q_gemv_w2 steps (one launch each); CUDA events",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "rows_per_s": round(world * rows / step_s, 1),
        "frac_of_8tbs": round(value / 8000.0, 4), "frac_of_measured_copy": round(value / peak, 4),
        "gpu_launches": steps, "clocks": clocks,
        "roofline": {"bound": "hbm", "kernel": f"w2_kernel<{synth.FORMAT_NAMES[fmt]}> (a warp a row, lanes over "
                                               "blocks, per-word dp4a sums)",
                     "achieved": round(roof_bytes / step_s / 1e9, 1), "peak": peak,
                     "peak_kind": f"{peak_kind} (HBM copy, burst)", "unit": "GB/s",
                     "frac": round(roof_bytes / step_s / 1e9 / peak, 4), "traffic": traffic_for(args.workload),
                     "algorithmic_bytes_per_launch": roof_bytes, "avg_launch_us": round(step_s * 1e6, 4)},
        "e2e": {"value": round(world * wbytes * n_e2e / e2e_s / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": int(a16.nbytes), "d2h_bytes_per_step": int(4 * rows * ncols),
                "steps": n_e2e, "how": "per step: the codes copied from pinned host memory, q_gemv_w2, the result "
                                       "copied back to pinned host memory, all on the stream; host wall clock"},
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        n = _oracle_threads()
        w2_oracle_pass(fmt, rows, K, Wh, a16, m, e, n)
        reps, t0c = 0, time.perf_counter()
        while True:
            w2_oracle_pass(fmt, rows, K, Wh, a16, m, e, n)
            reps += 1
            el = time.perf_counter() - t0c
            if el >= args.cpu_seconds:
                break
        res["cpu_baseline"] = {"value": round(wbytes * reps / el / 1e9, 4), "unit": "GB/s", "cores": n,
                               "kind": "oracle", "sample": f"{reps} full passes over all {rows} rows in {el:.1f} s, "
                                                           f"rows split over {n} threads of the scalar C oracle",
                               "cpu_model": cpu_model()}
    return res


def run_w2_reference(args):
    fmt, rows, K, ncols, seed, desc = W2[args.workload]
    Wh, a16, m, e = _w2_inputs(fmt, rows, K, ncols, seed)
    n = _oracle_threads()
    t0 = time.perf_counter()
    w2_oracle_pass(fmt, rows, K, Wh, a16, m, e, n)
    full = time.perf_counter() - t0
    budget = 100.0 / max(1, args.steps + args.warmup)
    rows_s = int(max(1, min(rows, rows * budget / max(full, 1e-6))))
    for _ in range(args.warmup):
        w2_oracle_pass(fmt, rows, K, Wh, a16, m, e, n, rows_s)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        w2_oracle_pass(fmt, rows, K, Wh, a16, m, e, n, rows_s)
    el = time.perf_counter() - t0
    value = synth.record_bytes(fmt, K) * rows_s * args.steps / el / 1e9
    sample = f"each step: {rows_s} of {rows} rows, split over {n} threads of the scalar C oracle"
    return {
        "impl": "reference", "metric": metric_for(args.workload), "value": round(value, 4), "unit": "GB/s",
        "n_gpus": 0, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el * 1e3 / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "int64/int128 exact, f32 rounding (scalar C)", "data": "synthetic (seeded PCG64)",
        "config": {"workload": desc, "rows": rows, "K": K, "ncols": ncols},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": n, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100000)
    ap.add_argument("--warmup", type=int, default=1000)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="q4k_4096x4096", choices=sorted(WORKLOADS) + sorted(GROUPED) + sorted(FFN) + sorted(KV) + sorted(FP8) +
                    sorted(STACK) + sorted(W2))
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--roof-launches", type=int, default=2000,
                    help="product-kernel launches per graph in the roofline timing (x3)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    if args.impl == "reference":
        if rank == 0:
            if args.workload in GROUPED:
                print(json.dumps(run_grouped_reference(args)), flush=True)
            elif args.workload in FFN:
                print(json.dumps(run_ffn_reference(args)), flush=True)
            elif args.workload in KV:
                print(json.dumps(run_kv_reference(args)), flush=True)
            elif args.workload in FP8:
                print(json.dumps(run_fp8_reference(args)), flush=True)
            elif args.workload in STACK:
                print(json.dumps(run_stack_reference(args)), flush=True)
            elif args.workload in W2:
                print(json.dumps(run_w2_reference(args)), flush=True)
            else:
                print(json.dumps(run_reference(args)), flush=True)
        return
    if world > 1:
        import torch
        import torch.distributed as tdist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        tdist.init_process_group("nccl")
    res = (run_grouped(args, rank, world) if args.workload in GROUPED else
           run_stack(args, rank, world) if args.workload in STACK else
           run_ffn(args, rank, world) if args.workload in FFN else
           run_kv(args, rank, world) if args.workload in KV else
           run_fp8(args, rank, world) if args.workload in FP8 else
           run_w2(args, rank, world) if args.workload in W2 else run_ours(args, rank, world))
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as tdist
        tdist.destroy_process_group()


if __name__ == "__main__":
    main()
