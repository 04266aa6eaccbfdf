#!/usr/bin/env python
"""Benchmark of the fused int4 dequantize-matmul on GB300.

Default workload: group-wise W4A16 GEMV, M = 1, K = N = 2048, G = 32 (bf16 x,
signed int4 W, f16 group scales) -- the decode step the int4 GEMV metric is
quoted on.  A step is one linear over one batch (one activation row) with a
weight matrix that is cold in L2: the timed loop rotates over enough weight
copies to exceed twice the L2 size, so every step streams its weights from
HBM.  Steps are replayed from CUDA graphs and timed with CUDA events.

Metric: weight GB/s = (packed int4 bytes + f16 scale bytes) per step / time.
Also reported: the roofline of the GEMV kernel against the measured HBM copy
bandwidth, the oracle timed on the host cores (cpu_baseline), an end-to-end
figure through the public API with host buffers, and extra lines for the
other workloads (W4A8 GEMV, decode batch, microdecoder, prefill).

--impl reference times the CPU oracle (plain C, row-parallel build) on the
same workload and metric.  Multi-GPU runs (torchrun) are replicas: each rank
runs the whole workload on its own GPU; there is no data-path collective.
"""
from __future__ import annotations

import argparse
import datetime as _dt
import json
import os
import platform
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

L2_FALLBACK = 129 * 1024 * 1024
HBM_FALLBACK_GBS = 6800.0


# ---------------------------------------------------------------- workloads

def _wl(kind, M, N, K, G, layout, desc):
    return dict(kind=kind, M=M, N=N, K=K, G=G, layout=layout, desc=desc, regime="decode" if M <= 16 else "prefill")


# The microdecoder frame: 5 layers x {q,k,v,o 1024x1024; gate,up 3072x1024;
# down 1024x3072} x 15 passes of W4A8 linears with per-row Q8 re-quantisation
# between them (a chain, not one linear: timed by run_microdecoder).
MICRODECODER = "microdecoder_frame"
MICRODECODER_DESC = ("W4A8 microdecoder frame: 5 layers x {q,k,v,o 1024x1024; gate,up 3072x1024; down 1024x3072} "
                     "x 15 passes, per-row Q8 re-quantisation between linears")

WORKLOADS = {
    "w4a16_gemv_m1": _wl("w4a16", 1, 2048, 2048, 32, 0,
                         "group-wise W4A16 GEMV, M=1, K=N=2048, G=32, bf16 x, f16 scales"),
    "w4a16_gemv_m1_k2047": _wl("w4a16", 1, 2048, 2047, 32, 0,
                               "group-wise W4A16 GEMV, M=1, K=2047 (odd, padded), N=2048, G=32"),
    "w4a8_gemv_m1": _wl("w4a8", 1, 2048, 2048, 0, 0,
                        "W4A8 linear_q4 GEMV, M=1, K=N=2048 (per-row Q8 quantize + linear)"),
    "w4a16_decode_m16_n13312": _wl("w4a16", 16, 13312, 2048, 128, 0, "W4A16 decode batch M=16, K=2048, N=13312, G=128"),
    "w4a16_decode_m1_n13312": _wl("w4a16", 1, 13312, 2048, 128, 0, "W4A16 M=1, K=2048, N=13312 (gate_up shape), G=128"),
    "w4a8_decode_m1_n13312": _wl("w4a8", 1, 13312, 2048, 0, 0, "W4A8 M=1, K=2048, N=13312 (gate_up shape)"),
    "w4a16_decode_m1_n13312_il": _wl("w4a16", 1, 13312, 2048, 128, 1,
                                     "W4A16 M=1, K=2048, N=13312, G=128, interleaved [N/64][K][32] layout"),
    "w4a8_decode_m16_n13312": _wl("w4a8", 16, 13312, 2048, 0, 0, "W4A8 decode batch M=16, K=2048, N=13312"),
    "w4a8_prefill_m2048_n2048": _wl("w4a8", 2048, 2048, 2048, 0, 0, "W4A8 prefill M=2048, K=2048, N=2048"),
    "w4a8_prefill_m2048_n3072": _wl("w4a8", 2048, 3072, 2048, 0, 0, "W4A8 prefill M=2048, K=2048, N=3072"),
    "w4a8_prefill_m2048_n13312": _wl("w4a8", 2048, 13312, 2048, 0, 0, "W4A8 prefill M=2048, K=2048, N=13312"),
    "w4a16_prefill_m2048_n2048": _wl("w4a16", 2048, 2048, 2048, 128, 0, "W4A16 prefill M=2048, K=2048, N=2048, G=128"),
    "w4a16_prefill_m2048_n3072": _wl("w4a16", 2048, 3072, 2048, 128, 0, "W4A16 prefill M=2048, K=2048, N=3072, G=128"),
    "w4a16_prefill_m2048_n13312": _wl("w4a16", 2048, 13312, 2048, 128, 0,
                                      "W4A16 prefill M=2048, K=2048, N=13312, G=128"),
    "w4a16_prefill_m2048_n13312_il": _wl("w4a16", 2048, 13312, 2048, 128, 1,
                                         "W4A16 prefill M=2048, K=2048, N=13312, G=128, straight from the "
                                         "interleaved [N/64][K][32] layout"),
    "w4a8_prefill_m2048_n13312_il": _wl("w4a8", 2048, 13312, 2048, 0, 1,
                                        "W4A8 prefill M=2048, K=2048, N=13312, interleaved [N/64][K][32] layout"),
    "w8a16_decode_m1_n13312": _wl("w8a16", 1, 13312, 2048, 0, 0,
                                  "linear_w8a16 (int8 weights, f32 channel scales, f32 activations), M=1, K=2048, "
                                  "N=13312"),
    "w8a16_prefill_m2048_n13312": _wl("w8a16", 2048, 13312, 2048, 0, 0,
                                      "linear_w8a16 prefill M=2048, K=2048, N=13312"),
    "w4a8g_decode_m1_n13312": _wl("w4a8g", 1, 13312, 2048, 128, 0,
                                  "grouped asymmetric W4A8 (f16 scales + zero points per group of 128), M=1, "
                                  "K=2048, N=13312 (per-row Q8 quantize + linear)"),
    "w4a16_b32_decode_m1_n13312": _wl("w4a16", 1, 13312, 2048, 32, 2,
                                      "W4A16 M=1, K=2048, N=13312, inline-scale blocks of 32 (f16 scale beside "
                                      "16 bytes of codes, 18 bytes per block)"),
    "w4a16_b32_decode_m16_n13312": _wl("w4a16", 16, 13312, 2048, 32, 2,
                                       "W4A16 decode batch M=16, K=2048, N=13312, inline-scale blocks of 32"),
    "w4a8g_prefill_m2048_n13312": _wl("w4a8g", 2048, 13312, 2048, 128, 0,
                                      "grouped asymmetric W4A8 prefill M=2048, K=2048, N=13312, G=128"),
}

# The decode-batch configuration: M in {1, 4, 16}, K = 2048, N in {13312 (gate_up), 3072}, W4A16 (G = 128) and
# W4A8, row-major and interleaved [N/64][K][32] weights.
for _kind in ("w4a16", "w4a8"):
    for _M in (1, 4, 16):
        for _N in (13312, 3072):
            for _lay in (0, 1):
                _name = f"{_kind}_decode_m{_M}_n{_N}" + ("_il" if _lay else "")
                if _name not in WORKLOADS:
                    WORKLOADS[_name] = _wl(
                        _kind, _M, _N, 2048, 128 if _kind == "w4a16" else 0, _lay,
                        f"{'W4A16' if _kind == 'w4a16' else 'W4A8'} decode M={_M}, K=2048, N={_N}"
                        + (", G=128" if _kind == "w4a16" else "") + (", interleaved [N/64][K][32] layout" if _lay else ""))

# Extra lines of the default run: every configuration of the benchmark set
# beside the headline (odd K, the decode batch grid, the prefill GEMMs).
EXTRA_DECODE = (["w4a16_gemv_m1_k2047", "w4a8_gemv_m1"]
                + [f"{k}_decode_m{m}_n{n}{l}" for k in ("w4a16", "w4a8") for m in (1, 4, 16) for n in (13312, 3072)
                   for l in ("", "_il")])
EXTRA_PREFILL = ([f"{k}_prefill_m2048_n{n}" for k in ("w4a8", "w4a16") for n in (2048, 3072, 13312)]
                 + ["w4a8_prefill_m2048_n13312_il", "w4a16_prefill_m2048_n13312_il"])


# DRAM bytes (read + write) per launch of the roofline's kernel from one ncu
# capture of that kernel on that workload; None where no capture matches the
# current kernel.
TRAFFIC = {
    "w4a16_gemv_m1": 2391552,                 # all-warp W4A16 GEMV, M=1, N=K=2048, G=32
    "w4a8_gemv_m1": 2137600,                  # all-warp fused quantize + W4A8 dp4a GEMV, M=1, N=K=2048
    "w4a16_decode_m1_n13312": 14088448,       # all-warp W4A16 GEMV, M=1, N=13312, G=128
    "w4a16_decode_m16_n13312": 14181376,      # streaming W4A16 GEMV, two activation tiles
    "w4a16_decode_m1_n13312_il": 14097664,    # staged W4A16 GEMV from the interleaved layout
    "w4a8g_decode_m1_n13312": 14320640,       # staged grouped W4A8 GEMV
    "w8a16_decode_m1_n13312": 27356416,       # staged W8A16 GEMV
    "w4a16_b32_decode_m1_n13312": 15372544,   # staged W4A16 GEMV on inline-scale blocks
}


def weight_bytes(w) -> int:
    N, K, G = w["N"], w["K"], w["G"]
    kp = K + (K & 1)
    packed = N * K if w["kind"] == "w8a16" else N * (kp // 2)
    if w["kind"] == "w4a16":
        scales = N * (kp // G) * 2
    elif w["kind"] == "w4a8g":
        scales = N * (kp // G) * 3  # f16 scale + one-byte zero point per group
    else:
        scales = N * 4
    return packed + scales


def step_bytes(w) -> int:
    """Algorithmic bytes of one linear launch: weights + scales + activations + output."""
    M, N, K = w["M"], w["N"], w["K"]
    # x side: bf16 x (W4A16); f32 x (W8A16); f32 x in, Q8 codes and scales out (W4A8);
    # Q8 codes and scales in (grouped W4A8, quantised by a separate call)
    xb = {"w4a16": M * K * 2, "w8a16": M * K * 4, "w4a8": 5 * M * K + 4 * M}.get(w["kind"], M * K + 4 * M)
    return weight_bytes(w) + xb + M * N * 4


def step_ops(w) -> int:
    return 2 * w["M"] * w["N"] * w["K"]


def metric_of(w, ms_per_step: float, n_gpus: int = 1):
    """(value, unit) of the workload's metric for a step time: weight GB/s for
    decode (M <= 16), tensor ops/s for prefill."""
    if w["regime"] == "decode":
        return n_gpus * weight_bytes(w) / (ms_per_step / 1e3) / 1e9, "GB/s"
    return n_gpus * step_ops(w) / (ms_per_step / 1e3) / 1e12, ("TFLOP/s" if w["kind"] in ("w4a16", "w8a16")
                                                               else "TOPS")


def metric_name(w) -> str:
    if w["regime"] == "decode":
        return f"{'int8' if w['kind'] == 'w8a16' else 'int4'} linear weight GB/s (M={w['M']} decode)"
    label = {"w4a8": "W4A8 TOPS", "w4a8g": "grouped W4A8 TOPS", "w8a16": "W8A16 TFLOP/s"}.get(w["kind"],
                                                                                             "W4A16 TFLOP/s")
    return f"{label} (M={w['M']} prefill)"


# ---------------------------------------------------------------- helpers

def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": HBM_FALLBACK_GBS, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled while the timed region runs."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.lines = []
        self.proc = None
        self.gpu_id = gpu_id

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50"]
        if self.gpu_id:
            cmd += ["-i", self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)

    def summary(self, t0: float, t1: float):
        rows = []
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                ts = _dt.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(parts[1]), float(parts[2]), parts[3], parts[4:9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "nvidia-smi gave no samples"}
        inside = [r for r in rows if t0 <= r[0] <= t1]
        note = None
        if not inside:
            # timed region shorter than the sampling period: nearest samples around it
            inside = sorted(rows, key=lambda r: min(abs(r[0] - t0), abs(r[0] - t1)))[:3]
            note = "timed region shorter than the 50 ms sampling period; nearest samples"
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in inside:
            for nm, v in zip(names[1:], r[4][1:]):
                if v.strip().lower() == "active":
                    reasons.add(nm)
        out = {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": max(r[2] for r in inside),
               "reasons": sorted(reasons), "samples": len(inside)}
        if note:
            out["note"] = note
        return out


def max_over_ranks(ms: float, world: int) -> float:
    """The slowest rank's time (replicas: every rank runs the whole workload;
    the job takes as long as its slowest rank).  Works on either backend: a
    CUDA tensor under NCCL, a CPU tensor under gloo."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([ms], device=dev, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_value(per_rank_units: float, seconds: float, world: int) -> float:
    """Whole-job throughput of `world` replicas, each processing
    `per_rank_units` in the slowest rank's `seconds`."""
    return world * per_rank_units / seconds


def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    return world, rank, local


# ---------------------------------------------------------------- CPU oracle timing

def oracle_inputs(w, seed=1001):
    from w4a16_int4_quantized_gb300 import synth
    if w["kind"] == "w4a16":
        return synth.w4a16_inputs(seed, w["M"], w["N"], w["K"], w["G"])
    x, W = synth.w4a8_inputs(seed, w["M"], w["N"], w["K"])
    return x, W


def oracle_call(w, openmp: bool = True, rows: int | None = None):
    """(call, what, cores, w_sampled): one oracle call of the workload on
    inputs prepared once (prefill: the first 16 activation rows; rows: only
    that many output channels)."""
    import oracle
    o = oracle.get(openmp=openmp)
    cores = os.cpu_count() if openmp else 1
    if w["regime"] == "prefill":
        w = dict(w, M=16, regime="prefill")
    if rows is not None and rows < w["N"]:
        w = dict(w, N=rows, desc=w["desc"] + f" (output channels sampled: {rows} of {w['N']})")
    if w["kind"] == "w4a16" and w["layout"] == 2:
        x, wp, s = oracle_inputs(w)
        blocks = o.blocks_b32(wp, s, w["K"])
        call = lambda: o.linear_w4a16_b32_exact(x, blocks, w["K"])
        what = "ref_linear_w4a16_b32_exact"
    elif w["kind"] == "w4a16":
        x, wp, s = oracle_inputs(w)
        call = lambda: o.linear_w4a16_lanes(x, wp, s, w["K"], w["G"])
        what = "ref_linear_w4a16_lanes"
    elif w["kind"] == "w8a16":
        from w4a16_int4_quantized_gb300 import synth
        x = synth.activations_f32(1001, w["M"], w["K"])
        wq = synth.raw_bytes(1002, w["N"] * w["K"]).view(np.int8).reshape(w["N"], w["K"])
        sw = np.full(w["N"], 1e-3, np.float32)
        call = lambda: o.linear_w8a16_exact(x, wq, sw)
        what = "ref_linear_w8a16_exact"
    elif w["kind"] == "w4a8g":
        from w4a16_int4_quantized_gb300 import synth
        xq, sx, wp, s, z = synth.q4_group_inputs(1001, w["M"], w["N"], w["K"], w["G"])
        call = lambda: o.linear_q4_group(xq, sx, wp, s, z, w["K"], w["G"])
        what = "ref_linear_q4_group"
    else:
        # the step: quantize_row_q8 of the activations, then linear_q4
        x, W = oracle_inputs(w)
        wp, sw = o.quantize_matrix_q4(W)
        call = lambda: o.linear_q4(*o.quantize_row_q8(x)[:2], wp, sw, w["K"])
        what = "ref_quantize_row_q8 + ref_linear_q4"
    return call, what, cores, w


def time_oracle(w, seconds: float, openmp: bool = True):
    """Runs the oracle on a bounded sample: whole calls until `seconds` elapse
    (prefill: calls on the first 16 activation rows, scaled to ops/s)."""
    call, what, cores, w = oracle_call(w, openmp)
    call()
    n, t0 = 0, time.perf_counter()
    while True:
        call()
        n += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    value, unit = metric_of(w, el * 1e3 / n)
    sample = f"{n} full calls of {what} on {w['desc']} ({el:.1f} s)"
    if w.get("layout") == 1:
        sample += "; the oracle reads the row-major form of the same codes"
    if w["regime"] == "prefill":
        sample = f"{n} calls of {what} on 16 of the {w['desc']} activation rows ({el:.1f} s), as ops/s"
    return {"value": value, "unit": unit, "cores": cores, "kind": "oracle", "sample": sample}, n, el


# ---------------------------------------------------------------- GPU measurement

class Workload:
    """Device-resident inputs for `copies` independent steps of one workload.

    step(i): the whole hot path of the workload on copy i -- W4A16: the
    linear; W4A8: the per-row Q8 quantizer on f32 activations, then the
    linear.  kernel(i): the linear alone (the roofline's kernel)."""

    def __init__(self, w, copies: int):
        import torch
        from w4a16_int4_quantized_gb300 import ops, synth
        self.w, self.ops = w, ops
        M, N, K, G = w["M"], w["N"], w["K"], w["G"]
        dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
        self.copies = copies
        if w["kind"] == "w4a16":
            x, wp, s = synth.w4a16_inputs(1001, M, N, K, G)
            x0, w0 = dev(x), dev(wp)
            if w["layout"] == 1:
                w0 = ops.pack_interleaved_n64(w0, K)
            elif w["layout"] == 2:
                w0 = ops.pack_block32(w0, dev(s), K)
            self.x = [x0.clone() for _ in range(copies)]
            self.wt = [w0.clone() for _ in range(copies)]
            self.s = [dev(s) for _ in range(copies)]
            self.ws = None
        elif w["kind"] == "w8a16":
            x0 = dev(synth.activations_f32(1001, M, K))
            w0 = dev(synth.raw_bytes(1002, N * K).view(np.int8).reshape(N, K))
            self.x = [x0.clone() for _ in range(copies)]
            self.wt = [w0.clone() for _ in range(copies)]
            self.s = [torch.full((N,), 1e-3, dtype=torch.float32, device="cuda") for _ in range(copies)]
            need = ops.workspace_bytes(ops.OP_LINEAR_W8A16, M, N, K)
            self.ws = torch.empty(need, dtype=torch.uint8, device="cuda") if need else None
        elif w["kind"] == "w4a8g":
            _, _, wp, s, z = synth.q4_group_inputs(1001, 1, N, K, G)
            xf = dev(synth.activations_f32(1001, M, K))
            xq, sx, _ = ops.quantize_row_q8(xf)
            w0 = dev(wp)
            if w["layout"] == 1:
                w0 = ops.pack_interleaved_n64(w0, K)
            self.xf = [xf.clone() for _ in range(copies)]
            self.x = [xq.clone() for _ in range(copies)]
            self.sx = [sx.clone() for _ in range(copies)]
            self.wt = [w0.clone() for _ in range(copies)]
            self.s = [dev(s) for _ in range(copies)]
            self.z = [dev(z) for _ in range(copies)]
            need = ops.workspace_bytes(ops.OP_LINEAR_Q4_GROUP, M, N, K, G)
            self.ws = torch.empty(need, dtype=torch.uint8, device="cuda") if need else None
        else:
            x, W = synth.w4a8_inputs(1001, M, N, K)
            xf = dev(x)
            xq, sx, _ = ops.quantize_row_q8(xf)
            wq, sw = ops.quantize_matrix_q4(dev(W))
            if w["layout"] == 1:
                wq = ops.pack_interleaved_n64(wq, K)
            self.xf = [xf.clone() for _ in range(copies)]
            self.x = [xq.clone() for _ in range(copies)]
            self.sx = [sx.clone() for _ in range(copies)]
            self.wt = [wq.clone() for _ in range(copies)]
            self.s = [sw.clone() for _ in range(copies)]
            need = ops.workspace_bytes(ops.OP_LINEAR_Q4, M, N, K)
            self.ws = torch.empty(need, dtype=torch.uint8, device="cuda") if need else None
        self.y = [torch.empty((M, N), dtype=torch.float32, device="cuda") for _ in range(copies)]
        torch.cuda.synchronize()

    @property
    def launches_per_step(self) -> int:
        w = self.w
        if w["kind"] == "w4a16":
            return 1
        if w["kind"] == "w8a16":
            return 1 + (1 if self.ws is not None else 0)  # (f32 -> bf16 prepass), linear
        if w["kind"] == "w4a8" and w["M"] == 1 and w["layout"] == 0 and w["N"] >= 1024:
            return 1  # the rows are quantised inside the linear
        if w["kind"] == "w4a8" and w["M"] > 16 and w["K"] % 8 == 0:
            return 2  # quantizer (codes and their f16 image), GEMM
        return 2 + (1 if self.ws is not None else 0)  # quantize, (int8 -> f16 prepass), linear

    def kernel(self, i: int, flags: int = 1):
        w, ops = self.w, self.ops
        c = i % self.copies
        if w["kind"] == "w4a16" and w["layout"] == 2:
            ops.linear_w4a16_b32(self.x[c], self.wt[c], K=w["K"], N=w["N"], flags=flags, out=self.y[c])
        elif w["kind"] == "w4a16":
            ops.linear_w4a16_group(self.x[c], self.wt[c], self.s[c], w["G"], K=w["K"], N=w["N"],
                                   layout=w["layout"], flags=flags, out=self.y[c])
        elif w["kind"] == "w8a16":
            ops.linear_w8a16(self.x[c], self.wt[c], self.s[c], flags=flags, out=self.y[c], workspace=self.ws)
        elif w["kind"] == "w4a8g":
            ops.linear_q4_group(self.x[c], self.sx[c], self.wt[c], self.s[c], self.z[c], w["G"], K=w["K"],
                                N=w["N"], layout=w["layout"], flags=flags, out=self.y[c], workspace=self.ws)
        elif self.launches_per_step == 1:  # W4A8 whose rows are quantised inside the linear: that one kernel
            self.step(i, flags)
        else:
            ops.linear_q4(self.x[c], self.sx[c], self.wt[c], self.s[c], K=w["K"], N=w["N"],
                          layout=w["layout"], flags=flags, out=self.y[c], workspace=self.ws)

    def step(self, i: int, flags: int = 1):
        w = self.w
        if w["kind"] == "w4a8":
            # quantize_row_q8 + linear_q4 as one library call (one kernel at M = 1)
            c = i % self.copies
            self.ops.linear_q4_f32(self.xf[c], self.wt[c], self.s[c], K=w["K"], N=w["N"], layout=w["layout"],
                                   flags=flags, out=self.y[c], xq=self.x[c], sx=self.sx[c], workspace=self.ws)
        elif w["kind"] not in ("w4a16", "w8a16"):
            c = i % self.copies
            M, K = self.xf[c].shape
            st = self.ops.raw.w4_quantize_row_q8(self.xf[c].data_ptr(), M, K, self.x[c].data_ptr(),
                                                  self.sx[c].data_ptr(), None, self.ops._stream())
            assert st == 0
            # the linear reads x only after griddepcontrol.wait (the quantizer
            # has finished); before it, only its weight fetch overlaps
            self.kernel(i, flags)
        else:
            self.kernel(i, flags)


def copies_for(w, l2_bytes: int) -> int:
    per = weight_bytes(w) + w["M"] * w["K"] * (2 if w["kind"] == "w4a16" else 5)
    return max(2, min(256, int(np.ceil(2.2 * l2_bytes / per))))


def time_steps(wl: Workload, steps: int, warmup: int, chunk: int = 256, kernel_only: bool = False):
    """Exactly `steps` steps replayed from CUDA graphs; returns (ms, t0, t1)."""
    import torch
    chunk = max(1, min(chunk if wl.w["regime"] == "decode" else 8, steps))
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()

    run = wl.kernel if kernel_only else wl.step

    def capture(n, base):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(n):
                run(base + i)
        return g

    with torch.cuda.stream(stream):
        for i in range(min(warmup, 8)):
            run(i)
    torch.cuda.synchronize()
    full = capture(chunk, 0)
    rem = steps % chunk
    tail = capture(rem, chunk) if rem else None
    with torch.cuda.stream(stream):
        for _ in range(max(warmup, 3)):
            full.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.time()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(steps // chunk):
            full.replay()
        if tail is not None:
            tail.replay()
        e1.record(stream)
    e1.synchronize()
    t1 = time.time()
    return e0.elapsed_time(e1), t0, t1


def time_e2e(w, steps: int, chunk: int = 64):
    """Public API with host buffers, every step: pinned x -> device, the
    step's library calls, y -> pinned host.  The per-step sequence (copies
    included) is captured once into a CUDA graph of `chunk` steps and
    replayed, as a serving loop would run it."""
    import torch
    from w4a16_int4_quantized_gb300 import ops, synth
    M, N, K, G = w["M"], w["N"], w["K"], w["G"]
    if w["kind"] == "w4a16":
        x, wp, s = synth.w4a16_inputs(1001, M, N, K, G)
        xh = torch.from_numpy(x.view(np.int16)).pin_memory()
        wd = torch.from_numpy(wp).cuda()
        sd = torch.from_numpy(s.view(np.int16)).cuda()
        xd = torch.empty_like(xh, device="cuda")
        yd = torch.empty((M, N), dtype=torch.float32, device="cuda")
        yh = torch.empty((M, N), dtype=torch.float32).pin_memory()

        if w["layout"] == 1:
            wd = ops.pack_interleaved_n64(wd, K)
        elif w["layout"] == 2:
            wd = ops.pack_block32(wd, sd, K)

        def step():
            xd.copy_(xh, non_blocking=True)
            if w["layout"] == 2:
                ops.linear_w4a16_b32(xd, wd, K=K, N=N, flags=ops.FLAG_PDL, out=yd)
            else:
                ops.linear_w4a16_group(xd, wd, sd, G, K=K, N=N, layout=w["layout"], flags=ops.FLAG_PDL, out=yd)
            yh.copy_(yd, non_blocking=True)
        h2d = xh.numel() * 2
    elif w["kind"] == "w8a16":
        xh = torch.from_numpy(synth.activations_f32(1001, M, K)).pin_memory()
        wd = torch.from_numpy(synth.raw_bytes(1002, N * K).view(np.int8).reshape(N, K).copy()).cuda()
        sd = torch.full((N,), 1e-3, dtype=torch.float32, device="cuda")
        xd = torch.empty_like(xh, device="cuda")
        yd = torch.empty((M, N), dtype=torch.float32, device="cuda")
        yh = torch.empty((M, N), dtype=torch.float32).pin_memory()
        need = ops.workspace_bytes(ops.OP_LINEAR_W8A16, M, N, K)
        ws = torch.empty(need, dtype=torch.uint8, device="cuda") if need else None

        def step():
            xd.copy_(xh, non_blocking=True)
            ops.linear_w8a16(xd, wd, sd, flags=ops.FLAG_PDL, out=yd, workspace=ws)
            yh.copy_(yd, non_blocking=True)
        h2d = xh.numel() * 4
    elif w["kind"] == "w4a8g":
        _, _, wp, s, z = synth.q4_group_inputs(1001, 1, N, K, G)
        xh = torch.from_numpy(synth.activations_f32(1001, M, K)).pin_memory()
        wd, sd, zd = torch.from_numpy(wp).cuda(), torch.from_numpy(s.view(np.int16)).cuda(), torch.from_numpy(z).cuda()
        if w["layout"] == 1:
            wd = ops.pack_interleaved_n64(wd, K)
        xd = torch.empty_like(xh, device="cuda")
        xq = torch.empty((M, K), dtype=torch.int8, device="cuda")
        sx = torch.empty(M, dtype=torch.float32, device="cuda")
        yd = torch.empty((M, N), dtype=torch.float32, device="cuda")
        yh = torch.empty((M, N), dtype=torch.float32).pin_memory()
        need = ops.workspace_bytes(ops.OP_LINEAR_Q4_GROUP, M, N, K, G)
        ws = torch.empty(need, dtype=torch.uint8, device="cuda") if need else None

        def step():
            xd.copy_(xh, non_blocking=True)
            st = ops.raw.w4_quantize_row_q8(xd.data_ptr(), M, K, xq.data_ptr(), sx.data_ptr(), None, ops._stream())
            assert st == 0
            ops.linear_q4_group(xq, sx, wd, sd, zd, G, K=K, N=N, layout=w["layout"], flags=ops.FLAG_PDL, out=yd, workspace=ws)
            yh.copy_(yd, non_blocking=True)
        h2d = xh.numel() * 4
    else:
        x, W = synth.w4a8_inputs(1001, M, N, K)
        xh = torch.from_numpy(x).pin_memory()
        wq, sw = ops.quantize_matrix_q4(torch.from_numpy(W).cuda())
        if w["layout"] == 1:
            wq = ops.pack_interleaved_n64(wq, K)
        xd = torch.empty_like(xh, device="cuda")
        xq = torch.empty((M, K), dtype=torch.int8, device="cuda")
        sx = torch.empty(M, dtype=torch.float32, device="cuda")
        yd = torch.empty((M, N), dtype=torch.float32, device="cuda")
        yh = torch.empty((M, N), dtype=torch.float32).pin_memory()
        need = ops.workspace_bytes(ops.OP_LINEAR_Q4, M, N, K)
        ws = torch.empty(need, dtype=torch.uint8, device="cuda") if need else None

        def step():
            xd.copy_(xh, non_blocking=True)
            ops.linear_q4_f32(xd, wq, sw, K=K, N=N, layout=w["layout"], flags=ops.FLAG_PDL, out=yd, xq=xq, sx=sx,
                              workspace=ws)
            yh.copy_(yd, non_blocking=True)
        h2d = xh.numel() * 4
    stream = torch.cuda.Stream()
    chunk = max(1, min(chunk, steps))
    with torch.cuda.stream(stream):
        for _ in range(5):
            step()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for _ in range(chunk):
            step()
    tail = None
    if steps % chunk:
        tail = torch.cuda.CUDAGraph()
        with torch.cuda.graph(tail, stream=stream):
            for _ in range(steps % chunk):
                step()
    with torch.cuda.stream(stream):
        graph.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(steps // chunk):
            graph.replay()
        if tail is not None:
            tail.replay()
        e1.record(stream)
    e1.synchronize()
    ms = e0.elapsed_time(e1)
    value, unit = metric_of(w, ms / steps)
    return {"value": value, "unit": unit, "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(M * N * 4),
            "ms_per_step": ms / steps,
            "how": "per step: pinned host x -> device, the library calls, y -> pinned host; CUDA graph of "
                   f"{chunk} steps replayed"}


def cpu_model() -> str:
    """The host CPU's model name (lscpu), for the CPU baseline's record."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.strip().lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return platform.processor() or platform.machine()


def measure_line(name: str, l2: int, peaks, sampler, cpu_seconds: float | None):
    """One workload of the benchmark set: the step (the whole hot path) and the
    roofline's kernel alone, both from CUDA-graph replays over rotating inputs
    larger than L2, with the clocks seen and the oracle timed on a bounded sample."""
    import torch
    from w4a16_int4_quantized_gb300 import ops
    w = WORKLOADS[name]
    wl = Workload(w, copies_for(w, l2))
    steps = 2048 if w["regime"] == "decode" else 32
    ms, t0, t1 = time_steps(wl, steps, 3)
    kms, _, _ = time_steps(wl, steps, 3, kernel_only=True)
    value, unit = metric_of(w, ms / steps)
    wl.copies = 1  # warm: every step on input copy 0, whose weights then stay in L2
    wms, _, _ = time_steps(wl, steps, 3)
    warm_value, _ = metric_of(w, wms / steps)
    per_launch = kms / 1e3 / steps
    if w["regime"] == "decode":
        peak = float(peaks.get("hbm_gbs", HBM_FALLBACK_GBS))
        ach = step_bytes(w) / per_launch / 1e9
        roof = {"bound": "hbm", "achieved": round(ach, 1), "peak": peak, "unit": "GB/s", "frac": round(ach / peak, 4),
                "traffic": TRAFFIC.get(name), "bytes_per_launch": step_bytes(w),
                "us_per_launch": round(per_launch * 1e6, 3), "peak_source": "measured hbm_gbs (copy)"}
    else:
        peak = float(peaks.get("bf16_tflops", 1900.0))
        ach = step_ops(w) / per_launch / 1e12
        roof = {"bound": "tensor", "achieved": round(ach, 1), "peak": peak, "unit": "TFLOP/s",
                "frac": round(ach / peak, 4), "traffic": TRAFFIC.get(name), "flops_per_launch": step_ops(w),
                "us_per_launch": round(per_launch * 1e6, 3),
                "peak_source": "measured bf16_tflops (burst: the call is timed on its own; kind::f16 runs at the "
                               "bf16 rate)"}
    line = {"workload": name, "desc": w["desc"], "metric": metric_name(w), "value": round(value, 2), "unit": unit,
            "us_per_step": round(ms * 1e3 / steps, 3), "steps": steps, "launches_per_step": wl.launches_per_step,
            "roofline": roof, "clocks": sampler.summary(t0, t1),
            "warm_l2_resident": {"value": round(warm_value, 2), "unit": unit,
                                 "us_per_step": round(wms * 1e3 / steps, 3)}}
    if w["kind"] == "w4a8" and w["regime"] == "prefill":
        line["step"] = "quantize_row_q8 + linear_q4 (linear_q4_f32); roofline: linear_q4 alone (int8 -> f16 prepass + GEMM)"
        kv, _ = metric_of(w, kms / steps)
        line["linear_only"] = {"value": round(kv, 2), "unit": unit, "us_per_call": round(per_launch * 1e6, 3)}
    del wl
    torch.cuda.empty_cache()
    if cpu_seconds:
        cb, _, _ = time_oracle(w, cpu_seconds)
        cb["cpu_model"] = cpu_model()
        line["cpu_baseline"] = cb
    return line


def extra_lines(l2: int, peaks, sampler, cpu_seconds: float | None):
    out = [measure_line(n, l2, peaks, sampler, cpu_seconds) for n in EXTRA_DECODE + EXTRA_PREFILL]
    from w4a16_int4_quantized_gb300 import ops
    int8 = ops.probe_mma_peak(0)
    for ln in out:
        if ln["workload"].startswith("w4a8_prefill"):
            ln["roofline"]["int8_mma_sync_peak_tops"] = round(int8, 1)
            ln["roofline"]["frac_of_int8_peak"] = round(ln["roofline"]["achieved"] / int8, 3)
    return out


# ---------------------------------------------------------------- arms

def run_reference_microdecoder(args):
    per_step = min(20.0, args.cpu_seconds / max(1, args.steps))
    if args.warmup:
        time_oracle_microdecoder(0.2)
    total_n, total_s, cb = 0, 0.0, None
    for _ in range(args.steps):
        cb, n, el = time_oracle_microdecoder(per_step)
        total_n += n
        total_s += el
    from w4a16_int4_quantized_gb300 import synth
    ms_frame = total_s * 1e3 / total_n * synth.MICRODECODER_PASSES
    value = microdecoder_weight_bytes() * synth.MICRODECODER_PASSES / (ms_frame / 1e3) / 1e9
    cb = dict(cb, value=value, ms_per_frame=ms_frame,
              sample=f"{total_n} oracle passes over {args.steps} steps ({total_s:.1f} s); " + cb["sample"])
    line = {"impl": "reference", "metric": "microdecoder effective int4 weight GB/s (frame)", "value": value,
            "unit": "GB/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms_frame, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "s8", "data": "synthetic", "config": {"workload": MICRODECODER, "desc": MICRODECODER_DESC},
            "cpu_baseline": cb,
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_reference(args, world, rank):
    if rank != 0:
        return
    if args.workload == MICRODECODER:
        run_reference_microdecoder(args)
        return
    w = WORKLOADS[args.workload]
    # inputs prepared once; each step is at least one whole oracle call, and
    # the steps share about --cpu-seconds, so any --steps ends in bounded time
    call, what, cores, ws = oracle_call(w)
    call()
    t = time.perf_counter()
    call()
    t = time.perf_counter() - t
    if args.steps * t > 3 * args.cpu_seconds and w["N"] > 64:
        # too many steps for whole calls in the budget: each step computes a
        # sample of the output channels, scaled to the metric by its bytes
        rows = max(64, int(w["N"] * 3 * args.cpu_seconds / (args.steps * t)) // 64 * 64)
        call, what, cores, ws = oracle_call(w, rows=rows)
    for _ in range(max(0, args.warmup)):
        call()
    per_step = min(20.0, args.cpu_seconds / max(1, args.steps))
    total_n, total_s = 0, 0.0
    for _ in range(args.steps):
        t0 = time.perf_counter()
        while True:
            call()
            total_n += 1
            el = time.perf_counter() - t0
            if el >= per_step:
                break
        total_s += el
    value, unit = metric_of(ws, total_s * 1e3 / total_n)
    sample = f"{total_n} calls of {what} on {ws['desc']} over {args.steps} steps ({total_s:.1f} s)"
    if w["regime"] == "prefill":
        sample += "; 16 of the activation rows per call, as ops/s"
    cb = {"value": value, "unit": unit, "cores": cores, "kind": "oracle", "sample": sample, "cpu_model": cpu_model()}
    line = {"impl": "reference", "metric": metric_name(w), "value": value, "unit": unit,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": total_s * 1e3 / max(1, total_n), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": args.workload, "desc": w["desc"]},
            "cpu_baseline": cb,
            "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def microdecoder_weight_bytes() -> int:
    """Packed codes + f32 channel scales of one pass (all 35 linears)."""
    from w4a16_int4_quantized_gb300 import synth
    return sum(n * (k // 2) + 4 * n for _, n, k in synth.MICRODECODER_LINEARS) * synth.MICRODECODER_LAYERS


def microdecoder_frame_ops(run_linear, run_quant, layers, passes, x0):
    """The frame's dataflow, shared by the GPU and the oracle legs: per layer
    q, k, v read h; o reads Q8(v); gate and up read Q8(o); down reads Q8(up);
    the next h is Q8(down).  run_linear(layer, name, (q, s)) -> y and
    run_quant(y) -> (q, s) are supplied by the leg."""
    h = run_quant(x0)
    y = None
    for _ in range(passes):
        for li in range(len(layers)):
            run_linear(li, "q", h)
            run_linear(li, "k", h)
            v = run_quant(run_linear(li, "v", h))
            o = run_quant(run_linear(li, "o", v))
            run_linear(li, "gate", o)
            u = run_quant(run_linear(li, "up", o))
            y = run_linear(li, "down", u)
            h = run_quant(y)
    return h, y


class Microdecoder:
    """Frames of the weight-resident microdecoder through the public API: 35
    W4A8 linears + 20 per-row re-quantisations per pass, 15 passes, plus the
    input quantisation; all buffers preallocated so a frame can be captured
    in a CUDA graph.  `copies` independent weight sets (frame i uses set
    i % copies) make the working set larger than L2 when asked."""

    def __init__(self, copies: int = 1):
        import torch
        from w4a16_int4_quantized_gb300 import ops, synth
        self.ops, self.synth = ops, synth
        dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
        self.sets = []
        for c in range(copies):
            layers = []
            for L in synth.microdecoder_weights(3003 + 100 * c):
                layers.append({name: (*ops.quantize_matrix_q4(dev(W)), W.shape[1]) for name, W in L.items()})
            self.sets.append(layers)
        self.x0 = dev(synth.activations_f32(3004, 1, 1024))
        f = lambda n: torch.empty((1, n), dtype=torch.float32, device="cuda")
        self.y = {name: f(n) for name, n, _ in synth.MICRODECODER_LINEARS}
        # the four re-quantisation sites of a layer, in call order: h (x0, then
        # each down output), v, o, up
        self.sites = [(torch.empty((1, n), dtype=torch.int8, device="cuda"),
                       torch.empty(1, dtype=torch.float32, device="cuda")) for n in (1024, 1024, 1024, 3072)]
        # the chain path writes every linear's own output buffer
        self.y_chain = [[{name: f(n) for name, n, _ in synth.MICRODECODER_LINEARS}
                         for _ in range(synth.MICRODECODER_LAYERS)] for _ in range(copies)]
        self.desc = [self.descriptors(c) for c in range(copies)]
        self.chain_ws = torch.zeros(ops.chain_workspace_bytes(self.desc[0], 1024), dtype=torch.uint8, device="cuda")
        torch.cuda.synchronize()

    launches_per_frame = {"per_call": 1 + 15 * 5 * 11, "per_call_fused": 15 * 5 * 7, "chain": 1}

    def descriptors(self, c: int):
        """(w, sw, y, input) per linear of weight set c, in the frame's dataflow order."""
        out = []
        names = [n for n, _, _ in self.synth.MICRODECODER_LINEARS]
        for li, L in enumerate(self.sets[c]):
            base = 7 * li
            h_in = -1 if li == 0 else base - 1
            ins = {"q": h_in, "k": h_in, "v": h_in, "o": base + 2, "gate": base + 3, "up": base + 3,
                   "down": base + 5}
            out += [(L[n][0], L[n][1], self.y_chain[c][li][n], ins[n]) for n in names]
        return out

    def frame_chain(self, i: int = 0):
        """The frame as one w4_chain_q4 call (one persistent kernel)."""
        c = i % len(self.sets)
        d = self.desc[c]
        self.ops.chain_q4(self.x0, d, self.synth.MICRODECODER_PASSES, len(d) - 1, workspace=self.chain_ws)
        return d[-1][2]

    def frame(self, i: int = 0):
        ops = self.ops
        layers = self.sets[i % len(self.sets)]
        calls = [0]

        def quant(x):
            q, s = self.sites[calls[0] % 4]
            calls[0] += 1
            n = x.shape[1]
            assert q.shape[1] == n
            st = ops.raw.w4_quantize_row_q8(x.data_ptr(), 1, n, q.data_ptr(), s.data_ptr(), None, ops._stream())
            if st != 0:
                raise RuntimeError(f"w4_quantize_row_q8: status {st}")
            return q, s

        def linear(li, name, h):
            pk, sw, K = layers[li][name]
            return ops.linear_q4(h[0], h[1], pk, sw, K=K, flags=ops.FLAG_PDL, out=self.y[name])

        return microdecoder_frame_ops(linear, quant, layers, self.synth.MICRODECODER_PASSES, self.x0)

    def frame_fused(self, i: int = 0):
        """The frame call by call with w4_linear_q4_f32: every linear takes the
        f32 output before it and quantises it itself (one launch per linear)."""
        ops = self.ops
        layers = self.sets[i % len(self.sets)]
        scratch = {1024: self.sites[0], 3072: self.sites[3]}

        def linear(li, name, x):
            pk, sw, K = layers[li][name]
            q, s = scratch[K]
            return ops.linear_q4_f32(x, pk, sw, K=K, flags=ops.FLAG_PDL, out=self.y[name], xq=q, sx=s)[0]

        h = self.x0
        y = None
        for _ in range(self.synth.MICRODECODER_PASSES):
            for li in range(len(layers)):
                linear(li, "q", h)
                linear(li, "k", h)
                v = linear(li, "v", h)
                o = linear(li, "o", v)
                linear(li, "gate", o)
                u = linear(li, "up", o)
                y = linear(li, "down", u)
                h = y
        return y


def time_microdecoder(copies: int, frames: int, warmup: int, mode: str = "chain"):
    """Exactly `frames` frames replayed from one CUDA graph per weight set;
    returns (ms_per_frame, t0, t1)."""
    import torch
    md = Microdecoder(copies)
    run = {"chain": md.frame_chain, "per_call_fused": md.frame_fused}.get(mode, md.frame)
    st = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(st):
        for i in range(min(max(warmup, 1), copies * 2)):
            run(i)
    torch.cuda.synchronize()
    graphs = []
    for c in range(copies):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=st):
            run(c)
        graphs.append(g)
    with torch.cuda.stream(st):
        for i in range(max(warmup, 3)):
            graphs[i % copies].replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.time()
    with torch.cuda.stream(st):
        e0.record(st)
        for i in range(frames):
            graphs[i % copies].replay()
        e1.record(st)
    e1.synchronize()
    t1 = time.time()
    ms = e0.elapsed_time(e1) / frames
    del graphs, md
    torch.cuda.empty_cache()
    return ms, t0, t1


def time_microdecoder_e2e(frames: int):
    """Public API with host buffers: pinned x0 -> device, one frame (one
    w4_chain_q4 call, replayed from a CUDA graph), the final down output ->
    pinned host."""
    import torch
    md = Microdecoder(1)
    xh = md.x0.cpu().pin_memory()
    yh = torch.empty((1, 1024), dtype=torch.float32).pin_memory()
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        md.frame_chain(0)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        y = md.frame_chain(0)
    torch.cuda.synchronize()

    def step():
        md.x0.copy_(xh, non_blocking=True)
        g.replay()
        yh.copy_(y, non_blocking=True)
    with torch.cuda.stream(st):
        for _ in range(3):
            step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(st):
        e0.record(st)
        for _ in range(frames):
            step()
        e1.record(st)
    e1.synchronize()
    ms = e0.elapsed_time(e1) / frames
    del g, md
    torch.cuda.empty_cache()
    return ms, xh.numel() * 4, yh.numel() * 4


def time_oracle_microdecoder(seconds: float, openmp: bool = True):
    """The oracle on a bounded sample of the frame: whole passes (35 linears +
    20 re-quantisations) until `seconds` elapse, scaled to frames."""
    import oracle
    from w4a16_int4_quantized_gb300 import synth
    o = oracle.get(openmp=openmp)
    layers = [{name: (*o.quantize_matrix_q4(W), W.shape[1]) for name, W in L.items()}
              for L in synth.microdecoder_weights(3003)]
    x0 = synth.activations_f32(3004, 1, 1024)
    linear = lambda li, name, h: o.linear_q4(h[0], h[1], layers[li][name][0], layers[li][name][1], layers[li][name][2])
    quant = lambda y: o.quantize_row_q8(y)[:2]
    microdecoder_frame_ops(linear, quant, layers, 1, x0)
    n, t0 = 0, time.perf_counter()
    while True:
        microdecoder_frame_ops(linear, quant, layers, 1, x0)
        n += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    ms_frame = el * 1e3 / n * synth.MICRODECODER_PASSES
    gbs = microdecoder_weight_bytes() * synth.MICRODECODER_PASSES / (ms_frame / 1e3) / 1e9
    return {"value": gbs, "unit": "GB/s", "cores": os.cpu_count() if openmp else 1, "kind": "oracle",
            "sample": f"{n} whole passes (35 ref_linear_q4 + 20 ref_quantize_row_q8 each) of the frame "
                      f"({el:.1f} s), scaled x{synth.MICRODECODER_PASSES} to frames",
            "ms_per_frame": ms_frame}, n, el


def microdecoder_line(l2: int, peak_gbs: float, frames: int, warmup: int):
    """Frame time and effective weight GB/s of the one-kernel chain path, of
    the per-call path (quantize_row_q8 + linear_q4: 826 launches) and of the
    per-call path through w4_linear_q4_f32 (525 launches), each L2-resident
    (one weight set, the cache residency that motivates int4 here) and with
    rotating weight sets larger than L2."""
    from w4a16_int4_quantized_gb300 import synth
    wbytes = microdecoder_weight_bytes()
    per_frame = wbytes * synth.MICRODECODER_PASSES
    rot = max(2, int(np.ceil(2.2 * l2 / wbytes)))
    out = {}
    for mode in ("chain", "per_call", "per_call_fused"):
        for label, copies in (("rotating", rot), ("l2_resident", 1)):
            ms, t0, t1 = time_microdecoder(copies, frames, warmup, mode)
            out[f"{mode}_{label}"] = {"ms_per_frame": round(ms, 4), "frames_per_s": round(1e3 / ms, 1),
                                      "weight_gbs": round(per_frame / (ms / 1e3) / 1e9, 1), "weight_sets": copies,
                                      "frac_of_hbm": round(per_frame / (ms / 1e3) / 1e9 / peak_gbs, 4),
                                      "launches_per_frame": Microdecoder.launches_per_frame[mode],
                                      "t0": t0, "t1": t1}
    return out, wbytes, rot


def microdecoder_extra(md: dict, sampler, cpu_seconds):
    """The default run's microdecoder line: each mode's figures (from
    microdecoder_line) with the clocks sampled while it ran, and the oracle's
    frame on the host cores beside them (cpu_seconds None: no oracle)."""
    line = {"workload": MICRODECODER, "desc": MICRODECODER_DESC, "metric": "effective int4 weight GB/s"}
    for k, v in md.items():
        line[k] = {kk: vv for kk, vv in v.items() if kk not in ("t0", "t1")}
        line[k]["clocks"] = sampler.summary(v["t0"], v["t1"])
    if cpu_seconds is not None:
        cb, _, _ = time_oracle_microdecoder(cpu_seconds)
        cb["cpu_model"] = cpu_model()
        line["cpu_baseline"] = cb
    return line


def run_microdecoder(args, world, rank, local):
    import torch
    from w4a16_int4_quantized_gb300 import build, synth
    if local == 0:
        build.build()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    from w4a16_int4_quantized_gb300 import ops
    torch.cuda.set_device(local)
    props = torch.cuda.get_device_properties(local)
    l2 = int(getattr(props, "L2_cache_size", 0) or L2_FALLBACK)
    peaks, peak_src = measured_peaks()
    peak = float(peaks.get("hbm_gbs", HBM_FALLBACK_GBS))
    ops.device_status(clear=True)
    gpu_id = None
    try:
        gpu_id = "GPU-" + str(props.uuid)
    except Exception:
        pass
    frames = args.steps
    sampler = ClockSampler(gpu_id)
    sampler.start()
    time.sleep(0.3)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    res, wbytes, rot = microdecoder_line(l2, peak, frames, args.warmup)
    time.sleep(0.2)
    sampler.stop()
    r = res["chain_rotating"]
    ms = max_over_ranks(r["ms_per_frame"], world)
    status = ops.device_status()
    if rank != 0:
        return
    per_frame = wbytes * synth.MICRODECODER_PASSES
    value = replica_value(per_frame, ms / 1e3, world) / 1e9
    e_ms, h2d, d2h = time_microdecoder_e2e(min(frames, 200))
    cpu = None
    if not args.no_cpu:
        cpu, _, _ = time_oracle_microdecoder(args.cpu_seconds)
        cpu["cpu_model"] = cpu_model()
    line = {"metric": "microdecoder effective int4 weight GB/s (frame)", "value": round(value, 1), "unit": "GB/s",
            "n_gpus": world, "steps": frames, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "s8", "data": "synthetic",
            "config": {"workload": MICRODECODER, "desc": MICRODECODER_DESC,
                       "step": "one frame = one w4_chain_q4 call (one persistent kernel)",
                       "weight_bytes_per_pass": wbytes, "passes_per_frame": synth.MICRODECODER_PASSES,
                       "parallelism": "replicas" if world > 1 else "single",
                       "l2": f"inputs larger than L2: {rot} rotating weight sets ({rot * wbytes / 2**20:.0f} MiB) "
                             f"vs L2 {l2 / 2**20:.0f} MiB",
                       "timing": "CUDA events around CUDA-graph replays of exactly `steps` frames"},
            "paths": {k: {kk: vv for kk, vv in v.items() if kk not in ("t0", "t1")} for k, v in res.items()},
            "roofline": {"bound": "hbm", "achieved": round(per_frame / (ms / 1e3) / 1e9, 1), "peak": peak,
                         "unit": "GB/s", "frac": round(per_frame / (ms / 1e3) / 1e9 / peak, 4), "traffic": None,
                         "peak_source": f"{peak_src} hbm_gbs (copy)",
                         "note": "weight bytes of the whole frame / frame time of the one-kernel chain; "
                                 "bound by the 299 grid barriers between dependent stages, not by bytes"},
            "cpu_baseline": cpu,
            "e2e": {"value": round(per_frame / (e_ms / 1e3) / 1e9, 1), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e_ms},
            "gpu_launches": frames * Microdecoder.launches_per_frame["chain"],
            "clocks": sampler.summary(r["t0"], r["t1"]),
            "device_status": status}
    print(json.dumps(line), flush=True)


def run_ours(args, world, rank, local):
    import torch
    from w4a16_int4_quantized_gb300 import build
    if rank == 0:
        build.build()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    from w4a16_int4_quantized_gb300 import ops
    torch.cuda.set_device(local)
    props = torch.cuda.get_device_properties(local)
    l2 = int(getattr(props, "L2_cache_size", 0) or L2_FALLBACK)
    peaks, peak_src = measured_peaks()
    w = WORKLOADS[args.workload]
    copies = copies_for(w, l2)
    wl = Workload(w, copies)
    ops.device_status(clear=True)

    gpu_id = None
    try:
        gpu_id = "GPU-" + str(props.uuid)
    except Exception:
        pass
    sampler = ClockSampler(gpu_id)
    sampler.start()
    time.sleep(0.3)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    # the timed region (exactly `steps` steps) is run `repeats` times; the
    # median is reported, the individual times beside it
    runs = []
    for r in range(max(1, args.repeats)):
        ms_r, t0_r, t1_r = time_steps(wl, args.steps, args.warmup)
        runs.append(ms_r)
        if r == 0:
            t0 = t0_r
        t1 = t1_r
    ms = statistics.median(runs)
    torch.cuda.synchronize()
    time.sleep(0.2)
    sampler.stop()
    ms_max = max_over_ranks(ms, world)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    status = ops.device_status()
    value, unit = metric_of(w, ms_max / args.steps, world)
    # the roofline's kernel (the linear) timed alone, same graphs and copies
    kms, _, _ = time_steps(wl, min(args.steps, 4096 if w["regime"] == "decode" else 64), args.warmup,
                           kernel_only=True)
    kn = min(args.steps, 4096 if w["regime"] == "decode" else 64)
    per_launch_s = kms / 1e3 / kn
    if w["regime"] == "decode":
        peak = float(peaks.get("hbm_gbs", HBM_FALLBACK_GBS))
        achieved = step_bytes(w) / per_launch_s / 1e9
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": TRAFFIC.get(args.workload), "peak_source": f"{peak_src} hbm_gbs (copy)",
                "bytes_per_launch": step_bytes(w), "us_per_launch": round(per_launch_s * 1e6, 3)}
    else:
        peak = float(peaks.get("bf16_tflops_sustained", peaks.get("bf16_tflops", 1700.0)))
        achieved = step_ops(w) / per_launch_s / 1e12
        roof = {"bound": "tensor", "achieved": round(achieved, 1), "peak": peak, "unit": "TFLOP/s",
                "frac": round(achieved / peak, 4), "traffic": TRAFFIC.get(args.workload),
                "peak_source": f"{peak_src} bf16_tflops_sustained (kind::f16 runs at the bf16 rate)",
                "flops_per_launch": step_ops(w), "us_per_launch": round(per_launch_s * 1e6, 3)}
        if w["kind"] == "w4a8":
            # the metric's "% int8 peak": the int8 tensor rate of this part (legacy mma.sync s8), measured now
            int8 = ops.probe_mma_peak(0)
            roof["int8_mma_sync_peak_tops"] = round(int8, 1)
            roof["frac_of_int8_peak"] = round(achieved / int8, 3)
    launches = args.steps * wl.launches_per_step
    if rank != 0:
        return
    # warm, beside the cold headline: every step on input copy 0, whose
    # weights then stay in L2 between steps
    wl.copies = 1
    wn = min(args.steps, 4096 if w["regime"] == "decode" else 64)
    wms, _, _ = time_steps(wl, wn, args.warmup)
    warm_value, _ = metric_of(w, wms / wn)
    warm = {"value": round(warm_value, 2), "unit": unit, "ms_per_step": wms / wn, "steps": wn,
            "note": "one input copy, L2-resident between steps; the headline rotates copies beyond L2"}
    del wl
    torch.cuda.empty_cache()
    e2e = time_e2e(w, min(args.steps, 2000 if w["regime"] == "decode" else 20))
    cpu = None
    if not args.no_cpu:
        cpu, _, _ = time_oracle(w, args.cpu_seconds)
        cpu["cpu_model"] = cpu_model()
    extra = []
    if not args.no_extra and args.workload == "w4a16_gemv_m1":
        sampler = ClockSampler(gpu_id)
        sampler.start()
        time.sleep(0.3)
        extra = extra_lines(l2, peaks, sampler, None if args.no_cpu else min(args.cpu_seconds, 1.0))
        md, _, _ = microdecoder_line(l2, float(peaks.get("hbm_gbs", HBM_FALLBACK_GBS)), 200, 3)
        sampler.stop()
        extra.append(microdecoder_extra(md, sampler, None if args.no_cpu else min(args.cpu_seconds, 1.0)))
    line = {
        "metric": metric_name(w),
        "value": round(value, 2), "unit": unit, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_max / args.steps, "repeats": len(runs),
        "ms_per_step_each": [round(r / args.steps, 7) for r in runs], "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": {"w4a16": "bf16", "w8a16": "f32"}.get(w["kind"], "s8"), "data": "synthetic",
        "config": {"workload": args.workload, "desc": w["desc"], "M": w["M"], "N": w["N"], "K": w["K"],
                   "G": w["G"], "parallelism": "replicas" if world > 1 else "single",
                   "l2": f"inputs larger than L2: {copies} rotating input copies "
                         f"({copies * weight_bytes(w) / 2**20:.0f} MiB of weights) vs L2 {l2 / 2**20:.0f} MiB",
                   "step": {"w4a8": "linear_q4_f32 (quantize_row_q8 + linear_q4 in one call)",
                            "w4a8g": "quantize_row_q8 + linear_q4_group",
                            "w8a16": "linear_w8a16"}.get(
                       w["kind"], "linear_w4a16_group"),
                   "timing": "CUDA events around CUDA-graph replays of exactly `steps` steps; the timed region "
                             "is repeated `repeats` times and the median reported"},
        "roofline": roof,
        "warm_l2_resident": warm,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": sampler.summary(t0, t1),
        "device_status": status,
        "extra": extra,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=65536)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS) + [MICRODECODER], default="w4a16_gemv_m1")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-extra", action="store_true")
    ap.add_argument("--repeats", type=int, default=7)
    args = ap.parse_args()
    if args.impl == "reference":
        world = int(os.environ.get("WORLD_SIZE", "1"))
        rank = int(os.environ.get("RANK", "0"))
        run_reference(args, world, rank)
        return
    world, rank, local = dist_setup(args.gpus)
    if args.workload == MICRODECODER:
        run_microdecoder(args, world, rank, local)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
