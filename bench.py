#!/usr/bin/env python
"""Benchmark of the quantized tensor-core GEMM path on GB300.

One step = one pass of the whole hot path over synthetic inputs resident in
HBM:
  qgemm_s8   8192 x 8192 x 8192, int8 uniform [-128,127]  -> int32 (exact)
  qgemm_s4   8192 x 8192 x 8192, int4 uniform [-8,7]      -> int32 (exact)
  gemm_f16   8192 x 8192 x 8192, N(0,1) fp16 -> fp16 (fp32 accumulation)
  w4a16_gemm M=1, N=K=4096, group 128, one call per weight set over a
             rotation of distinct weight sets totalling > 2x L2 (a decode
             step through consecutive layers); the same rotation at M=16
             and M=128
  w4a4       quantize X (4096 x 8192 fp32) with X.U (rank 32), then the
             block-scaled GEMM against W (8192 x 8192) quantized and
             prepared once, as inference weights are + XU.V + b
L2 is flushed (a 256 MiB write) before every op; every op's working set is
also larger than L2.

After the timed step, `sweep` times the square GEMMs at N = 512 ... 4096
(the INT8 512 and INT4 2048 workloads among them) back to back, L2-hot
where the working set fits in L2 and marked so; `cpu_baseline.per_config`
times the oracle per workload (in full where it finishes in seconds, else on
a 256-row sample, extrapolated to the whole problem and marked so).

Headline `value`: INT8 GEMM TOPS at N=8192 (2*N^3 / time of qgemm_s8,
including its operand conversion).  `breakdown` holds every op's throughput
and roofline fraction.  `--impl reference` times the CPU oracle instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "INT8/INT4 GEMM TOPS at N=8192 & % tensor peak; W4A16 M=1 HBM GB/s"
N_SQ = 8192
W16_N = W16_K = 4096
W16_MS = (1, 16, 128)
W4_M, W4_N, W4_K, W4_R = 4096, 8192, 8192, 32
FLUSH_BYTES = 256 << 20

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# Nominal dense tensor rates relative to bf16/fp16 (2.25 PFLOP/s): fp8 4.5, fp4 13.5.
FP8_RATIO, FP4_RATIO = 2.0, 6.0
# DRAM bytes (read + write) of one qgemm_s8 main-kernel launch at 8192^3, from
# Nsight Compute (dram__bytes_read.sum + dram__bytes_write.sum); None until
# measured for the current kernel (the capture command is in the profiles).
S8_MAIN_DRAM_BYTES = 2 * (531950336 + 118928384)
S8_TRAFFIC_SOURCE = ("one launch at 4096x8192x8192 (-k tc_gemm2 -c 1), read + write bytes scaled by "
                     "the tile count (x2) to 8192^3 (the tc_gemm2 traffic summary under profiles/)")

# Performance-regression floors: (breakdown entry, key) -> lowest accepted
# fraction of its peak, about 15% under what GB300 measures.  The line
# reports which floors were missed; --check-floors also exits 1 on a miss.
FLOORS = {
    ("int8_gemm_8192", "frac_of_f16_peak"): 0.69,
    ("int4_gemm_8192", "frac_of_fp8_peak"): 0.64,
    ("fp16_gemm_8192", "frac_of_f16_peak"): 0.77,
    ("w4a16_m1_4096", "frac_of_hbm"): 0.32,
    ("w4a16_m16_4096", "frac_of_hbm"): 0.18,
    ("w4a16_m128_4096", "frac_of_hbm"): 0.13,
    ("w4a4_4096x8192x8192_r32", "frac_of_fp8_peak"): 0.16,
}

# Square sweep sizes measured after the step (8192 is the step itself).
SWEEP_N = (512, 1024, 2048, 4096)

# One-knob ablations (--ablate NAME): the library setter, the values tried
# (the default first) and the ops whose speed the knob can change.  The
# W4A16 rotations are CUDA graphs: a knob that changes the kernels they
# launch re-captures them.
RECAPTURE_W16 = ("pdl", "w4a16_tc")
ABLATIONS = {
    "gemm_path": ("qg_set_gemm_path", (0, 1, 2), ("s8", "s4", "f16", "w4a4_gemm")),
    "w4a4_tile": ("qg_set_w4a4_pair_form", (0, 1), ("w4a4_gemm",)),
    "pdl": ("qg_set_pdl", (1, 0), ("w4a16", "w4a16_m16", "w4a16_m128")),
    "w4a16_tc": ("qg_set_w4a16_tc_form", (0, 1), ("w4a16_m128",)),
    "s8_chunk": ("qg_set_s8_chunk", (16, 8, 4), ("s8",)),
    "l2_policy": ("qg_set_l2_policy", (0, 1, 2), ("s8", "s4", "f16")),
}


def check_floors(breakdown: dict, floors: dict = FLOORS) -> dict:
    """Compares the breakdown's roofline fractions with the floors."""
    failed = []
    for (entry, key), floor in floors.items():
        got = breakdown.get(entry, {}).get(key)
        if got is None or got < floor:
            failed.append({"op": entry, "key": key, "value": got, "floor": floor})
    return {"ok": not failed, "failed": failed}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


def replica_times(dist, device, total_ms: float, s8_ms: float):
    """Replicas only: every rank runs the same step on its own GPU.  The job
    takes as long as its slowest rank, so both the step total and the INT8
    GEMM time are the maximum over ranks (one all_reduce); without a process
    group they are returned as they are."""
    if dist is None:
        return total_ms, s8_ms
    import torch
    t = torch.tensor([total_ms, s8_ms], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t[0].item()), float(t[1].item())


def job_tops(ops_per_rank_step: float, steps: int, world: int, max_ms: float) -> float:
    """Whole-job throughput: the work of all ranks over the slowest rank's time."""
    return world * ops_per_rank_step * steps / (max_ms * 1e-3) / 1e12


def env_rank():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi clock/throttle samples (every 50 ms); stop(t0, t1) keeps the
    samples taken inside the timed region [t0, t1] (time.time() seconds)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,timestamp")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    @staticmethod
    def _when(stamp: str):
        """Seconds since the epoch of an nvidia-smi timestamp (local time)."""
        import datetime
        for fmt in ("%Y/%m/%d %H:%M:%S.%f", "%Y/%m/%d %H:%M:%S"):
            try:
                return datetime.datetime.strptime(stamp, fmt).timestamp()
            except ValueError:
                pass
        return None

    def stop(self, t0: float | None = None, t1: float | None = None):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        rows = []
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 10:
                continue
            try:
                rows.append((self._when(parts[9]), float(parts[1]), float(parts[2]),
                             {n for n, v in zip(names, parts[5:9]) if v.lower() == "active"}))
            except ValueError:
                continue
        inside = [r for r in rows if t0 is not None and r[0] is not None and t0 <= r[0] <= t1]
        use = inside if inside else rows
        return {"sm_mhz": statistics.median(r[1] for r in use) if use else None,
                "sm_max_mhz": max(r[2] for r in use) if use else None,
                "reasons": sorted(set().union(*(r[3] for r in use))) if use else [],
                "samples": len(use), "samples_in_timed_region": len(inside),
                "sampling_ms": 50}


# --------------------------------------------------------------- workload

class Workload:
    """Synthetic inputs of every op, resident on the device."""

    def __init__(self, dev):
        import numpy as np
        import torch
        import bit_quantized_tensor_gb300 as qg
        from bit_quantized_tensor_gb300 import inputs
        self.qg, self.torch, self.dev = qg, torch, dev

        def t(a):
            return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

        n = N_SQ
        self.A8, self.B8 = t(inputs.s8_uniform(n, n, 1002)), t(inputs.s8_uniform(n, n, 2002))
        self.A4 = t(inputs.s4_packed_uniform(n, n, 1002))
        self.B4 = t(inputs.s4_packed_uniform(n, n, 2002))
        self.Af, self.Bf = t(inputs.f16_normal(n, n, 1002)), t(inputs.f16_normal(n, n, 2002))
        self.C32 = torch.empty((n, n), dtype=torch.int32, device=dev)
        self.C16 = torch.empty((n, n), dtype=torch.float16, device=dev)
        self.ws8 = torch.empty(qg.workspace_size(qg.QG_OP_S8, n, n, n), dtype=torch.uint8, device=dev)
        self.ws4 = torch.empty(qg.workspace_size(qg.QG_OP_S4, n, n, n), dtype=torch.uint8, device=dev)

        # W4A16: distinct weight sets totalling more than 2x L2
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        per_set = W16_N * W16_K // 2 + W16_N * (W16_K // 128) * 2
        self.w16_sets = max(8, 2 * l2 // per_set + 2)
        # decode (M=1) plus the M=16 and M=128 shapes of the same layer
        self.X16 = {m: t(inputs.f16_normal(m, W16_K, 1003)) for m in W16_MS}
        self.W16 = [t(inputs.s4_packed_uniform(W16_N, W16_K, 2003 + 100 * i))
                    for i in range(self.w16_sets)]
        self.S16 = [t(inputs.f16_uniform(W16_N, W16_K // 128, 0.005, 0.02, 3003 + 100 * i))
                    for i in range(self.w16_sets)]
        self.Y16 = {m: torch.empty((m, W16_N), dtype=torch.float16, device=dev) for m in W16_MS}
        self.w16_bytes = {m: per_set + 2 * m * W16_K + 2 * m * W16_N for m in W16_MS}

        # W4A4: weights quantized once (outside any timed region)
        self.X4 = t(inputs.f32_normal(W4_M, W4_K, 1004))
        Wf = t(inputs.f32_normal(W4_N, W4_K, 2004))
        # low-rank factors in linear-layer weight layout: Ut rank x K, Vt N x rank
        self.Ut = t(inputs.f16_normal(W4_K, W4_R, 3004, sigma=0.02).T)
        self.Vt = t(inputs.f16_normal(W4_R, W4_N, 3005, sigma=0.02).T)
        self.bias = t(inputs.f16_normal(1, W4_N, 3006, sigma=0.1)[0])
        self.qw, self.sw, _ = qg.w4a4_quantize(Wf)
        del Wf
        self.q_out = (torch.empty((W4_M, W4_K // 2), dtype=torch.uint8, device=dev),
                      torch.empty((W4_M, W4_K // 64), dtype=torch.float16, device=dev),
                      torch.empty((W4_M, W4_R), dtype=torch.float16, device=dev))
        self.Y4 = torch.empty((W4_M, W4_N), dtype=torch.float16, device=dev)
        self.ws_w4 = torch.empty(qg.workspace_size(qg.QG_OP_W4A4, W4_M, W4_N, W4_K),
                                 dtype=torch.uint8, device=dev)
        # the weight side prepared once, as weights are (reported beside the step)
        self.packed_w4 = qg.w4a4_prepack_weights(self.qw, self.sw, W4_K)
        self.ws_w4p = torch.empty(qg.workspace_size(qg.QG_OP_W4A4_PREPACKED, W4_M, W4_N, W4_K),
                                  dtype=torch.uint8, device=dev)
        self.flush_buf = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
        torch.cuda.synchronize()
        # The decode rotation is replayed as one CUDA graph (programmatic
        # dependent launch edges are kept), so host launch cost is not timed.
        self.capture_w16()

    def capture_w16(self):
        """(Re)captures the W4A16 rotations, e.g. after the PDL switch changed."""
        torch = self.torch
        self.w16_graph = {}
        for m in W16_MS:
            self._w4a16_calls(m)
            torch.cuda.synchronize()
            self.w16_graph[m] = torch.cuda.CUDAGraph()
            with torch.cuda.graph(self.w16_graph[m]):
                self._w4a16_calls(m)
            torch.cuda.synchronize()

    # each op returns the number of library kernels it launched
    def s8(self):
        self.qg.qgemm_s8(self.A8, self.B8, C=self.C32, ws=self.ws8)
        return 2  # operand expansion (A and B in one launch) + GEMM

    def s4(self):
        self.qg.qgemm_s4(self.A4, self.B4, N_SQ, C=self.C32, ws=self.ws4)
        return 2

    def f16(self):
        self.qg.gemm_f16(self.Af, self.Bf, C=self.C16)
        return 1

    def _w4a16_calls(self, m):
        for i in range(self.w16_sets):
            self.qg.w4a16_gemm(self.X16[m], self.W16[i], self.S16[i], Y=self.Y16[m])

    def w4a16(self):
        self.w16_graph[1].replay()
        return self.w16_sets

    def w4a16_m16(self):
        self.w16_graph[16].replay()
        return self.w16_sets

    def w4a16_m128(self):
        self.w16_graph[128].replay()
        return self.w16_sets

    def w4a4_quant(self):
        self.qg.w4a4_quantize(self.X4, self.Ut, out=self.q_out)
        return 1

    def w4a4_gemm(self):
        """The GEMM against weights prepared once (w4a4_prepack_weights)."""
        q, s, xu = self.q_out
        self.qg.w4a4_gemm_prepacked(q, s, self.packed_w4, W4_N, W4_K, XU=xu, Vt=self.Vt, bias=self.bias,
                                    Y=self.Y4, ws=self.ws_w4p)
        return 3  # X operand expansion, X scale transpose, GEMM

    def w4a4_gemm_unprepared(self):
        """The same GEMM from the quantized weights, converted on every call."""
        q, s, xu = self.q_out
        self.qg.w4a4_gemm(q, s, self.qw, self.sw, W4_K, XU=xu, Vt=self.Vt, bias=self.bias,
                          Y=self.Y4, ws=self.ws_w4)
        return 4  # operand expansion, two scale transposes, GEMM

    def flush(self):
        self.flush_buf.fill_(1)


WORKLOAD = ("INT8/INT4/FP16 GEMM 8192^3, W4A16 M=1/16/128 N=K=4096 g128, "
            "W4A4 4096x8192x8192 r32, weights prepared once (one step = all eight ops)")
OPS = ["s8", "s4", "f16", "w4a16", "w4a16_m16", "w4a16_m128", "w4a4_quant", "w4a4_gemm"]
MAIN_KERNEL_OPS = {"s8", "s4", "f16", "w4a4_gemm"}  # ops with a timed tcgen05 GEMM kernel


def run_ours(args, rank, world, local_rank):
    import torch
    import bit_quantized_tensor_gb300 as qg

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    qg.lib()
    wl = Workload(dev)
    stream = torch.cuda.current_stream()

    ev = {op: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)] for op in OPS}
    kev = {op: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(args.steps)] for op in MAIN_KERNEL_OPS}
    for lst in list(ev.values()) + list(kev.values()):
        for a, b in lst:  # instantiate the driver events
            a.record(stream)
            b.record(stream)
    torch.cuda.synchronize()

    def step(i=None):
        launches = 0
        for op in OPS:
            wl.flush()
            if i is not None and op in kev:
                k0, k1 = kev[op][i]
                qg.lib().qg_set_profile_events(k0.cuda_event, k1.cuda_event)
            if i is not None:
                ev[op][i][0].record(stream)
            launches += getattr(wl, op)()
            if i is not None:
                ev[op][i][1].record(stream)
            qg.lib().qg_set_profile_events(None, None)
        return launches

    for _ in range(max(args.warmup, 0)):
        step()
    torch.cuda.synchronize()
    assert qg.device_status() == qg.QG_OK, "device-side wait timed out during warm-up"

    clocks = ClockSampler(local_rank)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    t0 = time.perf_counter()
    w0 = time.time()
    launches = 0
    for i in range(args.steps):
        launches += step(i)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    w1 = time.time()
    if dist:
        dist.barrier()
    clk = clocks.stop(w0, w1)
    assert qg.device_status() == qg.QG_OK, "device-side wait timed out in the timed region"

    # W4A4 with the weights converted on every call: timed after the step,
    # same flush and events
    unp = []
    for i in range(-max(args.warmup, 0), min(args.steps, 50)):
        wl.flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        wl.w4a4_gemm_unprepared()
        b.record(stream)
        if i >= 0:
            unp.append((a, b))
    torch.cuda.synchronize()
    w4_unp_ms = statistics.median(a.elapsed_time(b) for a, b in unp)
    peaks, peak_src = load_peaks()
    bf16 = float(peaks["bf16_tflops"])
    hbm = float(peaks["hbm_gbs"])
    sweep = (measure_sweep(wl, stream, bf16, steps=max(5, min(args.steps, 30)), warmup=max(args.warmup, 1))
             if args.sweep else None)

    t_op = {op: [a.elapsed_time(b) for a, b in ev[op]] for op in OPS}          # ms
    t_k = {op: [a.elapsed_time(b) for a, b in kev[op]] for op in MAIN_KERNEL_OPS}
    step_ms = [sum(t_op[op][i] for op in OPS) for i in range(args.steps)]
    total_ms, s8_ms = replica_times(dist, dev, sum(step_ms), sum(t_op["s8"]))

    med = {op: statistics.median(v) for op, v in t_op.items()}
    medk = {op: statistics.median(v) for op, v in t_k.items()}
    gemm_ops = 2.0 * N_SQ ** 3
    w4_ops = 2.0 * W4_M * W4_N * W4_K + 2.0 * W4_M * W4_N * W4_R

    def tops(ops, ms):
        return ops / (ms * 1e-3) / 1e12

    s8_tops = job_tops(gemm_ops, args.steps, world, s8_ms)

    w16_call_us = med["w4a16"] * 1e3 / wl.w16_sets
    w16_gbs = wl.w16_bytes[1] / (w16_call_us * 1e-6) / 1e9

    def w16_line(op, m):
        us = med[op] * 1e3 / wl.w16_sets
        gbs = wl.w16_bytes[m] / (us * 1e-6) / 1e9
        return {"GB/s": round(gbs, 1), "frac_of_hbm": round(gbs / hbm, 3), "us_per_call": round(us, 3),
                "TFLOPS": round(2.0 * m * W16_N * W16_K / (us * 1e-6) / 1e12, 2),
                "weight_sets": wl.w16_sets}
    breakdown = {
        "int8_gemm_8192": {"TOPS": round(tops(gemm_ops, med["s8"]), 1),
                           "kernel_TOPS": round(tops(gemm_ops, medk["s8"]), 1),
                           "mma_kind": "f16 (int8 carried exactly in fp16, fp32 chunks of K<=1024)",
                           "frac_of_f16_peak": round(tops(gemm_ops, med["s8"]) / bf16, 3)},
        "int4_gemm_8192": {"TOPS": round(tops(gemm_ops, med["s4"]), 1),
                           "kernel_TOPS": round(tops(gemm_ops, medk["s4"]), 1),
                           "mma_kind": "f8f6f4 e4m3 (int4 carried exactly)",
                           "frac_of_fp8_peak": round(tops(gemm_ops, med["s4"]) / (FP8_RATIO * bf16), 3)},
        "fp16_gemm_8192": {"TFLOPS": round(tops(gemm_ops, med["f16"]), 1),
                           "frac_of_f16_peak": round(tops(gemm_ops, med["f16"]) / bf16, 3)},
        "w4a16_m1_4096": {"GB/s": round(w16_gbs, 1), "us_per_call": round(w16_call_us, 3),
                          "frac_of_hbm": round(w16_gbs / hbm, 3), "weight_sets": wl.w16_sets,
                          "launch": "CUDA graph of the rotation, programmatic dependent launch"},
        "w4a16_m16_4096": w16_line("w4a16_m16", 16),
        "w4a16_m128_4096": w16_line("w4a16_m128", 128),
        "w4a4_4096x8192x8192_r32": {
            "quantize_us": round(med["w4a4_quant"] * 1e3, 1),
            "quantize_GB/s": round(W4_M * W4_K * 4 / (med["w4a4_quant"] * 1e-3) / 1e9, 1),
            "gemm_us": round(med["w4a4_gemm"] * 1e3, 1),
            "gemm": "w4a4_gemm_prepacked: weights prepared once by w4a4_prepack_weights; per call "
                    "the X operand conversion, its scale table and the GEMM kernel",
            "TOPS": round(tops(w4_ops, med["w4a4_quant"] + med["w4a4_gemm"]), 1),
            "kernel_TOPS": round(tops(w4_ops, medk["w4a4_gemm"]), 1),
            "mma_kind": "f8f6f4 e4m3 exact 64-block partials, scales applied in fp32",
            "frac_of_fp8_peak": round(tops(w4_ops, med["w4a4_quant"] + med["w4a4_gemm"])
                                      / (FP8_RATIO * bf16), 3),
            "kernel_frac_of_fp8_peak": round(tops(w4_ops, medk["w4a4_gemm"]) / (FP8_RATIO * bf16), 3),
            "mfu_vs_fp4_peak": round(tops(w4_ops, med["w4a4_quant"] + med["w4a4_gemm"])
                                     / (FP4_RATIO * bf16), 3),
            "gemm_unprepared_us": round(w4_unp_ms * 1e3, 1),
            "unprepared": "w4a4_gemm (weights converted on every call), timed after the step"},
        "op_ms_median": {op: round(v, 4) for op, v in med.items()},
    }
    k_ms = medk["s8"]
    achieved = tops(gemm_ops, k_ms)
    roofline = {"bound": "tensor",
                "kernel": "tc_gemm2_kernel<Tc2Cfg<F16,S32>> (qgemm_s8 main GEMM, CTA pairs)",
                "achieved": round(achieved, 1), "peak": bf16, "unit": "TFLOP/s",
                "peak_source": f"{peak_src} bf16 dense (fp16 kind runs at the bf16 rate)",
                "frac": round(achieved / bf16, 3), "traffic": S8_MAIN_DRAM_BYTES,
                "traffic_unit": "bytes per launch (DRAM read + write, Nsight Compute; see traffic_source)",
                "traffic_source": S8_TRAFFIC_SOURCE,
                # the method's bytes: int8 A and B in, int32 C out
                "algorithmic_bytes": 2 * N_SQ * N_SQ + 4 * N_SQ * N_SQ,
                # what this kernel must move at least: its fp16 copies of A and B, int32 C
                "kernel_operand_bytes": 2 * 2 * N_SQ * N_SQ + 4 * N_SQ * N_SQ}

    result = {
        "metric": METRIC, "value": round(s8_tops, 1), "unit": "TOPS", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total_ms / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "s8", "data": "synthetic",
        "config": {"workload": WORKLOAD, "N": N_SQ,
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "l2": "256 MiB write before every op; every working set > L2",
                   "wall_s_timed_region": round(wall, 3)},
        "breakdown": breakdown, "sweep": sweep, "roofline": roofline, "clocks": clk,
        "gpu_launches": launches, "floors": check_floors(breakdown),
    }
    if rank == 0 and args.e2e:
        result["e2e"] = measure_e2e(wl, args)
    if rank == 0 and world == 1 and args.cpu_baseline:
        result["cpu_baseline"] = oracle_baseline(args.cpu_seconds)
        result["cpu_baseline"]["per_config"] = oracle_per_config()
    if dist:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(result))
    return result


def run_ablation(args, local_rank):
    """Times the ops a knob can change at each of its values (same inputs,
    flushes and events as the main step) and prints one JSON line per value:
    an ablation of one parameter at a time, not a bench line."""
    import torch
    import bit_quantized_tensor_gb300 as qg

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    qg.lib()
    wl = Workload(dev)
    stream = torch.cuda.current_stream()
    setter, values, ops = ABLATIONS[args.ablate]
    try:
        for v in values:
            assert getattr(qg.lib(), setter)(v) == qg.QG_OK
            if args.ablate in RECAPTURE_W16:
                wl.capture_w16()
            ev = {op: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                       for _ in range(args.steps)] for op in ops}
            for i in range(-max(args.warmup, 0), args.steps):
                for op in ops:
                    wl.flush()
                    if i >= 0:
                        ev[op][i][0].record(stream)
                    getattr(wl, op)()
                    if i >= 0:
                        ev[op][i][1].record(stream)
            torch.cuda.synchronize()
            assert qg.device_status() == qg.QG_OK
            med = {op: statistics.median(a.elapsed_time(b) for a, b in ev[op]) for op in ops}
            print(json.dumps({"ablate": args.ablate, "setting": v, "default": v == values[0],
                              "steps": args.steps, "op_ms_median": {op: round(t, 4) for op, t in med.items()}}))
    finally:
        getattr(qg.lib(), setter)(values[0])
        if args.ablate in RECAPTURE_W16:
            wl.capture_w16()


def measure_e2e(wl, args):
    """The INT8 GEMM end to end through the public binding: qgemm_s8_host
    with A and B in page-locked host memory and C written back to page-locked
    host memory.  Every step's host-to-device copies of A and B and the
    device-to-host copy of C happen inside the call (overlapped with the
    conversion and GEMM of finished pieces on the library's own streams) and
    inside the timed region, which runs from the call to the stream
    synchronize on the host clock."""
    import torch
    qg, n = wl.qg, N_SQ
    hA = wl.A8.cpu().pin_memory()
    hB = wl.B8.cpu().pin_memory()
    hC = torch.empty((n, n), dtype=torch.int32).pin_memory()
    ws = torch.empty(qg.workspace_size(qg.QG_OP_S8_HOST, n, n, n), dtype=torch.uint8, device=wl.dev)
    stream = torch.cuda.current_stream()

    def once():
        qg.qgemm_s8_host(hA, hB, C=hC, ws=ws, stream=stream)
        stream.synchronize()

    for _ in range(2):
        once()
    head = qg.qgemm_s8(wl.A8[:4], wl.B8).cpu()
    assert torch.equal(hC[:4], head), "end-to-end result differs from the device result"
    ts = []
    for _ in range(max(3, args.steps)):
        t0 = time.perf_counter()
        once()
        ts.append(time.perf_counter() - t0)
    t = statistics.median(ts)
    return {"value": round(2.0 * n ** 3 / t / 1e12, 1), "unit": "TOPS",
            "h2d_bytes_per_step": 2 * n * n, "d2h_bytes_per_step": 4 * n * n,
            "op": "qgemm_s8_host 8192^3 from and to pinned host memory (8 x 2 pieces: copy-in, "
                  "conversion + GEMM and copy-out overlapped on the library's three streams)"}


def sweep_working_set(op: str, n: int) -> int:
    """Bytes one call touches in HBM/L2: inputs, output and the converted
    operand copies it writes and reads."""
    if op == "s8":
        return 2 * n * n + 4 * n * n + 2 * 2 * n * n
    if op == "s4":
        return n * n + 4 * n * n + 2 * n * n
    return 2 * 2 * n * n + 2 * n * n


GRAPH_CALLS = 20


def graph_ms_per_call(fn, stream, reps: int) -> float:
    """Median over `reps` replays (timed on `stream`, the current stream) of
    a CUDA graph of GRAPH_CALLS calls of `fn`, divided by GRAPH_CALLS (ms
    per call)."""
    import torch
    fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):  # the library launches on the capture stream
        for _ in range(GRAPH_CALLS):
            fn()
    g.replay()
    torch.cuda.synchronize()
    times = []
    for _ in range(max(reps, 3)):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        g.replay()
        b.record(stream)
        b.synchronize()
        times.append(a.elapsed_time(b) / GRAPH_CALLS)
    del g
    return statistics.median(times)


def measure_sweep(wl, stream, bf16: float, steps: int = 30, warmup: int = 3,
                  sizes=SWEEP_N) -> dict:
    """The square GEMMs at the sweep sizes: back to back (no flush), median
    of `steps` calls, the whole call and its main kernel (library-recorded
    events).  A size whose working set fits in L2 is reported L2-hot."""
    import numpy as np
    import torch
    from bit_quantized_tensor_gb300 import inputs
    qg, dev = wl.qg, wl.dev
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    peak = {"s8": bf16, "s4": FP8_RATIO * bf16, "f16": bf16}
    kind = {"s8": "f16", "s4": "fp8", "f16": "f16"}
    out = {}

    def t(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    for n in sizes:
        A8, B8 = t(inputs.s8_uniform(n, n, 1002)), t(inputs.s8_uniform(n, n, 2002))
        A4, B4 = t(inputs.s4_packed_uniform(n, n, 1002)), t(inputs.s4_packed_uniform(n, n, 2002))
        Af, Bf = t(inputs.f16_normal(n, n, 1002)), t(inputs.f16_normal(n, n, 2002))
        C32 = torch.empty((n, n), dtype=torch.int32, device=dev)
        C16 = torch.empty((n, n), dtype=torch.float16, device=dev)
        ws8 = torch.empty(qg.workspace_size(qg.QG_OP_S8, n, n, n), dtype=torch.uint8, device=dev)
        ws4 = torch.empty(qg.workspace_size(qg.QG_OP_S4, n, n, n), dtype=torch.uint8, device=dev)
        calls = {"s8": lambda: qg.qgemm_s8(A8, B8, C=C32, ws=ws8),
                 "s4": lambda: qg.qgemm_s4(A4, B4, n, C=C32, ws=ws4),
                 "f16": lambda: qg.gemm_f16(Af, Bf, C=C16)}
        for op, fn in calls.items():
            evs = []
            for i in range(-warmup, steps):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                ka, kb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                ka.record(stream)
                kb.record(stream)
                qg.lib().qg_set_profile_events(ka.cuda_event, kb.cuda_event)
                a.record(stream)
                fn()
                b.record(stream)
                qg.lib().qg_set_profile_events(None, None)
                if i >= 0:
                    evs.append((a, b, ka, kb))
            torch.cuda.synchronize()
            ms_call = statistics.median(a.elapsed_time(b) for a, b, _, _ in evs)
            kms = statistics.median(ka.elapsed_time(kb) for _, _, ka, kb in evs)
            # The same calls replayed as a CUDA graph of GRAPH_CALLS back to
            # back: per-call GPU time without the host's enqueue latency,
            # which dominates a single small call timed from the host.
            ms = graph_ms_per_call(fn, stream, steps)
            ops = 2.0 * n ** 3
            ws = sweep_working_set(op, n)
            out[f"{'int8' if op == 's8' else 'int4' if op == 's4' else 'fp16'}_{n}"] = {
                "TOPS" if op != "f16" else "TFLOPS": round(ops / ms / 1e9, 1),
                "kernel_TOPS": round(ops / kms / 1e9, 1),
                f"frac_of_{kind[op]}_peak": round(ops / ms / 1e9 / peak[op], 3),
                f"kernel_frac_of_{kind[op]}_peak": round(ops / kms / 1e9 / peak[op], 3),
                "us": round(ms * 1e3, 2), "us_single_call": round(ms_call * 1e3, 2),
                "working_set_bytes": ws,
                "timing": f"us: a CUDA graph of {GRAPH_CALLS} back-to-back calls, per call; "
                          "us_single_call: one call between events (host enqueue included); "
                          "kernel_TOPS: the main kernel between library-recorded events of a single call",
                "l2": "hot (working set fits in L2, back-to-back calls)" if ws <= l2
                      else "working set larger than L2 (back-to-back calls)"}
        del A8, B8, A4, B4, Af, Bf, C32, C16, ws8, ws4
    assert qg.device_status() == qg.QG_OK, "device-side wait timed out in the sweep"
    return out


def oracle_per_config() -> dict:
    """The CPU oracle timed per workload on the host cores: in full where it
    finishes in seconds (INT8 512, INT4 2048, the sweep up to 2048, W4A16 at
    M = 1, 16, 128), on the first rows of the output otherwise (N = 4096 and
    8192: 128 rows of the integer GEMMs, 32 of the fp64 FP16 GEMM; 64 rows of
    the W4A4 GEMM), with the time for the whole problem extrapolated linearly
    in rows and marked so.  About 15 s of host time in all."""
    import oracle
    from bit_quantized_tensor_gb300 import inputs
    oracle.build()
    res = {}

    def timed(label, ops, rows_done, rows_all, fn, unit="TOPS"):
        t0 = time.perf_counter()
        fn()
        dt = time.perf_counter() - t0
        full = dt * rows_all / rows_done
        res[label] = {"seconds": round(dt, 3), "rows": rows_done, "of_rows": rows_all,
                      "extrapolated": rows_done < rows_all,
                      "seconds_whole_problem": round(full, 2),
                      unit: round(ops / full / 1e12, 6)}

    for n in SWEEP_N + (N_SQ,):
        r = n if n <= 2048 else 128
        A8, B8 = inputs.s8_uniform(r, n, 1002), inputs.s8_uniform(n, n, 2002)
        timed(f"int8_{n}", 2.0 * n ** 3, r, n, lambda: oracle.gemm_s8(A8, B8))
        A4, B4 = inputs.s4_packed_uniform(r, n, 1002), inputs.s4_packed_uniform(n, n, 2002)
        timed(f"int4_{n}", 2.0 * n ** 3, r, n, lambda: oracle.gemm_s4(A4, B4, n))
        r = n if n <= 2048 else 32
        Af, Bf = inputs.f16_normal(r, n, 1002), inputs.f16_normal(n, n, 2002)
        timed(f"fp16_{n}", 2.0 * n ** 3, r, n, lambda: oracle.gemm_f16(Af, Bf), unit="TFLOPS")
    W = inputs.s4_packed_uniform(W16_N, W16_K, 2003)
    S = inputs.f16_uniform(W16_N, W16_K // 128, 0.005, 0.02, 3003)
    for m in W16_MS:
        X = inputs.f16_normal(m, W16_K, 1003)
        timed(f"w4a16_m{m}_4096", 2.0 * m * W16_N * W16_K, m, m, lambda: oracle.w4a16(X, W, S, 128))
    r = 64
    X4 = inputs.f32_normal(r, W4_K, 1004)
    qx, sx = oracle.w4a4_quantize(X4, 64)
    qw, sw = oracle.w4a4_quantize(inputs.f32_normal(W4_N, W4_K, 2004), 64)
    U = inputs.f16_normal(W4_K, W4_R, 3004, sigma=0.02)
    V = inputs.f16_normal(W4_R, W4_N, 3005, sigma=0.02)
    b = inputs.f16_normal(1, W4_N, 3006, sigma=0.1)[0]
    xu = oracle.lowrank_xu(X4, U)
    timed("w4a4_4096x8192x8192_r32", 2.0 * W4_M * W4_N * W4_K + 2.0 * W4_M * W4_N * W4_R, r, W4_M,
          lambda: oracle.w4a4_gemm(qx, sx, qw, sw, 64, W4_K, XU=xu, V=V, bias=b))
    return {"cores": oracle.threads(), "kind": "oracle", "configs": res}


def oracle_operands():
    """The seeded 8192^3 INT8 operands of the headline GEMM (host arrays)."""
    from bit_quantized_tensor_gb300 import inputs
    return inputs.s8_uniform(N_SQ, N_SQ, 1002), inputs.s8_uniform(N_SQ, N_SQ, 2002)


def oracle_baseline(seconds: float, rows: int | None = None, operands=None):
    """The CPU oracle on a bounded sample of the INT8 GEMM: `rows` rows of
    C = A . B^T at N = K = 8192 (sized to about `seconds` when None), timed on
    the host cores."""
    import oracle
    oracle.build()
    n = N_SQ
    A, B = operands if operands is not None else oracle_operands()
    cores = oracle.threads()
    if rows is None:
        probe = max(cores, 4)
        t0 = time.perf_counter()
        oracle.gemm_s8(A[:probe], B)
        dt = time.perf_counter() - t0
        rows = int(min(n, max(probe, probe * seconds / max(dt, 1e-3))))
        rows = max(cores, rows // cores * cores)
    t0 = time.perf_counter()
    oracle.gemm_s8(A[:rows], B)
    dt = time.perf_counter() - t0
    return {"value": round(2.0 * rows * n * n / dt / 1e12, 6), "unit": "TOPS", "cores": cores,
            "kind": "oracle", "seconds": round(dt, 2), "rows": rows,
            "sample": f"{rows} rows of the 8192^3 INT8 GEMM (C[rows] = A[rows] . B^T, int64 "
                      f"accumulation), {cores} threads"}


def run_reference(args, rank, world):
    """The CPU oracle as the reference arm, on the same metric."""
    if rank != 0:
        return
    import oracle
    oracle.build()
    ops = oracle_operands()
    # one sample size for every step: about cpu_seconds for the whole run
    rows = oracle_baseline(args.cpu_seconds / max(args.steps, 1), operands=ops)["rows"]
    for _ in range(max(args.warmup, 0)):
        oracle_baseline(0.0, rows=rows, operands=ops)
    vals, t0 = [], time.perf_counter()
    last = None
    for _ in range(args.steps):
        last = oracle_baseline(0.0, rows=rows, operands=ops)
        vals.append(last["value"])
    wall = time.perf_counter() - t0
    value = round(statistics.median(vals), 6)
    res = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TOPS",
           "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(wall * 1e3 / max(args.steps, 1), 1), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "s8", "data": "synthetic",
           "config": {"workload": WORKLOAD, "N": N_SQ,
                      "measured": "the headline INT8 GEMM 8192^3 only, on a bounded row sample "
                                  "per step (see cpu_baseline.sample)"},
           "cpu_baseline": {"value": value, "unit": "TOPS", "cores": last["cores"],
                            "kind": "oracle", "sample": last["sample"]},
           "e2e": {"value": value, "unit": "TOPS", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(res))


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-e2e", dest="e2e", action="store_false")
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--no-sweep", dest="sweep", action="store_false",
                    help="skip the square-GEMM sweep after the step (e.g. for a launch list of the step)")
    ap.add_argument("--cpu-seconds", type=float, default=6.0,
                    help="target CPU seconds of the oracle baseline sample")
    ap.add_argument("--check-floors", action="store_true",
                    help="exit 1 when an op falls under its regression floor")
    ap.add_argument("--ablate", choices=sorted(ABLATIONS),
                    help="time the ops one knob changes at each of its values instead (one line per value)")
    args = ap.parse_args()
    rank, world, local_rank = env_rank()
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    import __graft_entry__
    __graft_entry__.build_library()
    if args.ablate:
        if rank == 0:
            run_ablation(args, local_rank)
        return
    result = run_ours(args, rank, world, local_rank)
    if args.check_floors and rank == 0 and not result["floors"]["ok"]:
        raise SystemExit(1)


if __name__ == "__main__":
    main()
