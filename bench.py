#!/usr/bin/env python
"""Benchmark of the W8A8 quantized linear layer on one GB300 (or N replicas).

Workload: W8A8 per-channel linear, N=10240, K=2560, M in {1, 128, 1024, 4096,
8192} (seed 0; x ~ N(0,1) fp16 with 26 of the 2560 K-channels x30, weights
~ N(0, 0.02) quantized per output channel on the GPU before timing).  One
step = the whole path for every M of the sweep: per-token activation
quantization, then the INT8 GEMM (M > 1) or the INT8 matrix-vector kernel
(M = 1) with the fused dequant to fp16.

value    = sum over the sweep of 2*M*N*K integer ops / device time of the step
           (TOPS), inputs resident in HBM; L2 is flushed (a 2 x L2 write,
           then a 2 x L2 read) before every call, outside the timed events.
           Each call (quantizer and GEMM back to back, or the fused decode
           kernel) is one CUDA-event interval; the per-kernel split (detail,
           roofline) comes from a separate untimed pass with an event between
           the two kernels.
e2e      = the same metric through the C ABI's ``linear`` call with pinned
           host buffers: host->device copy of x, the layer, device->host copy
           of y, all inside the timed events; from M = 1024 on, in chunks of
           512 rows whose copies and layer calls overlap on three streams.
           The copies and linear() calls of each M are captured once into a
           CUDA graph and replayed every step (eager_value: the same calls
           enqueued by the host every step).
roofline = the dominant kernel (the GEMM at M=8192): 2*M*N*K / its average
           CUDA-event duration in the breakdown pass, against the measured
           dense fp16/bf16 tensor peak; traffic = DRAM bytes per launch from
           the committed ncu summary of that kernel, while its source is
           unchanged since the capture.
decode   = the decode matrix-vector path (M = 1) timed the way decode runs,
           layer after layer: back-to-back linear() calls over R distinct
           copies of the weights (R x 26 MB > 2 x L2), so every call streams
           its weights from HBM; GB/s = algorithmic bytes per call (INT8
           weights, their scales, x, y) / time per call.
cpu_baseline / --impl reference = the CPU oracle, as it stands, on a bounded
           sample of rows of the same workload.
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

import hashlib

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from w4a8_int8_quantized_gb300 import synth  # noqa: E402

WORKLOAD = synth.WORKLOADS["pc_sweep"]
N_OUT, K_IN, MS = WORKLOAD["N"], WORKLOAD["K"], WORKLOAD["Ms"]
METRIC = "W8A8 GEMM INT8 TOPS & ms (N=10240,K=2560,M=1..8192); decode GEMV HBM GB/s"
UNIT = "TOPS"
# Pages' M5 Pro per-channel latencies for this sweep (ms, "cider 소개",
# section "cider의 성능 측정 결과"): the same metric as a whole-sweep rate.
PAGES_MS = {1: 0.27, 128: 0.34, 1024: 1.23, 4096: 4.41, 8192: 8.71}
PAGES_TOPS = sum(2.0 * m * N_OUT * K_IN for m in MS) / (sum(PAGES_MS.values()) * 1e-3) / 1e12
E2E_CHUNK_ROWS = 512  # rows per pipelined chunk of the e2e measurement
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


GEMM_PROFILE = os.path.join(ROOT, "profiles", "gemm_tc_m8192_n10240_k2560.txt")
GEMM_SOURCE = os.path.join(ROOT, "w4a8_int8_quantized_gb300", "csrc", "gemm_tc.cu")


def gemm_traffic():
    """DRAM bytes per launch of the GEMM at M=8192 from the committed ncu
    summary, or None when the kernel source changed since that capture."""
    try:
        fields = {}
        with open(GEMM_PROFILE) as f:
            for line in f:
                if ":" in line:
                    k, v = line.split(":", 1)
                    fields[k.strip()] = v.strip()
        with open(GEMM_SOURCE, "rb") as f:
            sha = hashlib.sha256(f.read()).hexdigest()
        if fields.get("gemm_tc.cu sha256") != sha:
            return None
        return float(fields["dram bytes per launch"])
    except (OSError, KeyError, ValueError):
        return None


def config_dict():
    return {"workload": "W8A8 per-channel linear, N=10240, K=2560, M in {1,128,1024,4096,8192}",
            "N": N_OUT, "K": K_IN, "Ms": MS, "group_size": 0,
            "inputs": "seeded synthetic: x ~ N(0,1) fp16, 26 of 2560 K-channels x30; "
                      "W ~ N(0,0.02) fp16 quantized to INT8 per output channel",
            "l2": "flushed before every call (write of a 2 x L2 buffer, then a read of another), outside the timed events"}


def step_ops():
    return sum(2.0 * m * N_OUT * K_IN for m in MS)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            with open(p) as f:
                d = json.load(f)
            return d, "measured"
        except Exception:
            pass
    return dict(FALLBACK_PEAKS), "fallback"


def _peak(d, *names):
    """First numeric value among keys that contain one of `names`."""
    def walk(o, prefix=""):
        if isinstance(o, dict):
            for k, v in o.items():
                yield from walk(v, f"{prefix}{k}.")
        else:
            yield prefix[:-1], o
    for name in names:
        for k, v in walk(d):
            if k.split(".")[-1] == name and isinstance(v, (int, float)):
                return float(v)
    return None


# ------------------------------------------------------------------ clocks --

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu), "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            if self.thread is not None:
                self.thread.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------- distributed setup --

def dist_setup(backend):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, ws, device=None):
    if ws == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------------- CPU oracle --

def oracle_sample_step(rows: int, inputs):
    """The oracle on the first `rows` rows of every M of the sweep; returns
    (ops, seconds)."""
    import oracle
    ops, t = 0.0, 0.0
    wq, sw = inputs["wq_ref"], inputs["sw_ref"]
    for m in MS:
        r = min(m, rows)
        x = inputs["x"][m][:r]
        t0 = time.perf_counter()
        oracle.linear(x, wq, sw)
        t += time.perf_counter() - t0
        ops += 2.0 * r * N_OUT * K_IN
    return ops, t


def host_inputs():
    xs = {m: synth.activations(m, K_IN, seed=0, **WORKLOAD["act"]) for m in MS}
    W = synth.weights(N_OUT, K_IN, seed=0)
    return {"x": xs, "W": W}


def calibrate_rows(inputs, target_s):
    """Rows per M so that one oracle sample step takes about target_s."""
    rows = 2
    _, t = oracle_sample_step(rows, inputs)
    while t < min(0.5, target_s / 4) and rows < 8192:
        rows *= 2
        _, t = oracle_sample_step(rows, inputs)
    want = int(rows * target_s / max(t, 1e-3))
    return max(2, min(want, 8192)), t


def cpu_baseline(inputs, target_s=20.0):
    import oracle
    oracle.build()
    wq, sw = oracle.quantize_weight_int8(inputs["W"])
    inputs["wq_ref"], inputs["sw_ref"] = wq, sw
    rows, _ = calibrate_rows(inputs, target_s)
    ops, t = oracle_sample_step(rows, inputs)
    what = ("every row of every M of the sweep" if rows >= max(MS)
            else f"first {rows} rows of each M of the sweep")
    return {"value": ops / t / 1e12, "unit": UNIT, "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": f"{what} (N=10240, K=2560) through the oracle's quantize + int64 GEMM "
                      f"+ dequant; {t:.1f} s"}


def run_reference(args):
    ws, rank, _ = dist_setup("gloo")
    if rank != 0:
        return
    import oracle
    oracle.build()
    inputs = host_inputs()
    wq, sw = oracle.quantize_weight_int8(inputs["W"])
    inputs["wq_ref"], inputs["sw_ref"] = wq, sw
    # each step is a bounded sample sized so the whole run takes ~2-3 minutes
    per_step = max(1.0, 150.0 / max(1, args.steps + args.warmup))
    rows, _ = calibrate_rows(inputs, per_step)
    for _ in range(args.warmup):
        oracle_sample_step(rows, inputs)
    ops = t = 0.0
    for _ in range(args.steps):
        o, s = oracle_sample_step(rows, inputs)
        ops += o
        t += s
    value = ops / t / 1e12
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * t / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": value / PAGES_TOPS, "dtype": "int8", "data": "synthetic",
            "config": config_dict(), "impl": "reference",
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(),
                             "kind": "oracle",
                             "sample": f"first {rows} rows of each M of the sweep per step"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# -------------------------------------------------------------- GPU path --

def measure_workloads(w8, torch, device, flush_l2, l2_bytes, tflops_peak, hbm_peak, reps=20):
    """Every other workload of the layer, timed once per case with CUDA events
    (mean of `reps`; event timestamps on this GPU advance in steps of about
    2 us, so a median of single calls sits on a step and a mean over the
    jittered samples does not): the 512 x 512 per-channel layer, per group gs 128 /
    64, W4A8 at M = 2048 and M = 1, and the linear layers of an 8B-class
    decoder block at M = 4516 and M = 1.  GEMM-type calls run after an L2
    flush; decode calls run back to back over weight copies larger than L2
    (a decode step walks layer after layer).  Seeded synthetic inputs."""
    stream = torch.cuda.current_stream()

    def timed(fn, per_rep_flush=True, inner=1):
        ts = []
        for _ in range(reps):
            torch.cuda._sleep(int(2e6))  # the host enqueues the rep while the GPU waits
            if per_rep_flush:
                flush_l2()
            e0, e1 = (torch.cuda.Event(enable_timing=True) for _ in range(2))
            e0.record(stream)
            for i in range(inner):
                fn(i)
            e1.record(stream)
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1) / inner)
        return statistics.fmean(ts)

    def dev(a):
        return torch.from_numpy(a).to(device)

    out = {}

    def gemm_case(name, M, N, K, gs, wbits, act):
        x = dev(synth.activations(M, K, seed=0, **act))
        W = dev(synth.weights(N, K, seed=0))
        wq, sw = (w8.quantize_weight_int8(W, gs) if wbits == 8 else w8.pack_weight_int4(W))
        del W
        xq, sa = w8.quantize_act_per_token_h(x, gs)
        y = torch.empty((M, N), dtype=torch.float16, device=device)
        for _ in range(2):
            w8.quantize_act_per_token_h(x, gs, xq, sa)
            w8.w8a8_gemm_h(xq, sa, wq, sw, gs, wbits, y)
        q_ms = timed(lambda i: w8.quantize_act_per_token_h(x, gs, xq, sa))
        g_ms = timed(lambda i: w8.w8a8_gemm_h(xq, sa, wq, sw, gs, wbits, y))
        tops = 2.0 * M * N * K / (g_ms * 1e-3) / 1e12
        out[name] = {"M": M, "N": N, "K": K, "group_size": gs, "wbits": wbits,
                     "quant_ms": round(q_ms, 5), "gemm_ms": round(g_ms, 5),
                     "gemm_TOPS": round(tops, 1), "gemm_frac_of_peak": round(tops / tflops_peak, 4)}
        return g_ms + q_ms

    def decode_case(name, layers, wbits, act):
        """layers: [(N, K)]; one decode step = linear() on every layer in turn."""
        sets = []
        per_set = sum(n * (k if wbits == 8 else k // 2) for n, k in layers)
        copies = max(2, int(3 * l2_bytes // per_set) + 1)
        xs = [dev(synth.activations(1, k, seed=0, **act)) for _, k in layers]
        ys = [torch.empty((1, n), dtype=torch.float16, device=device) for n, _ in layers]
        base = []
        for n, k in layers:
            W = dev(synth.weights(n, k, seed=0))
            base.append(w8.quantize_weight_int8(W) if wbits == 8 else w8.pack_weight_int4(W))
            del W
        for c in range(copies):
            sets.append([(wq.clone(), sw) for wq, sw in base] if c else base)
        ws = [torch.empty(max(w8.w8a8_linear_workspace_bytes(1, k), 1), dtype=torch.uint8,
                          device=device) for _, k in layers]

        def step(i):
            for li, (wq, sw) in enumerate(sets[i % copies]):
                w8.linear(xs[li], wq, sw, 0, wbits, workspace=ws[li], y=ys[li])
        for i in range(copies):
            step(i)
        us = timed(step, per_rep_flush=False, inner=copies) * 1e3
        nbytes = sum(n * (k if wbits == 8 else k // 2) + 4 * n + 2 * k + 2 * n for n, k in layers)
        out[name] = {"layers": [list(l) for l in layers], "wbits": wbits, "weight_copies": copies,
                     "us_per_step": round(us, 3), "GBps": round(nbytes / (us * 1e-6) / 1e9, 1),
                     "frac_of_hbm": round(nbytes / (us * 1e-6) / 1e9 / hbm_peak, 4)}
        del sets

    def few_rows_case():
        """M = 2..32 rows of the N=10240, K=2560 layer: linear() (the few-row
        kernel up to 8 rows, the GEMM above) against the quantizer + the
        tensor-core GEMM on the same rows; each call after an L2 flush."""
        sweep = wl["pc_sweep"]
        W = dev(synth.weights(sweep["N"], sweep["K"], seed=0))
        wq, sw = w8.quantize_weight_int8(W)
        del W
        res = {}
        for M in (2, 4, 8, 16, 32):
            x = dev(synth.activations(M, sweep["K"], seed=0, **sweep["act"]))
            ws = torch.empty(w8.w8a8_linear_workspace_bytes(M, sweep["K"]), dtype=torch.uint8,
                             device=device)
            y = torch.empty((M, sweep["N"]), dtype=torch.float16, device=device)
            xh, sa = w8.quantize_act_per_token_h(x)
            w8.linear(x, wq, sw, workspace=ws, y=y)
            w8.w8a8_gemm_h(xh, sa, wq, sw, 0, 8, y)
            lin_ms = timed(lambda i: w8.linear(x, wq, sw, workspace=ws, y=y))

            def gemm_path(i):
                w8.quantize_act_per_token_h(x, 0, xh, sa)
                w8.w8a8_gemm_h(xh, sa, wq, sw, 0, 8, y)
            gemm_ms = timed(gemm_path)
            nbytes = sweep["N"] * sweep["K"] + 4 * sweep["N"] + M * (2 * sweep["K"] + 2 * sweep["N"])
            res[str(M)] = {"linear_us": round(lin_ms * 1e3, 3),
                           "linear_GBps": round(nbytes / (lin_ms * 1e-3) / 1e9, 1),
                           "tensor_core_gemm_us": round(gemm_ms * 1e3, 3),
                           "path": "few-row kernel" if M <= 8 else "tensor-core GEMM"}
        out["few_rows_N10240_K2560"] = res

    def weight_only_case():
        """The pages' comparison on this chip: W8A8 per channel (linear(),
        quantizer included) against the weight-only W8A16 / W4A16 GEMMs (fp16
        activations) over the N=10240, K=2560 sweep; ratio = weight-only time
        / W8A8 time, as the pages' PC/w8a16 and PC/w4a16 columns.  M = 1 runs
        the weight-only product through the tensor-core GEMM (there is no
        weight-only matrix-vector kernel)."""
        sweep = wl["pc_sweep"]
        N, K = sweep["N"], sweep["K"]
        W = dev(synth.weights(N, K, seed=0))
        wq, sw = w8.quantize_weight_int8(W)
        wp, s4 = w8.pack_weight_int4(W)
        del W
        res = {}
        for M in sweep["Ms"]:
            x = dev(synth.activations(M, K, seed=0, **sweep["act"]))
            ws = torch.empty(max(w8.w8a8_linear_workspace_bytes(M, K), 1), dtype=torch.uint8,
                             device=device)
            y = torch.empty((M, N), dtype=torch.float16, device=device)
            w8.linear(x, wq, sw, workspace=ws, y=y)
            w8.weight_only_gemm(x, wq, sw, 0, 8, y)
            w8.weight_only_gemm(x, wp, s4, 0, 4, y)
            pc = timed(lambda i: w8.linear(x, wq, sw, workspace=ws, y=y))
            w16 = timed(lambda i: w8.weight_only_gemm(x, wq, sw, 0, 8, y))
            w4 = timed(lambda i: w8.weight_only_gemm(x, wp, s4, 0, 4, y))
            ops = 2.0 * M * N * K
            res[str(M)] = {"w8a8_pc_ms": round(pc, 5), "w8a16_ms": round(w16, 5),
                           "w4a16_ms": round(w4, 5),
                           "w8a16_TFLOPs": round(ops / (w16 * 1e-3) / 1e12, 1),
                           "pc_over_w8a16": round(w16 / pc, 3), "pc_over_w4a16": round(w4 / pc, 3)}
        out["weight_only_vs_w8a8_N10240_K2560"] = res

    def in_gemm_conversion_case():
        """What quantization fused into the prefill GEMM would cost: the GEMM
        fed INT8 activation codes that its converter warps turn into fp16
        operands in shared memory (every weight tile re-converts the token
        tile) against the layer's path (fp16 codes straight to the MMA by
        TMA), at M = 8192 of the N=10240, K=2560 layer; each with its
        quantizer."""
        sweep = wl["pc_sweep"]
        M, N, K = 8192, sweep["N"], sweep["K"]
        x = dev(synth.activations(M, K, seed=0, **sweep["act"]))
        W = dev(synth.weights(N, K, seed=0))
        wq, sw = w8.quantize_weight_int8(W)
        del W
        y = torch.empty((M, N), dtype=torch.float16, device=device)
        xq, sa = w8.quantize_act_per_token(x)
        xh, sah = w8.quantize_act_per_token_h(x)
        w8.w8a8_gemm(xq, sa, wq, sw, 0, y)
        w8.w8a8_gemm_h(xh, sah, wq, sw, 0, 8, y)
        g8 = timed(lambda i: w8.w8a8_gemm(xq, sa, wq, sw, 0, y))
        g16 = timed(lambda i: w8.w8a8_gemm_h(xh, sah, wq, sw, 0, 8, y))
        q8 = timed(lambda i: w8.quantize_act_per_token(x, 0, xq, sa))
        q16 = timed(lambda i: w8.quantize_act_per_token_h(x, 0, xh, sah))
        ops = 2.0 * M * N * K
        out["activation_conversion_in_gemm_M8192"] = {
            "int8_codes_converted_in_gemm": {"gemm_ms": round(g8, 5), "quant_ms": round(q8, 5),
                                             "gemm_TOPS": round(ops / (g8 * 1e-3) / 1e12, 1)},
            "fp16_codes_by_tma": {"gemm_ms": round(g16, 5), "quant_ms": round(q16, 5),
                                  "gemm_TOPS": round(ops / (g16 * 1e-3) / 1e12, 1)}}

    wl = synth.WORKLOADS
    in_gemm_conversion_case()
    weight_only_case()
    few_rows_case()
    # the 512 x 512 per-channel layer: the whole linear() call
    small = wl["pc_small"]
    x = dev(synth.activations(128, 512, seed=0, **small["act"]))
    wq, sw = w8.quantize_weight_int8(dev(synth.weights(512, 512, seed=0)))
    y = torch.empty((128, 512), dtype=torch.float16, device=device)
    ws0 = torch.empty(w8.w8a8_linear_workspace_bytes(128, 512), dtype=torch.uint8, device=device)
    w8.linear(x, wq, sw, workspace=ws0, y=y)
    out["pc_small_M128_N512_K512"] = {"linear_ms": round(timed(
        lambda i: w8.linear(x, wq, sw, workspace=ws0, y=y)), 5)}
    for gs in wl["pg"]["gs"]:
        gemm_case(f"per_group_gs{gs}_M4096", 4096, 10240, 2560, gs, 8, wl["pg"]["act"])
    gemm_case("w4a8_M2048", 2048, 14336, 4096, 0, 4, wl["w4a8"]["act"])
    decode_case("w4a8_M1_decode", [(14336, 4096)], 4, wl["w4a8"]["act"])
    total = 0.0
    for lname, n, k in synth.BLOCK_LAYERS:
        total += gemm_case(f"block_{lname}_M4516", 4516, n, k, 0, 8, synth.BLOCK_ACT)
    ops = sum(2.0 * 4516 * n * k for _, n, k in synth.BLOCK_LAYERS)
    out["block_prefill_M4516_total"] = {"ms": round(total, 5),
                                         "TOPS": round(ops / (total * 1e-3) / 1e12, 1)}
    decode_case("block_decode_M1_step", [(n, k) for _, n, k in synth.BLOCK_LAYERS], 8,
                synth.BLOCK_ACT)
    return out


def run_ours(args):
    import ctypes

    import torch

    ws, rank, local = dist_setup("nccl")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    import w4a8_int8_quantized_gb300 as w8
    lib = w8.load()
    if not w8.w8a8_is_available():
        raise RuntimeError("libw8a8 needs a compute-capability 10.3 GPU")

    inputs = host_inputs()
    stream = torch.cuda.current_stream()
    s_ptr = ctypes.c_void_p(stream.cuda_stream)
    P = ctypes.c_void_p

    W = torch.from_numpy(inputs["W"]).to(device)
    wq, sw = w8.quantize_weight_int8(W)
    del W
    bufs = {}
    for m in MS:
        x = torch.from_numpy(inputs["x"][m]).to(device)
        # the codes in the format linear() uses: fp16 values for the GEMM
        # (M > 1), int8 for the matrix-vector kernel (M == 1)
        xq = torch.empty((m, K_IN), dtype=torch.int8 if m == 1 else torch.float16, device=device)
        sa = torch.empty((m, 1), dtype=torch.float32, device=device)
        y = torch.empty((m, N_OUT), dtype=torch.float16, device=device)
        ws_bytes = w8.w8a8_linear_workspace_bytes(m, K_IN, 0)
        wsb = torch.empty(ws_bytes, dtype=torch.uint8, device=device)
        xh = torch.from_numpy(inputs["x"][m]).pin_memory()
        yh = torch.empty((m, N_OUT), dtype=torch.float16).pin_memory()
        bufs[m] = dict(x=x, xq=xq, sa=sa, y=y, ws=wsb, xh=xh, yh=yh)
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    flush_w = torch.empty(max(2 * l2, 256 << 20) // 4, dtype=torch.int32, device=device)
    flush_r = torch.ones_like(flush_w)

    def flush_l2():
        # write a 2 x L2 buffer, then read another one: L2 ends up holding
        # clean lines of an unrelated buffer, so the timed call neither hits
        # in L2 nor pays for writing back the flush's dirty lines
        flush_w.fill_(1)
        flush_r.max()

    def check(st, what):
        if st != 0:
            raise RuntimeError(f"{what}: status {st}")

    # the two launches of linear(), called through their own C entry points
    # so that each is timed on its own
    def call_quant(m):
        if m == 1:
            return  # fused into the decode kernel
        b = bufs[m]
        f = lib.quantize_act_per_token_h
        check(f(P(b["x"].data_ptr()), m, K_IN, 0, P(b["xq"].data_ptr()),
                P(b["sa"].data_ptr()), s_ptr), "quantize")

    def call_gemm(m):
        b = bufs[m]
        if m == 1:
            # decode: linear() runs one fused kernel (quantize the row + MV)
            st = lib.linear(P(b["x"].data_ptr()), P(wq.data_ptr()), P(sw.data_ptr()), m, N_OUT,
                            K_IN, 0, 8, P(b["ws"].data_ptr()), b["ws"].numel(),
                            P(b["y"].data_ptr()), s_ptr)
        else:
            st = lib.w8a8_gemm_h(P(b["xq"].data_ptr()), P(b["sa"].data_ptr()), P(wq.data_ptr()),
                                 P(sw.data_ptr()), m, N_OUT, K_IN, 0, 8, P(b["y"].data_ptr()),
                                 s_ptr)
        check(st, "gemm")

    def call_linear(m, x, y):
        b = bufs[m]
        check(lib.linear(P(x.data_ptr()), P(wq.data_ptr()), P(sw.data_ptr()), m, N_OUT, K_IN, 0,
                         8, P(b["ws"].data_ptr()), b["ws"].numel(), P(y.data_ptr()), s_ptr),
              "linear")

    def kernel_step(record, split=False):
        # one event interval per call (the quantizer and the GEMM back to
        # back); `split` adds an event between the two kernels for the
        # per-kernel breakdown, which costs device time of its own (~2 us)
        evs = []
        for m in MS:
            flush_l2()
            e0, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(2))
            e1 = torch.cuda.Event(enable_timing=True) if split else None
            e0.record(stream)
            call_quant(m)
            if split:
                e1.record(stream)
            call_gemm(m)
            e2.record(stream)
            evs.append((m, e0, e1, e2))
        if record is not None:
            record.append(evs)

    # e2e: from M = 2 chunk_rows on, the rows go in chunks of chunk_rows, the
    # host->device copy of chunk i+1, the layer on chunk i and the
    # device->host copy of chunk i-1 overlapping on three streams (the copy
    # engines of the two directions and the SMs work at once); smaller M runs
    # copy, layer, copy in order (there the host enqueues more slowly than
    # the GPU would run chunks)
    s_h2d, s_comp, s_d2h = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    comp_ptr = ctypes.c_void_p(s_comp.cuda_stream)

    chunk_rows = args.e2e_chunk_rows

    def e2e_chunks(m):
        return m // chunk_rows if m >= 2 * chunk_rows else 1

    def linear_rows(m, r0, r1, sptr):
        b = bufs[m]
        x, y = b["x"][r0:r1], b["y"][r0:r1]
        check(lib.linear(P(x.data_ptr()), P(wq.data_ptr()), P(sw.data_ptr()), r1 - r0, N_OUT,
                         K_IN, 0, 8, P(b["ws"].data_ptr()), b["ws"].numel(), P(y.data_ptr()),
                         sptr), "linear")

    def e2e_call(m, e0, origin):
        """One M end to end: copy-in, linear(), copy-out.  `origin` is the
        stream the call starts and ends on (e0 is recorded there)."""
        b = bufs[m]
        C = e2e_chunks(m)
        if C == 1:
            with torch.cuda.stream(origin):
                b["x"].copy_(b["xh"], non_blocking=True)
            check(lib.linear(P(b["x"].data_ptr()), P(wq.data_ptr()), P(sw.data_ptr()), m, N_OUT,
                             K_IN, 0, 8, P(b["ws"].data_ptr()), b["ws"].numel(),
                             P(b["y"].data_ptr()), P(origin.cuda_stream)), "linear")
            with torch.cuda.stream(origin):
                b["yh"].copy_(b["y"], non_blocking=True)
            return
        for st in (s_h2d, s_comp, s_d2h):
            st.wait_event(e0)
        ends = []
        for i in range(C):
            r0, r1 = m * i // C, m * (i + 1) // C
            with torch.cuda.stream(s_h2d):
                b["x"][r0:r1].copy_(b["xh"][r0:r1], non_blocking=True)
                eh = torch.cuda.Event()
                eh.record(s_h2d)
            s_comp.wait_event(eh)
            linear_rows(m, r0, r1, comp_ptr)
            ec = torch.cuda.Event()
            ec.record(s_comp)
            s_d2h.wait_event(ec)
            with torch.cuda.stream(s_d2h):
                b["yh"][r0:r1].copy_(b["y"][r0:r1], non_blocking=True)
        for st in (s_h2d, s_comp, s_d2h):
            ev = torch.cuda.Event()
            ev.record(st)
            origin.wait_event(ev)

    def e2e_step(record, graphs=None):
        # eager: the host enqueues every copy and linear() call of every
        # chunk; graphs: each M's calls were captured once into a CUDA graph
        # (the same linear() calls and host copies), replayed here
        evs = []
        for m in MS:
            flush_l2()
            e0, e1 = (torch.cuda.Event(enable_timing=True) for _ in range(2))
            e0.record(stream)
            if graphs is None:
                e2e_call(m, e0, stream)
            else:
                graphs[m].replay()
            e1.record(stream)
            evs.append((m, e0, e1))
        if record is not None:
            record.append(evs)

    # warm-up (also sets the kernels' shared-memory attributes)
    for _ in range(max(3, args.warmup)):
        kernel_step(None)
    torch.cuda.synchronize()

    peaks, peak_src = load_peaks()
    rec = []
    barrier(ws)
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        torch.cuda._sleep(int(2e6))  # queue depth: the CPU enqueues ahead of the GPU
        wall0 = time.perf_counter()
        for _ in range(args.steps):
            kernel_step(rec)
        torch.cuda.synchronize()
        wall = time.perf_counter() - wall0
    barrier(ws)
    torch.cuda.synchronize()

    call_ms = {m: 0.0 for m in MS}
    for evs in rec:
        for m, e0, _, e2 in evs:
            call_ms[m] += e0.elapsed_time(e2) / args.steps
    step_ms = sum(call_ms.values())
    step_ms = max_over_ranks(step_ms, ws, device)
    value = ws * step_ops() / (step_ms * 1e-3) / 1e12

    # per-kernel breakdown (untimed pass): an event between the quantizer and
    # the GEMM of each call
    n_split = max(20, args.steps // 4)
    rec_split = []
    torch.cuda.synchronize()
    torch.cuda._sleep(int(2e6))
    for _ in range(n_split):
        kernel_step(rec_split, split=True)
    torch.cuda.synchronize()
    per_m = {m: {"quant_ms": 0.0, "gemm_ms": 0.0} for m in MS}
    for evs in rec_split:
        for m, e0, e1, e2 in evs:
            per_m[m]["quant_ms"] += e0.elapsed_time(e1) / n_split
            per_m[m]["gemm_ms"] += e1.elapsed_time(e2) / n_split

    # e2e through linear() with host buffers: eager, then as CUDA graphs
    def e2e_measure(graphs):
        for _ in range(2):
            e2e_step(None, graphs)
        rec2 = []
        torch.cuda.synchronize()
        torch.cuda._sleep(int(2e6))
        for _ in range(args.steps):
            e2e_step(rec2, graphs)
        torch.cuda.synchronize()
        ms = sum(e0.elapsed_time(e1) for evs in rec2 for _, e0, e1 in evs) / args.steps
        ms = max_over_ranks(ms, ws, device)
        return ws * step_ops() / (ms * 1e-3) / 1e12

    e2e_eager = e2e_measure(None)
    e2e_value, e2e_graph_error = e2e_eager, None
    if not args.e2e_eager_only:
        graphs = {}
        try:
            for m in MS:
                g = torch.cuda.CUDAGraph()
                cap = torch.cuda.Stream()
                with torch.cuda.graph(g, stream=cap):
                    fork = torch.cuda.Event()
                    fork.record(cap)
                    e2e_call(m, fork, cap)
                graphs[m] = g
            torch.cuda.synchronize()
        except RuntimeError as ex:  # capture refused: report the eager number and why
            e2e_graph_error = str(ex).splitlines()[0][:200]
            torch.cuda.synchronize()
        # every rank takes the same branch (the measurement has a collective)
        if max_over_ranks(0.0 if e2e_graph_error is None else 1.0, ws, device) == 0.0:
            e2e_value = e2e_measure(graphs)
        elif e2e_graph_error is None:
            e2e_graph_error = "graph capture failed on another rank"
    # the outputs the chunked three-stream path copied back must equal one
    # linear() call over all rows on one stream (bit for bit: the rows of a
    # chunk are computed exactly as in the whole call)
    e2e_mismatch = 0
    for m in MS:
        b = bufs[m]
        y_ref = torch.empty_like(b["y"])
        call_linear(m, b["x"], y_ref)
        torch.cuda.synchronize()
        e2e_mismatch += int((y_ref.cpu().view(torch.int16) != b["yh"].view(torch.int16)).sum())

    # decode, back to back over distinct weight copies
    decode = None
    if rank == 0 and not args.no_decode:
        n_copies = max(4, int(3 * l2 // (N_OUT * K_IN)) + 1)
        copies = [wq.clone() for _ in range(n_copies)]
        b1 = bufs[1]

        def decode_round():
            for c in copies:
                check(lib.linear(P(b1["x"].data_ptr()), P(c.data_ptr()), P(sw.data_ptr()), 1,
                                 N_OUT, K_IN, 0, 8, P(b1["ws"].data_ptr()), b1["ws"].numel(),
                                 P(b1["y"].data_ptr()), s_ptr), "decode")

        for _ in range(3):
            decode_round()
        torch.cuda.synchronize()
        times = []
        for _ in range(max(10, min(args.steps, 100))):
            torch.cuda._sleep(int(1e6))
            e0, e1 = (torch.cuda.Event(enable_timing=True) for _ in range(2))
            e0.record(stream)
            decode_round()
            e1.record(stream)
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1) * 1e3 / n_copies)
        us = statistics.median(times)
        dbytes = N_OUT * K_IN + N_OUT * 4 + K_IN * 2 + N_OUT * 2
        hbm = _peak(peaks, "hbm_gbs") if peak_src == "measured" else None
        hbm_src = peak_src if hbm is not None else "fallback"
        hbm = hbm if hbm is not None else FALLBACK_PEAKS["hbm_gbs"]
        decode = {"us_per_call": round(us, 3), "GBps": round(dbytes / (us * 1e-6) / 1e9, 1),
                  "bytes_per_call": dbytes, "hbm_peak_gbs": hbm,
                  "frac_of_hbm": round(dbytes / (us * 1e-6) / 1e9 / hbm, 4),
                  "peak_source": f"{hbm_src} HBM copy bandwidth",
                  "method": f"back-to-back linear() calls, M=1, over {n_copies} distinct weight "
                            f"copies; median of {len(times)} rounds"}
        del copies

    detail = {}
    for m in MS:
        q = per_m[m]["quant_ms"]
        g = per_m[m]["gemm_ms"]
        c = call_ms[m]
        # ms / TOPS: the timed call; quant_ms / gemm_ms: the breakdown pass
        d = {"ms": round(c, 5), "TOPS": round(2.0 * m * N_OUT * K_IN / (c * 1e-3) / 1e12, 3),
             "quant_ms": round(q, 5), "gemm_ms": round(g, 5),
             "gemm_TOPS": round(2.0 * m * N_OUT * K_IN / (g * 1e-3) / 1e12, 3),
             }
        if m == 1:
            # fused decode kernel: int8 weights, their scales, x (fp16), y (fp16)
            d["gemv_GBps"] = round((N_OUT * K_IN + N_OUT * 4 + K_IN * 2 + N_OUT * 2)
                                   / (g * 1e-3) / 1e9, 1)
        else:
            # quantize_act_per_token_h: read x (fp16), write codes (fp16) and scales
            d["quant_GBps"] = round((m * K_IN * 4 + m * 4) / (q * 1e-3) / 1e9, 1)
        detail[str(m)] = d

    mdom = max(m for m in MS)
    dom_ms = per_m[mdom]["gemm_ms"]
    achieved = 2.0 * mdom * N_OUT * K_IN / (dom_ms * 1e-3) / 1e12
    peak = _peak(peaks, "bf16_tflops") if peak_src == "measured" else FALLBACK_PEAKS["bf16_tflops"]
    if peak is None:
        peak, peak_src = FALLBACK_PEAKS["bf16_tflops"], "fallback"
    roofline = {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak,
                "unit": "TFLOP/s", "frac": round(achieved / peak, 4), "traffic": gemm_traffic(),
                "kernel": f"w8a8 GEMM, M={mdom}, N={N_OUT}, K={K_IN}",
                "peak_source": f"{peak_src} dense bf16/fp16 tensor peak (burst)"}

    line = {"metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": ws,
            "steps": args.steps, "warmup": max(3, args.warmup),
            "ms_per_step": round(step_ms, 5), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": round(value / PAGES_TOPS, 3), "dtype": "int8",
            "data": "synthetic", "config": config_dict(), "roofline": roofline,
            "e2e": {"value": round(e2e_value, 3), "unit": UNIT,
                    "h2d_bytes_per_step": sum(m * K_IN * 2 for m in MS),
                    "d2h_bytes_per_step": sum(m * N_OUT * 2 for m in MS),
                    "method": (f"C ABI linear() per M from pinned host buffers, L2 flushed "
                               f"before each M; M >= {2 * chunk_rows} in chunks of "
                               f"{chunk_rows} rows with copy-in, layer and copy-out "
                               f"overlapped on three streams; "
                               + ("the calls and copies of each M captured once into a "
                                  "CUDA graph and replayed every step"
                                  if e2e_graph_error is None and not args.e2e_eager_only
                                  else "enqueued by the host every step")),
                    "eager_value": round(e2e_eager, 3),
                    "graph_capture_error": e2e_graph_error,
                    "outputs_equal_single_stream_linear": e2e_mismatch == 0,
                    "mismatched_outputs": e2e_mismatch},
            "gpu_launches": args.steps * (2 * len(MS) - 1),  # M=1 is one fused launch
            "clocks": clocks.summary(), "decode": decode, "detail": detail,
            "wall_s_timed_region": round(wall, 4)}
    if rank == 0 and not args.no_workloads:
        hbm = _peak(peaks, "hbm_gbs") if peak_src == "measured" else None
        line["workloads"] = measure_workloads(
            w8, torch, device, flush_l2, l2, peak,
            hbm if hbm is not None else FALLBACK_PEAKS["hbm_gbs"])
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(inputs)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_single(args):
    """One kernel of the path on one workload shape, called `--steps` times
    after `--warmup` calls, for profilers (ncu captures); prints the mean
    CUDA-event time per call (with no L2 flush between calls)."""
    import torch

    import w4a8_int8_quantized_gb300 as w8
    torch.cuda.set_device(0)
    w8.load()
    m, n, k, gs = args.m, args.n, args.k, args.gs
    x = torch.from_numpy(synth.activations(m, k, seed=0, **WORKLOAD["act"])).cuda()
    W = torch.from_numpy(synth.weights(n, k, seed=0)).cuda()
    if args.only == "w4a8":
        wq, sw = w8.pack_weight_int4(W)
    else:
        wq, sw = w8.quantize_weight_int8(W, gs)
    xq, sa = w8.quantize_act_per_token(x, gs)
    xqh, sah = w8.quantize_act_per_token_h(x, gs)
    y = torch.empty((m, n), dtype=torch.float16, device="cuda")

    def call():
        if args.only == "quant":
            w8.quantize_act_per_token_h(x, gs, xqh, sah)
        elif args.only == "quant_i8":
            w8.quantize_act_per_token(x, gs, xq, sa)
        elif args.only == "gemm":
            w8.w8a8_gemm_h(xqh, sah, wq, sw, gs, 8, y)
        elif args.only == "gemm_i8":
            w8.w8a8_gemm(xq, sa, wq, sw, gs, y)
        elif args.only == "w4a8":
            w8.w8a8_gemm_h(xqh, sah, wq, sw, 0, 4, y)
        else:
            w8.linear(x, wq, sw, gs, 4 if args.only == "linear4" else 8, y=y)

    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        call()
    e1.record()
    torch.cuda.synchronize()
    print(json.dumps({"only": args.only, "M": m, "N": n, "K": k, "gs": gs,
                      "ms_per_call": e0.elapsed_time(e1) / max(1, args.steps)}))


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true",
                    help="skip the timed CPU-oracle sample (about 15 s)")
    ap.add_argument("--no-decode", action="store_true",
                    help="skip the back-to-back decode measurement")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the timing of the other workloads (per group, W4A8, decoder block)")
    ap.add_argument("--only", choices=["quant", "quant_i8", "gemm", "gemm_i8", "w4a8", "linear",
                                       "linear4"],
                    help="run one kernel of the path on one shape (for profilers)")
    ap.add_argument("--e2e-chunk-rows", type=int, default=E2E_CHUNK_ROWS,
                    help="rows per pipelined chunk of the end-to-end measurement")
    ap.add_argument("--e2e-eager-only", action="store_true",
                    help="time the end-to-end path as enqueued by the host only (no CUDA graphs)")
    ap.add_argument("--m", type=int, default=8192)
    ap.add_argument("--n", type=int, default=N_OUT)
    ap.add_argument("--k", type=int, default=K_IN)
    ap.add_argument("--gs", type=int, default=0)
    args = ap.parse_args()
    if args.only:
        run_single(args)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
