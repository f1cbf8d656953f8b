#!/usr/bin/env python
"""Benchmark of the NVFP4 linear layer on B300.

One step = one pass of the hot path over one batch of the largest workload,
the square 16384 x 16384 x 16384 NVFP4 linear (X ~ N(0,1) with 0.1 %
outlier channels x50, W ~ N(0, 0.02) quantized offline): per-tensor amax of
X -> global scale, dynamic NVFP4 quantization of X, tcgen05 block-scaled
FP4 GEMM against the NVFP4 weights, bfloat16 out.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]
    python bench.py --config tiny|prefill|decode|dit|square [--mode fused] [--steps K]
    python bench.py --op gemm|quantize|linear|... --shape M,N,K

Prints one JSON line (rank 0). ``value`` is the whole-job TFLOP/s
(2 M N K per step, summed over ranks, divided by the max-over-ranks time).
The step's operands are ten times the size of L2. ``roofline`` times the
GEMM kernel alone; ``rows`` hold the other workloads (standalone quantize,
prefill, DiT, decode, the extension rows). The ``reference`` arm times the
CPU oracle (test infrastructure) on a bounded row sample of the same
workload. ``--config`` times nvfp4_linear on every shape of one named
workload (one JSON line per shape); ``--op`` times one kernel on one shape.
"""
from __future__ import annotations

import argparse
import csv
import io
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "NVFP4 linear TFLOPS & % dense-FP4 peak; quantize GB/s & % HBM peak (1 B300)"
L2_BYTES = 126 * 1024 * 1024
# dense FP4 peak = measured bf16 peak x the nominal fp4:bf16 ratio (13.5 / 2.25)
FP4_OVER_BF16 = 13.5 / 2.25


# sources of the GEMM kernel the benchmark step runs (CTA-pair kernel)
GEMM_SOURCES = ("gemm_pair.cu", "ptx.cuh", "tensor_map.cu")


def gemm_traffic_per_launch():
    """DRAM bytes per GEMM launch of the benchmark step from the committed
    ncu capture, valid only while the kernel source is the one captured."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "gemm_square_traffic.json")) as f:
            rec = json.load(f)
        h = hashlib.sha256()
        for name in GEMM_SOURCES:
            with open(os.path.join(ROOT, "nvfp4_block_scaled_28_b300", "csrc", name), "rb") as f:
                h.update(f.read())
        if h.hexdigest() == rec["source_sha256"]:
            return float(rec["traffic_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        pass
    return None


# Dense FP4 rate measured by the library's tcgen05 probe (bench.py --op mma_peak)
FP4_PROBE_PEAK_TFLOPS = 9230.0
# NVIDIA's nominal dense NVFP4 rate of one B300 (context only)
FP4_NOMINAL_DENSE_TFLOPS = 13500.0


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d["bf16_tflops_sustained"]),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0,
                "source": "fallback"}


# ------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.tmp = None

    def start(self):
        self.tmp = tempfile.TemporaryFile(mode="w+")
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.tmp, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.15)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.tmp.seek(0)
        rows = [r for r in csv.reader(io.StringIO(self.tmp.read())) if len(r) >= 8]
        sm, mx, pw, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[0]))
                mx.append(float(r[1]))
                pw.append(float(r[2]))
            except ValueError:
                continue
            for name, val in zip(names, r[4:8]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# -------------------------------------------------------------- distributed

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value: float, device: str = "cuda") -> float:
    """The largest of the ranks' values (the slowest rank's time sets the
    job's time); the value itself on a single process."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(flops_per_step: float, steps: int, world: int, elapsed_ms: float) -> float:
    """Whole-job TFLOP/s: every rank runs `steps` steps of `flops_per_step`
    (weak scaling, independent replicas) within the max-over-ranks time."""
    return world * flops_per_step * steps / (elapsed_ms * 1e-3) / 1e12


def physical_gpu_index(local_rank: int) -> int:
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        try:
            return int(vis.split(",")[local_rank])
        except (ValueError, IndexError):
            return local_rank
    return local_rank


# --------------------------------------------------------------- native arm

class Direct:
    """Pre-marshalled C-ABI calls (ctypes, no per-call Python checks) for
    the timed loop; argument checks already ran once through the binding."""

    def __init__(self, lib, stream):
        self.lib = lib
        self.stream = stream
        self._ws = {}

    def global_scale(self, X, g):
        return self.lib.nvfp4_global_scale(X.data_ptr(), X.shape[0], X.shape[1], X.stride(0),
                                           g.data_ptr(), self.stream)

    def quantize(self, X, g, q, sf, layout):
        return self.lib.nvfp4_quantize(X.data_ptr(), X.shape[0], X.shape[1], X.stride(0),
                                       g.data_ptr(), q.data_ptr(), sf.data_ptr(), layout,
                                       self.stream)

    def gemm(self, Aq, As, ga, Bq, Bs, gb, M, N, K, Y):
        # scratch of nvfp4_gemm_workspace_bytes, allocated once per shape
        need = int(self.lib.nvfp4_gemm_workspace_bytes(M, N, K))
        ws = None
        if need:
            import torch
            key = (M, N, K)
            if key not in self._ws:
                self._ws[key] = torch.empty(need, dtype=torch.uint8, device="cuda")
            ws = self._ws[key]
        return self.lib.nvfp4_gemm(Aq.data_ptr(), As.data_ptr(), ga.data_ptr(), Bq.data_ptr(),
                                   Bs.data_ptr(), gb.data_ptr(), M, N, K, Y.data_ptr(),
                                   Y.stride(0), None if ws is None else ws.data_ptr(), need,
                                   self.stream)

    def linear(self, X, Wq, Ws, gw, Y, gx, mode, ws):
        M, K = X.shape
        return self.lib.nvfp4_linear(X.data_ptr(), M, K, X.stride(0), Wq.data_ptr(),
                                     Ws.data_ptr(), gw.data_ptr(), Wq.shape[0], Y.data_ptr(),
                                     Y.stride(0), None if gx is None else gx.data_ptr(), mode,
                                     ws.data_ptr(), ws.numel(), self.stream)


    def linear_grouped(self, X, Wq, Ws, gw, group_n_arr, groups, Y, mode, ws):
        M, K = X.shape
        return self.lib.nvfp4_linear_grouped(
            X.data_ptr(), M, K, X.stride(0), Wq.data_ptr(), Ws.data_ptr(), gw.data_ptr(),
            group_n_arr, groups, Y.data_ptr(), Y.stride(0), None, mode, ws.data_ptr(),
            ws.numel(), self.stream)

    def linear_lora(self, X, Wq, Ws, gw, la, lb, r, scale, Y, ws):
        M, K = X.shape
        return self.lib.nvfp4_linear_lora(
            X.data_ptr(), M, K, X.stride(0), Wq.data_ptr(), Ws.data_ptr(), gw.data_ptr(),
            Wq.shape[0], la.data_ptr(), lb.data_ptr(), r, scale, Y.data_ptr(), Y.stride(0), None,
            ws.data_ptr(), ws.numel(), self.stream)

    def linear_bias_requant_dynamic(self, X, Wq, Ws, gw, bias, Y, gy, Yq, Ys, ws):
        M, K = X.shape
        n = Wq.shape[0]
        return self.lib.nvfp4_linear_bias_requant_dynamic(
            X.data_ptr(), M, K, X.stride(0), Wq.data_ptr(), Ws.data_ptr(), gw.data_ptr(), n,
            None if bias is None else bias.data_ptr(), Y.data_ptr(), Y.stride(0), gy.data_ptr(),
            Yq.data_ptr(), Ys.data_ptr(), None, ws.data_ptr(), ws.numel(), self.stream)

    def linear_bias_requant(self, X, Wq, Ws, gw, bias, Y, gy, Yq, Ys, ws):
        M, K = X.shape
        n = Wq.shape[0]
        return self.lib.nvfp4_linear_bias_requant(
            X.data_ptr(), M, K, X.stride(0), Wq.data_ptr(), Ws.data_ptr(), gw.data_ptr(), n,
            None if bias is None else bias.data_ptr(), None if Y is None else Y.data_ptr(),
            n if Y is None else Y.stride(0), None if gy is None else gy.data_ptr(),
            None if Yq is None else Yq.data_ptr(), None if Ys is None else Ys.data_ptr(), None,
            ws.data_ptr(), ws.numel(), self.stream)


def lib_lora_ws(nv, M, N, K, r):
    return nv.load_library().nvfp4_linear_lora_workspace_bytes(M, N, K, r)


def _ok(status, what):
    if status != 0:
        raise RuntimeError("%s failed with status %d" % (what, status))


def time_region(torch, fn, iters):
    """Average milliseconds of fn() over iters calls, CUDA events on the
    current stream."""
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    s.record()
    for i in range(iters):
        fn(i)
    e.record()
    torch.cuda.synchronize()
    return s.elapsed_time(e) / iters


def run_native(args):
    import torch
    import torch.distributed as dist

    import nvfp4_block_scaled_28_b300 as nv
    from nvfp4_block_scaled_28_b300 import workloads

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    lib = nv.load_library()
    stream = torch.cuda.current_stream()
    D = Direct(lib, stream.cuda_stream)
    peaks = measured_peaks()

    # The step: nvfp4_linear on the largest workload, 16384 x 16384 x 16384
    # with the activation's global scale computed from X (amax, quantize,
    # GEMM). Its operands (537 MB of X, 151 MB of weights, 537 MB of Y) are
    # ten times L2, so consecutive steps cannot find them there.
    wl = workloads.WORKLOADS["square"]
    M, K, Nn = wl.M[0], wl.K, wl.N[0]
    flops = 2.0 * M * Nn * K
    mode = nv.LINEAR_FUSED if args.mode == "fused" else nv.LINEAR_UNFUSED
    X = workloads.make_x(wl.x_kind, M, K, workloads.x_seed(wl) + 17 * rank, device="cuda")
    W = workloads.make_w(Nn, K, workloads.w_seed(wl), device="cuda")
    Wq, Ws, gw = nv.nvfp4_quantize_weight(W, nv.SF_MMA_128x4)
    del W
    Y = torch.empty((M, Nn), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(nv.linear_workspace_bytes(M, Nn, K, mode), dtype=torch.uint8, device="cuda")
    step_bytes = M * K * 2 + Nn * K // 2 + Nn * K // 16 + M * Nn * 2
    torch.cuda.empty_cache()
    # one checked call through the binding before the raw loop
    nv.nvfp4_linear(X, Wq, Ws, gw, Y=Y, mode=mode, workspace=ws)
    torch.cuda.synchronize()

    def step(i):
        _ok(D.linear(X, Wq, Ws, gw, Y, None, mode, ws), "linear")

    # per step: counter_reset_kernel (zeroes the quantizer's barrier counter),
    # quantize_fused_kernel (amax partials, grid barrier, g_x, quantization)
    # and gemm_pair_kernel, each a programmatic dependent of the one before
    kernels_per_step = 3
    ops_per_step = 3
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    sampler = ClockSampler(physical_gpu_index(local))
    sampler.start()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record()
    for i in range(args.steps):
        step(i)
    t1.record()
    torch.cuda.synchronize()
    clocks = sampler.stop()
    if world > 1:
        dist.barrier()
    elapsed_ms = t0.elapsed_time(t1)
    assert nv.nvfp4_device_error() == 0, "a kernel recorded a bounded-wait timeout"
    elapsed_ms = max_over_ranks(elapsed_ms)
    ms_per_step = elapsed_ms / args.steps
    value = job_rate(flops, args.steps, world, elapsed_ms)

    # ---- the dominant kernel (the GEMM) alone: GEMM-only launches on the
    # step's operands (X quantized as in the step) for at least a second,
    # CUDA events on the launching stream, clocks sampled meanwhile
    gx = nv.nvfp4_global_scale(X)
    Xq = ws[8448:8448 + M * K // 2].view(M, K // 2)
    sf_off = 8448 + (M * K // 2 + 255) // 256 * 256
    Xs = ws[sf_off:sf_off + nv.sf_bytes(M, K, nv.SF_MMA_128x4)]
    nv.nvfp4_quantize(X, gx, nv.SF_MMA_128x4, q=Xq, sf=Xs.view(nv.sf_shape(M, K, nv.SF_MMA_128x4)))
    gemm_fn = lambda i: _ok(D.gemm(Xq, Xs, gx, Wq, Ws, gw, M, Nn, K, Y), "gemm")
    probe_ms = time_region(torch, gemm_fn, 3)
    gemm_iters = max(20, int(math.ceil(args.gemm_seconds * 1e3 / max(probe_ms, 1e-3))))
    gsampler = ClockSampler(physical_gpu_index(local))
    gsampler.start()
    gemm_ms = time_region(torch, gemm_fn, gemm_iters)
    gclocks = gsampler.stop()
    quant_ms = ms_per_step - gemm_ms  # the rest of the step: counter reset + dynamic quantizer

    # ---- end to end through the C ABI with host buffers: every step copies
    # its X in from pinned host memory and its whole Y back out, inside the
    # timed region. The copies run on their own streams, double-buffered, so
    # step i's copy-in, step i-1's compute and step i-2's copy-out overlap
    # (the serving pattern); events order each buffer's reuse.
    Xh = X.cpu().pin_memory()
    Yh = [torch.empty((M, Nn), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    Xd = [X, torch.empty_like(X)]
    Yd = [Y, torch.empty_like(Y)]
    s_cmp = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_cmp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    e2e_iters = max(4, min(args.steps, args.e2e_steps))

    def e2e_step(i):
        b = i % 2
        with torch.cuda.stream(s_in):
            s_in.wait_event(ev_cmp[b])        # step i-2's compute has read Xd[b]
            Xd[b].copy_(Xh, non_blocking=True)
            ev_in[b].record(s_in)
        s_cmp.wait_event(ev_in[b])
        s_cmp.wait_event(ev_out[b])           # step i-2's Y has left Yd[b]
        _ok(D.linear(Xd[b], Wq, Ws, gw, Yd[b], None, mode, ws), "linear")
        ev_cmp[b].record(s_cmp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_cmp[b])
            Yh[b].copy_(Yd[b], non_blocking=True)
            ev_out[b].record(s_out)

    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize()
    t_a, t_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_a.record(s_cmp)
    s_in.wait_stream(s_cmp)
    s_out.wait_stream(s_cmp)
    for i in range(e2e_iters):
        e2e_step(i)
    s_cmp.wait_stream(s_in)
    s_cmp.wait_stream(s_out)
    t_b.record(s_cmp)
    torch.cuda.synchronize()
    e2e_ms = t_a.elapsed_time(t_b) / e2e_iters
    e2e_ms = max_over_ranks(e2e_ms)
    e2e = {"value": world * flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
           "h2d_bytes_per_step": int(Xh.numel() * 2), "d2h_bytes_per_step": int(Yh[0].numel() * 2),
           "ms_per_step": e2e_ms, "steps": e2e_iters,
           "pipeline": "copy-in, compute and copy-out on separate streams, double-buffered"}
    del Xh, Yh, Xd, Yd
    torch.cuda.empty_cache()

    # ---- roofline of the dominant kernel (the GEMM, timed alone: the burst
    # peak is its denominator)
    peak_burst = peaks["bf16_tflops"] * FP4_OVER_BF16
    peak_sust = peaks["bf16_tflops_sustained"] * FP4_OVER_BF16
    achieved = flops / (gemm_ms * 1e-3) / 1e12
    mhz = gclocks.get("sm_mhz")
    roofline = {"bound": "tensor",
                "kernel": "gemm_pair_kernel (tcgen05 cta_group::2 kind::mxf4nvf4)",
                "achieved": achieved, "peak": peak_burst, "unit": "TFLOP/s",
                "frac": achieved / peak_burst,
                "peak_note": "%s bf16 burst %s TFLOP/s x %.0f (fp4:bf16 nominal 13.5:2.25): the "
                             "GEMM is timed alone" % (peaks["source"], peaks["bf16_tflops"],
                                                      FP4_OVER_BF16),
                "frac_of_sustained_peak": achieved / peak_sust,
                "frac_of_probe_peak": achieved / FP4_PROBE_PEAK_TFLOPS,
                "probe_peak_note": "kind::mxf4nvf4 K=64 MMAs back to back at 2032 MHz "
                                   "(python bench.py --op mma_peak --variant 7)",
                "frac_of_nominal_fp4": achieved / FP4_NOMINAL_DENSE_TFLOPS,
                "gemm_ms": gemm_ms, "gemm_launches_timed": gemm_iters,
                "gemm_clocks": gclocks,
                "gemm_ms_x_sm_ghz": gemm_ms * mhz / 1e3 if mhz else None,
                "timing": "CUDA events over %d back-to-back GEMM-only launches (%.1f s) on the "
                          "step's operands, after the timed steps" % (gemm_iters,
                                                                     gemm_iters * gemm_ms / 1e3),
                "rest_of_step_ms": quant_ms,
                "traffic": gemm_traffic_per_launch(),
                "traffic_unit": "bytes per launch (ncu dram read + write)"}

    del X, Y, Wq, Ws, ws
    torch.cuda.empty_cache()
    rows = {}
    if not args.no_extras and rank == 0:
        rows = extra_rows(torch, nv, D, workloads, peaks)

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "nvfp4",
        "data": "synthetic (seeded; X ~ N(0,1) with 0.1% outlier channels x50, W ~ N(0,0.02))",
        "config": {"workload": "square NVFP4 linear M=N=K=16384 (dynamic activation global "
                               "scale: amax, quantize, GEMM)",
                   "M": M, "N": Nn, "K": K, "mode": args.mode,
                   "l2": "inputs larger than L2: %.0f MB of operands and output per step vs "
                         "126 MB of L2" % (step_bytes / 1e6),
                   "parallelism": "replicas" if world > 1 else "single"},
        "roofline": roofline,
        "e2e": e2e,
        "gpu_launches": ops_per_step * args.steps,
        "gpu_ops_per_step": {"kernels": kernels_per_step, "memsets": ops_per_step -
                             kernels_per_step,
                             "note": "counter_reset_kernel, quantize_fused_kernel, "
                                     "gemm_pair_kernel"},
        "clocks": clocks,
        "rows": rows,
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(rows_sample=args.cpu_rows)
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def extra_rows(torch, nv, D, workloads, peaks):
    """Per-row numbers on the other workloads (context, not the headline)."""
    out = {}
    hbm = peaks["hbm_gbs"]
    # a2: standalone activation quantize, 16384 x 16384 (given global scale)
    sq = workloads.WORKLOADS["square"]
    X = workloads.make_x(sq.x_kind, sq.M[0], sq.K, workloads.x_seed(sq), device="cuda")
    g = nv.nvfp4_global_scale(X)
    q = torch.empty((sq.M[0], sq.K // 2), dtype=torch.uint8, device="cuda")
    sf = torch.empty((sq.M[0], sq.K // 16), dtype=torch.uint8, device="cuda")
    ms = time_region(torch, lambda i: _ok(D.quantize(X, g, q, sf, nv.SF_ROW_MAJOR), "q"), 20)
    nbytes = sq.M[0] * sq.K * 2.5625
    out["quantize_16384x16384"] = {"ms": ms, "GB/s": nbytes / ms / 1e6,
                                   "frac_of_hbm": nbytes / ms / 1e6 / hbm}
    ms = time_region(torch, lambda i: _ok(D.global_scale(X, g), "amax"), 20)
    out["global_scale_16384x16384"] = {"ms": ms, "GB/s": sq.M[0] * sq.K * 2 / ms / 1e6}
    # F2: offline weight quantization of the 5120 x 5120 prefill weight under
    # each block-scale rule (global scale included)
    pf = workloads.WORKLOADS["prefill"]
    Wp = workloads.make_w(pf.N[0], pf.K, workloads.w_seed(pf), device="cuda")
    for rule, name in ((0, "absmax"), (1, "four_over_six"), (2, "mse")):
        nv.nvfp4_quantize_weight(Wp, nv.SF_MMA_128x4, rule=rule)
        ms = time_region(torch, lambda i: nv.nvfp4_quantize_weight(Wp, nv.SF_MMA_128x4,
                                                                   rule=rule), 5)
        out["weight_quantize_5120x5120_%s" % name] = {"ms": ms}
    del Wp
    del X, q, sf
    torch.cuda.empty_cache()
    # a4 on the LLM prefill projection: the whole linear (dynamic global
    # scale) and the GEMM alone, on 3 rotating input sets (> 2x L2 in all)
    pf = workloads.WORKLOADS["prefill"]
    M, n, K = pf.M[0], pf.N[0], pf.K
    psets = []
    for r in range(3):
        Xp = workloads.make_x(pf.x_kind, M, K, workloads.x_seed(pf) + 1000 * r, device="cuda")
        W = workloads.make_w(n, K, workloads.w_seed(pf) + 1000 * r, device="cuda")
        Wq, Ws, gw = nv.nvfp4_quantize_weight(W, nv.SF_MMA_128x4)
        del W
        gxp = nv.nvfp4_global_scale(Xp)
        Xq, Xs = nv.nvfp4_quantize(Xp, gxp, nv.SF_MMA_128x4)
        psets.append(dict(X=Xp, Wq=Wq, Ws=Ws, gw=gw, gx=gxp, Xq=Xq, Xs=Xs,
                          Y=torch.empty((M, n), dtype=torch.bfloat16, device="cuda"),
                          ws=torch.empty(nv.linear_workspace_bytes(M, n, K), dtype=torch.uint8,
                                         device="cuda")))
    fl = 2.0 * M * n * K
    lin = lambda i: _ok(D.linear(psets[i % 3]["X"], psets[i % 3]["Wq"], psets[i % 3]["Ws"],
                                 psets[i % 3]["gw"], psets[i % 3]["Y"], None, 0,
                                 psets[i % 3]["ws"]), "lin")
    gem = lambda i: _ok(D.gemm(psets[i % 3]["Xq"], psets[i % 3]["Xs"], psets[i % 3]["gx"],
                               psets[i % 3]["Wq"], psets[i % 3]["Ws"], psets[i % 3]["gw"], M, n,
                               K, psets[i % 3]["Y"]), "gemm")
    lin(0)
    ms_l = time_region(torch, lin, 200)
    ms_g = time_region(torch, gem, 200)
    out["prefill_linear_4096x5120x5120"] = {
        "ms": ms_l, "TFLOP/s": fl / ms_l / 1e9, "gemm_ms": ms_g, "gemm_TFLOP/s": fl / ms_g / 1e9,
        "gemm_frac_of_burst_peak": fl / ms_g / 1e9 / (peaks["bf16_tflops"] * FP4_OVER_BF16),
        "inputs": "3 rotating sets"}
    del psets
    torch.cuda.empty_cache()
    # DiT block linears
    dit = workloads.WORKLOADS["dit"]
    Xd = workloads.make_x(dit.x_kind, dit.M[0], dit.K, workloads.x_seed(dit), device="cuda")
    for n in dit.N:
        W = workloads.make_w(n, dit.K, workloads.w_seed(dit) + n, device="cuda")
        Wq, Ws, gw = nv.nvfp4_quantize_weight(W, nv.SF_MMA_128x4)
        Y = torch.empty((dit.M[0], n), dtype=torch.bfloat16, device="cuda")
        ws = torch.empty(nv.linear_workspace_bytes(dit.M[0], n, dit.K), dtype=torch.uint8,
                         device="cuda")
        ms = time_region(torch, lambda i: _ok(D.linear(Xd, Wq, Ws, gw, Y, None, 0, ws), "lin"), 20)
        out["dit_linear_4096x3072x%d" % n] = {"ms": ms,
                                               "TFLOP/s": 2.0 * dit.M[0] * n * dit.K / ms / 1e9}
    # F4: the attention's q, k, v projections (3 x 3072) as one grouped call
    # (X quantized once, one GEMM launch) against three separate linears
    import ctypes
    qkv = [nv.nvfp4_quantize_weight(workloads.make_w(3072, dit.K, workloads.w_seed(dit) + 7 + i,
                                                     device="cuda"), nv.SF_MMA_128x4)
           for i in range(3)]
    Wq3, Ws3, g3, gn3 = nv.pack_weight_groups(qkv)
    gn_arr = (ctypes.c_int64 * 3)(*gn3)
    gn_ptr = ctypes.cast(gn_arr, ctypes.c_void_p)
    Y3 = torch.empty((dit.M[0], sum(gn3)), dtype=torch.bfloat16, device="cuda")
    ws3 = torch.empty(nv.linear_workspace_bytes(dit.M[0], sum(gn3), dit.K), dtype=torch.uint8,
                      device="cuda")
    Ysep = [torch.empty((dit.M[0], 3072), dtype=torch.bfloat16, device="cuda") for _ in range(3)]
    _ok(D.linear_grouped(Xd, Wq3, Ws3, g3, gn_ptr, 3, Y3, 0, ws3), "grouped")  # set-up
    ms_g = time_region(torch, lambda i: _ok(D.linear_grouped(Xd, Wq3, Ws3, g3, gn_ptr, 3, Y3, 0,
                                                             ws3), "grouped"), 20)

    def sep(i):
        for (wq_, ws_, gw_), y_ in zip(qkv, Ysep):
            _ok(D.linear(Xd, wq_, ws_, gw_, y_, None, 0, ws3), "lin")

    ms_s = time_region(torch, sep, 20)
    fl3 = 2.0 * dit.M[0] * sum(gn3) * dit.K
    out["dit_qkv_grouped_4096x3072x(3x3072)"] = {
        "grouped_ms": ms_g, "separate_ms": ms_s, "TFLOP/s_grouped": fl3 / ms_g / 1e9,
        "TFLOP/s_separate": fl3 / ms_s / 1e9}
    del Xd, qkv, Wq3, Ws3, Y3, ws3, Ysep
    # F1: prefill layer with the bias add and the output's NVFP4
    # re-quantization in the GEMM epilogue, against the same layer followed
    # by a separate quantize pass over Y
    pf = workloads.WORKLOADS["prefill"]
    M, n, K = pf.M[0], pf.N[0], pf.K
    Xp = workloads.make_x(pf.x_kind, M, K, workloads.x_seed(pf), device="cuda")
    W = workloads.make_w(n, K, workloads.w_seed(pf), device="cuda")
    Wq, Ws, gw = nv.nvfp4_quantize_weight(W, nv.SF_MMA_128x4)
    del W
    bias = workloads.make_bias(n, seed=77, device="cuda")
    Y = torch.empty((M, n), dtype=torch.bfloat16, device="cuda")
    Yq = torch.empty((M, n // 2), dtype=torch.uint8, device="cuda")
    Ys = torch.empty(nv.sf_shape(M, n, nv.SF_MMA_128x4), dtype=torch.uint8, device="cuda")
    ws = torch.empty(nv.linear_workspace_bytes(M, n, K), dtype=torch.uint8, device="cuda")
    _ok(D.linear(Xp, Wq, Ws, gw, Y, None, 0, ws), "lin")
    gy = nv.nvfp4_global_scale(Y)
    fl = 2.0 * M * n * K
    ms_lin = time_region(torch, lambda i: _ok(D.linear(Xp, Wq, Ws, gw, Y, None, 0, ws), "lin"), 20)
    gxp = nv.nvfp4_global_scale(Xp)
    ms_lin_gx = time_region(torch, lambda i: _ok(D.linear(Xp, Wq, Ws, gw, Y, gxp, 0, ws), "lin"),
                            20)
    out["prefill_linear_4096x5120x5120_given_gx"] = {
        "ms": ms_lin_gx, "TFLOP/s": fl / ms_lin_gx / 1e9,
        "note": "given activation global scale (quantize_kernel + GEMM); the headline step "
                "computes it from X"}
    ms_seq = time_region(torch, lambda i: (_ok(D.linear(Xp, Wq, Ws, gw, Y, None, 0, ws), "lin"),
                                           _ok(D.quantize(Y, gy, Yq, Ys, nv.SF_MMA_128x4), "q")),
                         20)
    _ok(D.linear_bias_requant(Xp, Wq, Ws, gw, bias, Y, gy, Yq, Ys, ws), "epi")  # set-up
    ms_epi = time_region(torch, lambda i: _ok(D.linear_bias_requant(Xp, Wq, Ws, gw, bias, Y, gy,
                                                                    Yq, Ys, ws), "epi"), 20)
    ms_q = time_region(torch, lambda i: _ok(D.linear_bias_requant(Xp, Wq, Ws, gw, bias, None, gy,
                                                                  Yq, Ys, ws), "epi"), 20)
    # the output's global scale computed from the output: epilogue amax +
    # quantize of Y, against the unfused dynamic sequence (bias linear, the
    # global scale of Y, quantize)
    gyd = torch.empty(1, dtype=torch.float32, device="cuda")
    _ok(D.linear_bias_requant_dynamic(Xp, Wq, Ws, gw, bias, Y, gyd, Yq, Ys, ws), "dyn")
    ms_dyn = time_region(torch, lambda i: _ok(D.linear_bias_requant_dynamic(
        Xp, Wq, Ws, gw, bias, Y, gyd, Yq, Ys, ws), "dyn"), 20)

    def dyn_seq(i):
        _ok(D.linear_bias_requant(Xp, Wq, Ws, gw, bias, Y, None, None, None, ws), "bias")
        _ok(D.global_scale(Y, gyd), "g")
        _ok(D.quantize(Y, gyd, Yq, Ys, nv.SF_MMA_128x4), "q")

    dyn_seq(0)
    ms_dyn_seq = time_region(torch, dyn_seq, 20)
    out["prefill_linear_4096x5120x5120_epilogue"] = {
        "linear_ms": ms_lin,
        "linear_then_quantize_ms": ms_seq,
        "bias_requant_fused_ms": ms_epi,
        "bias_requant_fused_no_bf16_y_ms": ms_q,
        "TFLOP/s_fused": fl / ms_epi / 1e9,
        "TFLOP/s_fused_no_bf16_y": fl / ms_q / 1e9,
        "bias_requant_dynamic_g_y_ms": ms_dyn,
        "bias_then_global_scale_then_quantize_ms": ms_dyn_seq,
    }
    # F3: the same layer with a rank-32 LoRA correction (down projection in
    # the quantization pass, up projection as bfloat16 steps in the GEMM)
    la, lb = workloads.make_lora(32, K, n, seed=5, device="cuda")
    wsl = torch.empty(int(lib_lora_ws(nv, M, n, K, 32)), dtype=torch.uint8, device="cuda")
    lora_fn = lambda i: _ok(D.linear_lora(Xp, Wq, Ws, gw, la, lb, 32, 1.0, Y, wsl), "lora")
    lora_fn(0)  # first call: one-time kernel set-up outside the timed region
    ms_lora = time_region(torch, lora_fn, 20)
    out["prefill_linear_4096x5120x5120_lora_r32"] = {
        "linear_ms": ms_lin, "lora_ms": ms_lora, "TFLOP/s_lora": fl / ms_lora / 1e9}
    del Xp, Wq, Ws, Y, Yq, Ys, ws, wsl, la, lb
    torch.cuda.empty_cache()
    # a5: decode (weight-bandwidth bound), rotating 3 weight copies (> L2)
    dec = workloads.WORKLOADS["decode"]
    n = dec.N[0]
    wsets = []
    for r in range(3):
        W = workloads.make_w(n, dec.K, workloads.w_seed(dec) + r, device="cuda")
        wsets.append(nv.nvfp4_quantize_weight(W, nv.SF_MMA_128x4))
        del W
    wbytes = n * dec.K // 2 + n * dec.K // 16
    for m in dec.M:
        Xm = workloads.make_x(dec.x_kind, m, dec.K, workloads.x_seed(dec) + m, device="cuda")
        Y = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
        ws = torch.empty(nv.linear_workspace_bytes(m, n, dec.K), dtype=torch.uint8, device="cuda")
        for mode_name, mode_id in (("unfused", 0), ("fused", 1)):
            def f(i, Xm=Xm, Y=Y, ws=ws, mode_id=mode_id):
                Wq, Ws, gw = wsets[i % 3]
                _ok(D.linear(Xm, Wq, Ws, gw, Y, None, mode_id, ws), "lin")

            for i in range(20):  # steady state: the dependent-launch chain primed
                f(i)
            ms = time_region(torch, f, 200)
            row = {"ms": ms, "weight_GB/s": wbytes / ms / 1e6,
                   "frac_of_hbm": wbytes / ms / 1e6 / hbm,
                   "TFLOP/s": 2.0 * m * n * dec.K / ms / 1e9}
            if mode_id == 1:
                row["path"] = ("one kernel, X quantized in shared memory" if m <= 8 else
                               "unfused sequence (fused mode covers M <= 8)")
            out["decode_linear_M%d_%s" % (m, mode_name)] = row
    # F1 on a decode layer (M = 8): the bias and the output's re-quantization
    # in the decode kernel's epilogue (given g_y, and g_y from the output)
    # against the same layer followed by separate passes
    m = 8
    Xm = workloads.make_x(dec.x_kind, m, dec.K, workloads.x_seed(dec) + 1000 + m, device="cuda")
    bias_d = workloads.make_bias(n, seed=78, device="cuda")
    Y = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
    Yq = torch.empty((m, n // 2), dtype=torch.uint8, device="cuda")
    Ys = torch.empty(nv.sf_shape(m, n, nv.SF_MMA_128x4), dtype=torch.uint8, device="cuda")
    ws = torch.empty(nv.linear_workspace_bytes(m, n, dec.K), dtype=torch.uint8, device="cuda")
    gyd = torch.empty(1, dtype=torch.float32, device="cuda")
    W0 = wsets[0]
    _ok(D.linear_bias_requant(Xm, W0[0], W0[1], W0[2], bias_d, Y, None, None, None, ws), "b")
    gy = nv.nvfp4_global_scale(Y)

    def rot(fn):
        return lambda i: fn(wsets[i % 3])

    runs = {
        "bias_requant_fused_us": rot(lambda w: _ok(D.linear_bias_requant(
            Xm, w[0], w[1], w[2], bias_d, Y, gy, Yq, Ys, ws), "e")),
        "bias_then_quantize_us": rot(lambda w: (_ok(D.linear_bias_requant(
            Xm, w[0], w[1], w[2], bias_d, Y, None, None, None, ws), "b"),
            _ok(D.quantize(Y, gy, Yq, Ys, nv.SF_MMA_128x4), "q"))),
        "bias_requant_dynamic_g_y_us": rot(lambda w: _ok(D.linear_bias_requant_dynamic(
            Xm, w[0], w[1], w[2], bias_d, Y, gyd, Yq, Ys, ws), "d")),
        "bias_then_global_scale_then_quantize_us": rot(lambda w: (_ok(D.linear_bias_requant(
            Xm, w[0], w[1], w[2], bias_d, Y, None, None, None, ws), "b"),
            _ok(D.global_scale(Y, gyd), "g"), _ok(D.quantize(Y, gyd, Yq, Ys, nv.SF_MMA_128x4),
                                                  "q"))),
    }
    row = {}
    for name, fn in runs.items():
        for i in range(20):
            fn(i)
        row[name] = time_region(torch, fn, 200) * 1e3
    out["decode_linear_M8_epilogue"] = row
    torch.cuda.synchronize()
    return out


# ------------------------------------------------------------ CPU oracle leg

_SQ_SAMPLE_NOTE = ("%d of 16384 rows per step of the square workload (global scale and quantize "
                   "of the sampled activation rows, FP64 GEMM of those rows against all 16384 "
                   "weight rows; the weight is quantized once beforehand, untimed, as it is "
                   "offline on the GPU path)")


def _oracle_square_sample(rows_sample: int):
    """Quantize W once (offline in the real path), then time the oracle's
    step on `rows_sample` rows of X: global scale, quantize, GEMM rows."""
    import numpy as np
    import torch

    import oracle
    from nvfp4_block_scaled_28_b300 import workloads

    wl = workloads.WORKLOADS["square"]
    K, Nn = wl.K, wl.N[0]
    bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)
    wb = bits(workloads.make_w(Nn, K, workloads.w_seed(wl)))
    gw = oracle.global_scale(wb)
    wq, ws = oracle.quantize(wb, gw)
    del wb
    xb = bits(workloads.make_x(wl.x_kind, rows_sample, K, workloads.x_seed(wl)))

    def step():
        gx = oracle.global_scale(xb)
        xq, xs = oracle.quantize(xb, gx)
        return oracle.gemm(xq, xs, gx, wq, ws, gw)

    return step, 2.0 * rows_sample * Nn * K


def cpu_baseline(rows_sample: int):
    import oracle
    oracle.build()
    step, fl = _oracle_square_sample(rows_sample)
    t = time.perf_counter()
    step()
    dt = time.perf_counter() - t
    return {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": oracle.num_threads(),
            "kind": "oracle", "seconds": dt, "sample": _SQ_SAMPLE_NOTE % rows_sample}


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    oracle.build()
    # about 0.02 s of oracle work per sampled row on 16 host cores: keep the
    # whole run (steps + warm-up) within a couple of minutes
    rows = max(1, min(256, 3072 // max(1, args.steps + args.warmup)))
    step, fl = _oracle_square_sample(rows)
    for _ in range(args.warmup):
        step()
    t = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t
    value = fl * args.steps / dt / 1e12
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64 (oracle)", "data": "synthetic",
        "config": {"workload": "square NVFP4 linear M=N=K=16384 (dynamic activation global "
                               "scale: amax, quantize, GEMM)", "M": 16384, "N": 16384,
                   "K": 16384},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": _SQ_SAMPLE_NOTE % rows},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }))


def run_single_op(args):
    """One kernel on one shape, for profiling: --op gemm|quantize|linear|
    linear_bias_requant|linear_requant_only|linear_lora --shape M,N,K
    (quantize uses M,K). Prints the mean CUDA-event time."""
    import torch

    import nvfp4_block_scaled_28_b300 as nv
    from nvfp4_block_scaled_28_b300 import workloads

    lib = nv.load_library()
    D = Direct(lib, torch.cuda.current_stream().cuda_stream)
    if args.op == "mma_peak":
        ctas = torch.cuda.get_device_properties(0).multi_processor_count
        iters = args.iters
        cyc = torch.zeros(1, dtype=torch.int64, device="cuda")
        v = args.variant
        if v == 7:
            ctas &= ~1
        n_mma = 128 if v in (1, 2) else 256
        from nvfp4_block_scaled_28_b300 import _native
        probe = _native.load_probe()
        fn = lambda i: _ok(probe.nvfp4_mma_peak_probe(ctas, iters, v, cyc.data_ptr(), D.stream),
                           "peak")
        for i in range(max(1, args.warmup)):
            fn(i)
        sampler = ClockSampler(physical_gpu_index(0))
        sampler.start()
        ms = time_region(torch, fn, args.steps)
        clocks = sampler.stop()
        k_mma = 16 if v == 6 else 64
        fl = ctas * iters * 2.0 * 128 * n_mma * k_mma
        c = int(cyc.item())
        names = {0: "fp4 128x256x64", 1: "fp4 128x128x64", 2: "fp4 128x128x64, two warps",
                 3: "fp4 + 3 scale copies per MMA, same thread",
                 4: "fp4 + 3 scale copies per MMA, second warp",
                 5: "fp4 + commit/poll/fence per 4 MMAs", 6: "bf16 128x256x16",
                 7: "fp4 CTA pair 256x256x64 (per SM 128x256x64)"}
        print(json.dumps({"op": "mma_peak", "variant": v, "what": names[v], "N": n_mma,
                          "K": k_mma, "ctas": ctas, "iters": iters, "ms": ms,
                          "TFLOP/s": fl / ms / 1e9, "cycles_cta0": c,
                          "cycles_per_mma": c / (iters // 2 if v == 2 else iters),
                          "flop_per_cycle_per_sm": 2.0 * 128 * n_mma * k_mma * iters / c
                          if c else None,
                          "clocks": clocks}))
        return
    M, Nn, K = (int(v) for v in args.shape.split(","))
    _ok(lib.nvfp4_debug_select_gemm_kernel({"pair": 0, "single": 1}[args.kernel]),
        "select kernel")
    X = workloads.make_x("outlier", M, K, 1, device="cuda")
    g = nv.nvfp4_global_scale(X)
    if args.op == "quantize":
        q = torch.empty((M, K // 2), dtype=torch.uint8, device="cuda")
        sf = torch.empty((M, K // 16), dtype=torch.uint8, device="cuda")
        fn = lambda i: _ok(D.quantize(X, g, q, sf, nv.SF_ROW_MAJOR), "quantize")
        work, unit = M * K * 2.5625 / 1e9, "GB"
    else:
        W = workloads.make_w(Nn, K, 2, device="cuda")
        Wq, Ws, gw = nv.nvfp4_quantize_weight(W, nv.SF_MMA_128x4)
        del W
        Y = torch.empty((M, Nn), dtype=torch.bfloat16, device="cuda")
        if args.op == "gemm":
            Xq, Xs = nv.nvfp4_quantize(X, g, nv.SF_MMA_128x4)
            fn = lambda i: _ok(D.gemm(Xq, Xs, g, Wq, Ws, gw, M, Nn, K, Y), "gemm")
        elif args.op == "linear_lora":
            # rank-32 LoRA correction (--iters unused)
            la, lb = workloads.make_lora(32, K, Nn, seed=5, device="cuda")
            ws = torch.empty(int(lib_lora_ws(nv, M, Nn, K, 32)), dtype=torch.uint8,
                             device="cuda")
            fn = lambda i: _ok(D.linear_lora(X, Wq, Ws, gw, la, lb, 32, 1.0, Y, ws), "lora")
        elif args.op in ("linear_bias_requant", "linear_requant_only"):
            # bias add + NVFP4 re-quantization of Y in the GEMM epilogue
            # (requant_only: no bfloat16 Y is stored)
            ws = torch.empty(nv.linear_workspace_bytes(M, Nn, K), dtype=torch.uint8,
                             device="cuda")
            bias = workloads.make_bias(Nn, seed=3, device="cuda")
            _ok(D.linear(X, Wq, Ws, gw, Y, None, nv.LINEAR_UNFUSED, ws), "linear")
            gy = nv.nvfp4_global_scale(Y)
            Yq = torch.empty((M, Nn // 2), dtype=torch.uint8, device="cuda")
            Ys = torch.empty(nv.sf_shape(M, Nn, nv.SF_MMA_128x4), dtype=torch.uint8,
                             device="cuda")
            Yo = Y if args.op == "linear_bias_requant" else None
            fn = lambda i: _ok(D.linear_bias_requant(X, Wq, Ws, gw, bias, Yo, gy, Yq, Ys, ws),
                               "linear_bias_requant")
        else:
            mode = nv.LINEAR_FUSED if args.mode == "fused" else nv.LINEAR_UNFUSED
            ws = torch.empty(nv.linear_workspace_bytes(M, Nn, K, mode), dtype=torch.uint8,
                             device="cuda")
            fn = lambda i: _ok(D.linear(X, Wq, Ws, gw, Y, None, mode, ws), "linear")
        work, unit = 2.0 * M * Nn * K / 1e12, "TFLOP"
    for i in range(args.warmup):
        fn(i)
    ms = time_region(torch, fn, args.steps)
    assert nv.nvfp4_device_error() == 0
    print(json.dumps({"op": args.op, "shape": [M, Nn, K], "kernel": args.kernel, "ms": ms,
                      "rate": work / (ms * 1e-3), "unit": unit + "/s"}))


def run_config(args):
    """nvfp4_linear (dynamic activation global scale, --mode) on every shape
    of one named workload (--config tiny|prefill|decode|dit|square), its own
    activation recipe and seeds; three rotating input sets where they fit in
    a few GB. One JSON line per shape."""
    import torch

    import nvfp4_block_scaled_28_b300 as nv
    from nvfp4_block_scaled_28_b300 import workloads

    lib = nv.load_library()
    D = Direct(lib, torch.cuda.current_stream().cuda_stream)
    wl = workloads.WORKLOADS[args.config]
    mode = nv.LINEAR_FUSED if args.mode == "fused" else nv.LINEAR_UNFUSED
    peaks = measured_peaks()
    for n in wl.N:
        for m in wl.M:
            K = wl.K
            nsets = 3 if (m * K * 2 + n * K // 2) * 3 < (4 << 30) else 1
            sets = []
            for r in range(nsets):
                X = workloads.make_x(wl.x_kind, m, K, workloads.x_seed(wl) + 1000 * r + m,
                                     device="cuda")
                W = workloads.make_w(n, K, workloads.w_seed(wl) + 1000 * r + n, device="cuda")
                Wq, Ws, gw = nv.nvfp4_quantize_weight(W, nv.SF_MMA_128x4)
                del W
                sets.append((X, Wq, Ws, gw, torch.empty((m, n), dtype=torch.bfloat16,
                                                        device="cuda")))
            ws = torch.empty(nv.linear_workspace_bytes(m, n, K, mode), dtype=torch.uint8,
                             device="cuda")

            def fn(i, sets=sets, ws=ws):
                X, Wq, Ws, gw, Y = sets[i % len(sets)]
                _ok(D.linear(X, Wq, Ws, gw, Y, None, mode, ws), "linear")

            for i in range(max(args.warmup, 3)):
                fn(i)
            ms = time_region(torch, fn, args.steps)
            assert nv.nvfp4_device_error() == 0
            wbytes = n * K // 2 + n * K // 16
            print(json.dumps({"config": wl.name, "workload": wl.description, "M": m, "N": n,
                              "K": K, "mode": args.mode, "inputs": "%d rotating sets" % nsets,
                              "ms": ms, "TFLOP/s": 2.0 * m * n * K / ms / 1e9,
                              "weight_GB/s": wbytes / ms / 1e6,
                              "weight_frac_of_hbm": wbytes / ms / 1e6 / peaks["hbm_gbs"]}))
            del sets, ws
            torch.cuda.empty_cache()


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=600)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--gemm-seconds", type=float, default=1.5,
                    help="length of the GEMM-only roofline loop")
    ap.add_argument("--e2e-steps", type=int, default=16)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--mode", choices=["unfused", "fused"], default="unfused")
    ap.add_argument("--no-extras", action="store_true", help="skip the per-row extra numbers")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-rows", type=int, default=384)
    ap.add_argument("--op", choices=["gemm", "quantize", "linear", "linear_bias_requant",
                                     "linear_requant_only", "linear_lora", "mma_peak"],
                    default=None,
                    help="time a single kernel on --shape instead of the benchmark step")
    ap.add_argument("--shape", default="8192,8192,8192", help="M,N,K for --op")
    ap.add_argument("--config", choices=["tiny", "prefill", "decode", "dit", "square"],
                    default=None,
                    help="time nvfp4_linear on every shape of one named workload instead of "
                         "the benchmark step")
    ap.add_argument("--kernel", choices=["pair", "single"], default="pair",
                    help="--op: the GEMM kernel for M > 128 (CTA pairs on 256x256 tiles, or "
                         "the single-CTA kernel)")
    ap.add_argument("--iters", type=int, default=200000, help="--op mma_peak: MMAs per CTA")
    ap.add_argument("--variant", type=int, default=0,
                    help="--op mma_peak: N / accumulator-count / scale-copy variant")
    args = ap.parse_args()
    if args.warmup < 3 and args.op is None and args.config is None:
        ap.error("--warmup must be >= 3")
    if args.op is not None:
        run_single_op(args)
    elif args.config is not None:
        run_config(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_native(args)


if __name__ == "__main__":
    main()
