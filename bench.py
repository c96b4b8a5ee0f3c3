"""Benchmark of the W8A8 quantized linear layer on GB300.

One step = the run-time hot path on one batch: dynamic per-token activation
quantization (q8_quantize_act) followed by the INT8 GEMM with the fused
dequantization epilogue (q8_gemm_dequant). Weight quantization and column sums
are offline (done once, timed separately as `weight_prep_ms`).

Metric: TOPS = 2*M*N*K / step time (integer multiply-adds counted as 2 ops,
activation quantization included), on the large-prefill workload
(A [8192, 16384] x W [8192, 16384]^T, per-token x per-channel, fp32 out).
Inputs are synthetic and resident in HBM; L2 is flushed (256 MiB write)
before every timed step; each step is timed with CUDA events on the launching
stream, and the quantizer and the GEMM separately for the roofline.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (plain C, int64 accumulation) on the
host cores on a bounded row sample of the same workload. Under torchrun each
rank runs an independent replica (the path shards by tokens with no
exchange); rank 0 prints one JSON line.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

HEADLINE = "prefill16k"
DECODE = "decode"
METRIC = "W8A8 GEMM TOPS (2MNK/s incl. act quantize)"
L2_FLUSH_BYTES = 256 << 20
HBM_NOMINAL_GBS = 7900.0   # GB300 HBM3e, nominal; every HBM fraction is also given against it


def add_nominal_hbm(obj):
    """Beside every HBM fraction of the measured copy bandwidth, the same rate against the
    nominal HBM bandwidth (in place, recursively)."""
    if isinstance(obj, dict):
        if "frac_hbm" in obj and "GB/s" in obj:
            obj["frac_hbm_nominal"] = round(obj["GB/s"] / HBM_NOMINAL_GBS, 4)
        if "gemm_frac_hbm" in obj and "gemm_GB/s" in obj:
            obj["gemm_frac_hbm_nominal"] = round(obj["gemm_GB/s"] / HBM_NOMINAL_GBS, 4)
        if obj.get("bound") == "hbm" and obj.get("unit") == "GB/s" and "achieved" in obj:
            obj["frac_nominal"] = round(obj["achieved"] / HBM_NOMINAL_GBS, 4)
        for v in obj.values():
            add_nominal_hbm(v)
    elif isinstance(obj, list):
        for v in obj:
            add_nominal_hbm(v)
    return obj

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of one launch of the
# headline GEMM kernel on the headline workload, from the ncu capture of this kernel.
# It is reported only while the kernel's source files still hash to the fingerprint the
# capture was taken on.
MEASURED_TRAFFIC = {
    # the CTA-pair kernel loading the fp16 copy of the activation codes (the GEMM with a workspace)
    "tcgen05_pair_f16a": {"bytes": 1_700_581_632 + 259_416_832,
                          "sources": ("q8_gemm_tc2.cu", "q8_tc_ptx.cuh", "q8_internal.h"),
                          "sha256_16": "533255b7326eb1d8"},
}


def measured_traffic(kernel: str):
    """Captured DRAM bytes per launch of `kernel`, or None if there is no capture of
    the current source."""
    import hashlib
    rec = MEASURED_TRAFFIC.get(kernel)
    if rec is None:
        return None
    csrc = os.path.join(os.path.dirname(os.path.abspath(__file__)), "int8_quantized_gemm_gb300", "csrc")
    h = hashlib.sha256()
    try:
        for f in rec["sources"]:
            with open(os.path.join(csrc, f), "rb") as fh:
                h.update(fh.read())
    except OSError:
        return None
    return rec["bytes"] if h.hexdigest()[:16] == rec["sha256_16"] else None


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


def sustained_peak():
    """The bf16 dense rate measured as a seconds-long loop under the power cap (the denominator for a
    kernel timed inside a long run), with its source."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops_sustained"]), "measured"
    except Exception:
        return 1700.0, "fallback"


class ClockSampler:
    """Samples the SM clock and the clock-event (throttle) reasons through NVML about every
    millisecond while the timed region runs (reads only; nothing is set)."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, cuda_index: int):
        self.samples = []
        self.max_mhz = None
        self.stop = threading.Event()
        self.thread = None
        self.nvml = None
        try:
            import ctypes
            import torch
            nvml = ctypes.CDLL("libnvidia-ml.so.1")
            if nvml.nvmlInit_v2() != 0:
                return
            handle = ctypes.c_void_p()
            ok = False
            uuid = getattr(torch.cuda.get_device_properties(cuda_index), "uuid", None)
            if uuid is not None:
                ok = nvml.nvmlDeviceGetHandleByUUID(f"GPU-{uuid}".encode(), ctypes.byref(handle)) == 0
            if not ok:
                count = ctypes.c_uint()
                nvml.nvmlDeviceGetCount_v2(ctypes.byref(count))
                if count.value == 1:
                    ok = nvml.nvmlDeviceGetHandleByIndex_v2(0, ctypes.byref(handle)) == 0
            if not ok:
                return
            self.nvml, self.handle, self.ct = nvml, handle, ctypes
            mx = ctypes.c_uint()
            if nvml.nvmlDeviceGetMaxClockInfo(handle, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = mx.value
        except Exception:
            self.nvml = None

    def _run(self):
        ct, nvml, h = self.ct, self.nvml, self.handle
        clk, rs = ct.c_uint(), ct.c_ulonglong()
        get_reasons = getattr(nvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            nvml.nvmlDeviceGetCurrentClocksThrottleReasons
        while not self.stop.is_set():
            if nvml.nvmlDeviceGetClockInfo(h, 1, ct.byref(clk)) == 0 and get_reasons(h, ct.byref(rs)) == 0:
                self.samples.append((clk.value, rs.value))
            time.sleep(0.001)

    def __enter__(self):
        if self.nvml is not None:
            self.thread = threading.Thread(target=self._run, daemon=True)
            self.thread.start()
        return self

    def __exit__(self, *exc):
        self.stop.set()
        if self.thread:
            self.thread.join(timeout=2)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0, "source": "nvml"}
        reasons = set()
        for _, r in self.samples:
            for bit, name in self.REASONS.items():
                if r & bit:
                    reasons.add(name)
        return {"sm_mhz": statistics.median(c for c, _ in self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(reasons), "samples": len(self.samples), "source": "nvml"}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """The largest x over all ranks (every rank gets it): the job's time is its slowest rank's."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank: float, world: int, ms_per_step_max: float, scale: float = 1e12) -> float:
    """Whole-job throughput: the units all ranks processed in one step over the slowest rank's
    step time (weak scaling: every rank runs the same per-rank workload)."""
    return units_per_rank * world / (ms_per_step_max * 1e-3) / scale


# ------------------------------------------------------------------ our arm

_HOST_INPUTS = {}


def host_inputs(name):
    """The workload's fp32 A and W as numpy arrays (drawn once per process)."""
    if name not in _HOST_INPUTS:
        wl = workloads.WORKLOADS[name]
        _HOST_INPUTS[name] = (workloads.make_activations(wl), workloads.make_weights(wl))
    return _HOST_INPUTS[name]


def layer_inputs(name, device):
    import torch
    wl = workloads.WORKLOADS[name]
    a_h, w_h = host_inputs(name)
    return wl, torch.from_numpy(a_h).to(device), torch.from_numpy(w_h).to(device)


def step_bytes(wl):
    """Algorithmic bytes of one step: the activation quantizer (read A, write codes and scales, zero
    points when asymmetric) and the GEMM (codes of A and W, the scales, column sums and zero points
    when asymmetric, y)."""
    M, N, K = wl.M, wl.N, wl.K
    asym = not wl.act_symmetric
    na = M if wl.act_granularity == "row" else 1
    nw = N if wl.w_granularity == "row" else 1
    quant = 5 * M * K + 4 * na * (2 if asym else 1)
    gemm = M * K + N * K + 4 * nw + 4 * na * (2 if asym else 1) + (4 * N if asym else 0) + 4 * M * N
    return quant, gemm


def run_ours(args, world, rank, local):
    import torch
    import int8_quantized_gemm_gb300 as q8
    from int8_quantized_gemm_gb300 import build

    build.build()
    q8.load()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    stream = torch.cuda.current_stream()
    hbm_peak, tc_peak, peak_kind = peaks()

    wl, a, w = layer_inputs(HEADLINE, device)
    M, N, K = wl.M, wl.N, wl.K
    apr, wpr, sym = wl.act_granularity == "row", wl.w_granularity == "row", wl.act_symmetric

    # offline: weight quantization and column sums (timed once, not part of a step)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    qw, s_w = q8.q8_quantize_weight(w, per_row=wpr)
    colsum = q8.q8_colsum(qw)
    t1.record()
    torch.cuda.synchronize()
    weight_prep_ms = t0.elapsed_time(t1)
    del w

    qa = torch.empty((M, K), dtype=torch.int8, device=device)
    s_a = torch.empty(M if apr else 1, dtype=torch.float32, device=device)
    z_a = None if sym else torch.empty(M if apr else 1, dtype=torch.int32, device=device)
    y = torch.empty((M, N), dtype=torch.float32, device=device)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    kernel = q8.q8_gemm_pick(M, N, K)
    # the layer's scratch for an fp16 copy of the activation codes (allocated once, like every buffer):
    # the quantizer writes the int8 codes and, in the same pass, the codes as fp16 values into it;
    # the CTA-pair kernel loads that copy by TMA (the two calls q8_linear_ws makes)
    ws = gemm_workspace(q8, M, N, K, device)
    ws16 = ws.view(torch.float16)[:M * K].view(M, K) if ws is not None else None

    def quantize():
        if ws16 is not None:
            q8.q8_quantize_act_dual(a, per_row=apr, symmetric=sym, qa=qa, qa16=ws16, s_a=s_a, z_a=z_a)
        else:
            q8.q8_quantize_act(a, per_row=apr, symmetric=sym, qa=qa, s_a=s_a, z_a=z_a)

    def gemm():
        if ws16 is not None:
            q8.q8_gemm_f16a(ws16, s_a, z_a, qw, s_w, colsum, out=y)
        else:
            q8.q8_gemm_dequant(qa, s_a, z_a, qw, s_w, colsum, y=y)

    def step():
        quantize()
        gemm()

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    assert q8.q8_device_error() == 0

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    launches0 = q8.q8_launch_count()
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        wall0 = time.perf_counter()
        for i in range(args.steps):
            flush.zero_()
            evs[i][0].record(stream)
            quantize()
            evs[i][1].record(stream)
            gemm()
            evs[i][2].record(stream)
        torch.cuda.synchronize()
        wall1 = time.perf_counter()
    barrier(world)
    launches = q8.q8_launch_count() - launches0
    assert q8.q8_device_error() == 0
    quant_ms = [e[0].elapsed_time(e[1]) for e in evs]
    gemm_ms = [e[1].elapsed_time(e[2]) for e in evs]
    step_ms = [q + g for q, g in zip(quant_ms, gemm_ms)]
    ms_step = max_over_ranks(statistics.mean(step_ms), world)

    ops = 2.0 * M * N * K
    value = job_rate(ops, world, ms_step)
    gemm_avg = statistics.mean(gemm_ms)
    quant_avg = statistics.mean(quant_ms)
    gemm_tops = ops / (gemm_avg * 1e-3) / 1e12
    quant_bytes = M * K * (7 if ws16 is not None else 5) + 4 * M     # fp32 in; int8 (+ fp16) codes out
    quant_gbs = quant_bytes / (quant_avg * 1e-3) / 1e9
    gemm_bytes = M * K * (2 if ws16 is not None else 1) + N * K + 4 * N + 4 * M + 4 * M * N

    # ---- the same GEMM without the workspace: activation codes converted in shared memory per tile
    direct = measure_gemm_direct(q8, qa, s_a, z_a, qw, s_w, colsum, y, flush, args, tc_peak, ops)

    # ---- the same step run back to back for seconds, with the clock the power limit leaves
    sustained = None if args.no_sustained else measure_sustained(q8, quantize, gemm, flush, args, local, ops,
                                                                 args.sustained_s)

    # ---- end to end through the public API: pinned host A in, y back to pinned host
    e2e = None if args.no_e2e else measure_e2e(q8, a, y, step, qw, s_w, colsum, sym, ops, world, args)

    # ---- decode-shaped workload (HBM-bound): same step, reported beside the headline
    decode = None if args.no_decode else measure_decode(q8, device, args, hbm_peak, flush)

    # ---- W4A8: the same layers with int4 weights
    w4 = None if args.no_decode else measure_w4a8(q8, device, qa, s_a, flush, args, hbm_peak, ops, ws)

    # ---- block-scaled (E8M0 per K-group) weights on the same layers
    mx = None if args.no_decode else measure_mx(q8, device, qa, s_a, flush, args, hbm_peak, ops, ws)

    # ---- the same GEMM with the bias + bf16 epilogue (the pages' output side)
    epi = measure_epilogue_bf16(q8, qa, s_a, qw, s_w, flush, args, ops)

    # ---- the same step with the activation codes written as fp16 values (TMA-fed A operand)
    f16a = measure_f16a(q8, a, qw, s_w, y, flush, args, hbm_peak, tc_peak, ops) if sym else None

    # ---- fused RMSNorm + per-token quantization of the same activations (HBM-bound)
    rmsq = measure_rmsnorm_quantize(q8, a, qa, s_a, flush, args, hbm_peak)

    # ---- every workload of the scope: the small ones measured here, decode and the headline above
    configs = {}
    if not args.no_configs:
        for name in ("tiny", "prefill2k", "relu4k"):
            configs[name] = measure_config(q8, name, device, args, hbm_peak, tc_peak, flush)
        if decode is not None:
            dq, dg = decode["quant_ms"], decode["gemm_ms"]
            dwl = workloads.WORKLOADS[DECODE]
            dqb = step_bytes(dwl)[0]
            configs[DECODE] = {
                "workload": decode["workload"], "M": dwl.M, "N": dwl.N, "K": dwl.K, "gemm_kernel": decode["gemm_kernel"],
                "ms_per_step": decode["ms_per_step"], "TOPS": decode["TOPS"], "timing": decode["timing"],
                "quantizer": {"ms": dq, "GB/s": round(dqb / (dq * 1e-3) / 1e9, 1), "bytes": dqb,
                              "note": "16 rows: launch-latency bound"},
                "gemm": {"ms": dg, "GB/s": decode["gemm_GB/s"]},
                "roofline": {"bound": "hbm", "kernel": f"gemm_{decode['gemm_kernel']}", "achieved": decode["gemm_GB/s"],
                             "peak": hbm_peak, "unit": "GB/s", "frac": decode["gemm_frac_hbm"],
                             "algorithmic_bytes_per_launch": decode["algorithmic_bytes"], "ms_per_launch": dg}}
        configs[HEADLINE] = {
            "workload": f"{HEADLINE}: A fp32 [{M},{K}] per-token sym x W int8 [{N},{K}] per-channel sym",
            "M": M, "N": N, "K": K, "gemm_kernel": kernel, "ms_per_step": round(ms_step, 4),
            "TOPS": round(value / world, 2),
            "quantizer": {"ms": round(quant_avg, 4), "GB/s": round(quant_gbs, 1),
                          "frac_hbm": round(quant_gbs / hbm_peak, 4), "bytes": quant_bytes},
            "gemm": {"ms": round(gemm_avg, 4), "TFLOP/s": round(gemm_tops, 1)},
            "roofline": {"bound": "tensor", "kernel": f"gemm_{kernel}", "achieved": round(gemm_tops, 1),
                         "peak": tc_peak, "unit": "TFLOP/s", "frac": round(gemm_tops / tc_peak, 4),
                         "algorithmic_bytes_per_launch": gemm_bytes, "ms_per_launch": round(gemm_avg, 4)}}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = cpu_baseline(budget_s=args.cpu_budget)
        cores = len(os.sched_getaffinity(0))
        for name, entry in configs.items():
            entry["cpu_baseline"] = {"threaded": cpu} if name == HEADLINE else config_cpu(name, cores)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "TOPS", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
            "step_ms": {"mean": round(statistics.mean(step_ms), 4), "min": round(min(step_ms), 4),
                        "median": round(statistics.median(step_ms), 4)},
            "gemm_ms": {"mean": round(gemm_avg, 4), "min": round(min(gemm_ms), 4),
                        "median": round(statistics.median(gemm_ms), 4)},
            "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "int8", "data": "synthetic",
            "config": {"workload": f"{HEADLINE}: A fp32 [{M},{K}] per-token sym x W int8 [{N},{K}] per-channel"
                                   f" sym -> y fp32 [{M},{N}]",
                       "M": M, "N": N, "K": K, "gemm_kernel": kernel,
                       "gemm_path": ("the quantizer writes the int8 codes and, in the same pass, the codes as fp16 "
                                     "values into the layer's workspace (q8_quantize_act_dual); the CTA-pair kernel "
                                     "loads that copy by TMA (q8_gemm_f16a): the two calls of q8_linear_ws")
                       if ws is not None else "q8_gemm_dequant",
                       "l2": "flushed before every step (256 MiB write)",
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "roofline": {"bound": "tensor",
                         "kernel": f"gemm_{kernel}" + (" (fp16 copy of the codes)" if ws is not None else ""),
                         "achieved": round(gemm_tops, 1),
                         "peak": tc_peak, "unit": "TFLOP/s", "frac": round(gemm_tops / tc_peak, 4),
                         "peak_source": f"{peak_kind} bf16 dense burst (the GEMM runs tcgen05 kind::f16; fp16 = bf16 rate)",
                         "timing": "CUDA events around the whole GEMM call (the tensor-core kernel and the K-split "
                                   "kernels)",
                         "traffic": measured_traffic(kernel + ("_f16a" if ws is not None else "")),
                         "algorithmic_bytes_per_launch": gemm_bytes, "ms_per_launch": round(gemm_avg, 4)},
            "quantizer": {"ms": round(quant_avg, 4), "GB/s": round(quant_gbs, 1), "frac_hbm": round(quant_gbs / hbm_peak, 4),
                          "bytes": quant_bytes},
            "decode": decode,
            "rmsnorm_quantize": rmsq,
            "gemm_bias_bf16": epi,
            "f16_codes": f16a,
            "gemm_int8_direct": direct,
            "configs": configs,
            "sustained": sustained,
            "w4a8": w4,
            "block_scaled": mx,
            "e2e": e2e,
            "gpu_launches": int(launches),
            "weight_prep_ms": round(weight_prep_ms, 3),
            "clocks": clocks.summary(),
            "cpu_baseline": cpu,
            "wall_s_timed": round(wall1 - wall0, 3),
        }
        print(json.dumps(add_nominal_hbm(line)))


def gemm_workspace(q8, M, N, K, device):
    """The GEMM's optional scratch (an fp16 copy of the activation codes) for this shape, or None."""
    import torch
    n = q8.q8_gemm_workspace(M, N, K)
    return torch.empty(n, dtype=torch.uint8, device=device) if n else None


def measure_gemm_direct(q8, qa, s_a, z_a, qw, s_w, colsum, y, flush, args, tc_peak, ops):
    """The headline GEMM without a workspace (q8_gemm_dequant): the CTA-pair kernel converts every
    activation code to fp16 in shared memory once per 256-column tile; L2 flushed per launch."""
    import torch
    for _ in range(max(3, args.warmup)):
        flush.zero_()
        q8.q8_gemm_dequant(qa, s_a, z_a, qw, s_w, colsum, y=y)
    torch.cuda.synchronize()
    ms = []
    for _ in range(max(5, args.steps)):
        flush.zero_()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        q8.q8_gemm_dequant(qa, s_a, z_a, qw, s_w, colsum, y=y)
        e1.record()
        torch.cuda.synchronize()
        ms.append(e0.elapsed_time(e1))
    assert q8.q8_device_error() == 0
    mean = statistics.mean(ms)
    tf = ops / (mean * 1e-3) / 1e12
    return {"api": "q8_gemm_dequant (no workspace)", "ms": round(mean, 4), "TFLOP/s": round(tf, 1),
            "frac": round(tf / tc_peak, 4)}


def measure_e2e(q8, a, y, step, qw, s_w, colsum, sym, ops, world, args):
    """The layer through the public host-buffer call q8_linear_host: A in pinned host memory,
    y back to pinned host memory, both copies inside the timed region (overlapped with the
    device work slice by slice). For comparison, the same step with one whole copy in, the
    device step and one whole copy out in sequence (`serial_ms_per_step`)."""
    import torch
    M, K = a.shape
    N = y.shape[1]
    a_host = torch.empty((M, K), dtype=torch.float32, pin_memory=True)
    a_host.copy_(a.cpu())
    y_host = torch.empty((M, N), dtype=torch.float32, pin_memory=True)
    ws = torch.empty(q8.q8_linear_host_workspace(M, N, K), dtype=torch.uint8, device=a.device)
    stream = torch.cuda.current_stream()
    steps = max(10, args.steps)

    def timed(fn):
        for _ in range(2):
            fn()
        torch.cuda.synchronize()
        barrier(world)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return max_over_ranks(e0.elapsed_time(e1) / steps, world)

    def serial():
        a.copy_(a_host, non_blocking=True)
        step()
        y_host.copy_(y, non_blocking=True)

    ms_serial = timed(serial)
    ms = timed(lambda: q8.q8_linear_host(a_host, qw, s_w, colsum, y_host, symmetric=sym, workspace=ws))
    return {"value": round(job_rate(ops, world, ms), 3), "unit": "TOPS", "h2d_bytes_per_step": M * K * 4,
            "d2h_bytes_per_step": M * N * 4, "ms_per_step": round(ms, 3), "api": "q8_linear_host",
            "serial_ms_per_step": round(ms_serial, 3)}


def measure_decode(q8, device, args, hbm_peak, flush, kernels=("decode", "decode_tc", "tcgen05_pair", "skinny")):
    """Decode-shaped workload (16 tokens, HBM-bound): the step with each GEMM kernel."""
    import torch
    wl, a, w = layer_inputs(DECODE, device)
    M, N, K = wl.M, wl.N, wl.K
    qw, s_w = q8.q8_quantize_weight(w, per_row=True)
    del w
    qa = torch.empty((M, K), dtype=torch.int8, device=device)
    s_a = torch.empty(M, dtype=torch.float32, device=device)
    y = torch.empty((M, N), dtype=torch.float32, device=device)
    pick = q8.q8_gemm_pick(M, N, K)
    gemm_bytes = N * K + M * K + 4 * N + 4 * M + 4 * M * N

    def timed(kernel):
        """Mean times over back-to-back launches (one event pair around a graph of n launches).
        No L2 flush: W (N K bytes) is larger than L2, so each launch streams it from HBM, and
        a flush would add its dirty-line write-back to the next launch."""
        def quant():
            q8.q8_quantize_act(a, qa=qa, s_a=s_a)

        def gemm():
            q8.q8_gemm_dequant(qa, s_a, None, qw, s_w, y=y, kernel=kernel)

        def layer():
            # the default kernel through the one-call layer (its weight stream may start while the
            # quantizer runs); an explicit kernel as the two calls
            if kernel == pick:
                q8.q8_linear(a, qw, s_w, qa=qa, s_a=s_a, y=y)
            else:
                quant()
                gemm()

        def loop(fn, n):
            # n launches captured in one CUDA graph, so that host launch overhead (the 16-row
            # quantizer runs for a few microseconds) does not enter the device time
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, capture_error_mode="thread_local"):
                for _ in range(n):
                    fn()
            graph.replay()
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            graph.replay()
            e1.record()
            torch.cuda.synchronize()
            return e0.elapsed_time(e1) / n

        for _ in range(max(3, args.warmup)):
            quant()
            gemm()
        torch.cuda.synchronize()
        n = max(20, args.steps)
        q_ms = loop(quant, n)
        g_ms = loop(gemm, n)
        s_ms = loop(layer, n)
        return q_ms, g_ms, s_ms

    per_kernel = {}
    quant_ms = gq = step = None
    for kernel in kernels:
        qm, gm, sm = timed(kernel)
        per_kernel[kernel] = {"gemm_ms": round(gm, 4),
                              "gemm_frac_hbm": round(gemm_bytes / (gm * 1e-3) / 1e9 / hbm_peak, 4)}
        if kernel == pick:
            quant_ms, gq, step = qm, gm, sm
    return {"workload": f"{DECODE}: A [{M},{K}] x W int8 [{N},{K}]", "gemm_kernel": pick,
            "timing": "mean over back-to-back launches in a CUDA graph; W exceeds L2, no flush",
            "ms_per_step": round(step, 4), "TOPS": round(2.0 * M * N * K / (step * 1e-3) / 1e12, 2),
            "quant_ms": round(quant_ms, 4), "gemm_ms": round(gq, 4),
            "gemm_GB/s": round(gemm_bytes / (gq * 1e-3) / 1e9, 1),
            "gemm_frac_hbm": round(gemm_bytes / (gq * 1e-3) / 1e9 / hbm_peak, 4),
            "algorithmic_bytes": gemm_bytes, "per_kernel": per_kernel}


def flushed_ms(fn, flush, args):
    """Mean CUDA-event time of fn() with the L2 flushed before every launch."""
    import torch
    for _ in range(max(3, args.warmup)):
        flush.zero_()
        fn()
    torch.cuda.synchronize()
    ms = []
    for _ in range(max(5, args.steps)):
        flush.zero_()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        torch.cuda.synchronize()
        ms.append(e0.elapsed_time(e1))
    return statistics.mean(ms)


def measure_w4a8(q8, device, qa, s_a, flush, args, hbm_peak, ops, ws=None):
    """W4A8 (packed int4 weights): the decode GEMM (graph-timed back-to-back launches that cycle
    through three copies of the int4 weights: one copy, N K / 2 = 117 MB, fits in the 129 MB L2,
    so each launch reads a copy last touched 235 MB of traffic earlier) and the prefill GEMM (L2
    flushed per launch), without and with the layer's workspace (the codes copied once as fp16
    values, loaded by TMA; the copy is inside the timed call)."""
    import torch

    def graph_ms(fn, n):
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, capture_error_mode="thread_local"):
            for _ in range(n):
                fn()
        graph.replay()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        graph.replay()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n

    wl, a_d, w_d = layer_inputs(DECODE, device)
    Md, Nd, Kd = wl.M, wl.N, wl.K
    qw4, s4 = q8.q8_quantize_weight_int4(w_d)
    del w_d
    copies = [qw4, qw4.clone(), qw4.clone()]
    qad, sad, _ = q8.q8_quantize_act(a_d)
    yd = torch.empty((Md, Nd), dtype=torch.float32, device=device)
    turn = [0]

    def dec():
        q8.q8_gemm_w4a8(qad, sad, None, copies[turn[0] % 3], s4, out=yd)
        turn[0] += 1
    for _ in range(3):
        dec()
    dms = graph_ms(dec, 3 * max(7, args.steps))
    dbytes = Nd * Kd // 2 + Md * Kd + 4 * Nd + 4 * Md + 4 * Md * Nd
    del qw4, copies, yd

    M, K = qa.shape
    wlh = workloads.WORKLOADS[HEADLINE]
    wp = torch.from_numpy(workloads.make_weights(wlh)).to(device)
    qw4p, s4p = q8.q8_quantize_weight_int4(wp)
    del wp
    y = torch.empty((M, qw4p.shape[0]), dtype=torch.float32, device=device)
    pms = flushed_ms(lambda: q8.q8_gemm_w4a8(qa, s_a, None, qw4p, s4p, out=y), flush, args)
    prefill_ws = None
    if ws is not None and ws.numel() >= 2 * M * K:
        wms = flushed_ms(lambda: q8.q8_gemm_w4a8(qa, s_a, None, qw4p, s4p, out=y, workspace=ws), flush, args)
        prefill_ws = {"api": "q8_gemm_w4a8_ws", "gemm_ms": round(wms, 4), "TFLOP/s": round(ops / (wms * 1e-3) / 1e12, 1)}
    return {"decode": {"workload": f"{DECODE}: A [{Md},{Kd}] x W int4 [{Nd},{Kd}]", "gemm_ms": round(dms, 4),
                       "GB/s": round(dbytes / (dms * 1e-3) / 1e9, 1),
                       "frac_hbm": round(dbytes / (dms * 1e-3) / 1e9 / hbm_peak, 4), "algorithmic_bytes": dbytes},
            "prefill": {"workload": f"{HEADLINE}: A [{M},{K}] x W int4 [{qw4p.shape[0]},{K}]", "gemm_ms": round(pms, 4),
                        "TFLOP/s": round(ops / (pms * 1e-3) / 1e12, 1)},
            "prefill_ws": prefill_ws}


def measure_mx(q8, device, qa, s_a, flush, args, hbm_peak, ops, ws=None):
    """Block-scaled int8 weights (one E8M0 scale per 32 or 128 K): the prefill GEMM (L2 flushed
    per launch) for both granularities, without and with the layer's workspace, and the decode
    layer (CUDA graph of back-to-back launches; the int8 weights, 235 MB, exceed L2)."""
    import torch
    M, K = qa.shape
    wlh = workloads.WORKLOADS[HEADLINE]
    wp = torch.from_numpy(workloads.make_weights(wlh)).to(device)
    out = {}
    for G in (32, 128):
        qw, sf = q8.q8_quantize_weight_mx(wp, G)
        y = torch.empty((M, qw.shape[0]), dtype=torch.float32, device=device)
        mean = flushed_ms(lambda: q8.q8_gemm_mx(qa, s_a, qw, sf, G, out=y), flush, args)
        out[f"prefill_g{G}"] = {"workload": f"{HEADLINE}: A [{M},{K}] x W int8 [{qw.shape[0]},{K}], E8M0 per {G} K",
                                "gemm_ms": round(mean, 4), "TFLOP/s": round(ops / (mean * 1e-3) / 1e12, 1)}
        if ws is not None and ws.numel() >= 2 * M * K:
            wms = flushed_ms(lambda: q8.q8_gemm_mx(qa, s_a, qw, sf, G, out=y, workspace=ws), flush, args)
            out[f"prefill_g{G}"]["ws"] = {"api": "q8_gemm_mx_ws", "gemm_ms": round(wms, 4),
                                          "TFLOP/s": round(ops / (wms * 1e-3) / 1e12, 1)}
        del qw, sf, y
    del wp
    wl, a_d, w_d = layer_inputs(DECODE, device)
    Md, Nd, Kd = wl.M, wl.N, wl.K
    qw, sf = q8.q8_quantize_weight_mx(w_d, 32)
    del w_d
    qad, sad, _ = q8.q8_quantize_act(a_d)
    yd = torch.empty((Md, Nd), dtype=torch.float32, device=device)
    for _ in range(3):
        q8.q8_gemm_mx(qad, sad, qw, sf, 32, out=yd)
    n = max(20, args.steps)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, capture_error_mode="thread_local"):
        for _ in range(n):
            q8.q8_gemm_mx(qad, sad, qw, sf, 32, out=yd)
    graph.replay()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    graph.replay()
    e1.record()
    torch.cuda.synchronize()
    dms = e0.elapsed_time(e1) / n
    dbytes = Nd * Kd + Nd * Kd // 32 + Md * Kd + 4 * Md + 4 * Md * Nd   # codes, E8M0 bytes, tokens, s_a, y
    out["decode_g32"] = {"workload": f"{DECODE}: A [{Md},{Kd}] x W int8 [{Nd},{Kd}], E8M0 per 32 K (decode kernel)",
                         "gemm_ms": round(dms, 4), "GB/s": round(dbytes / (dms * 1e-3) / 1e9, 1),
                         "frac_hbm": round(dbytes / (dms * 1e-3) / 1e9 / hbm_peak, 4)}
    return out


def measure_epilogue_bf16(q8, qa, s_a, qw, s_w, flush, args, ops):
    """The headline GEMM with a bias and bf16 output (q8_gemm_epilogue), L2 flushed before each
    launch: the output write halves (2 bytes per element)."""
    import torch
    N = qw.shape[0]
    bias = torch.from_numpy(workloads.gaussian((N,), 50)).to(qa.device)
    out = torch.empty((qa.shape[0], N), dtype=torch.bfloat16, device=qa.device)
    for _ in range(max(3, args.warmup)):
        flush.zero_()
        q8.q8_gemm_epilogue(qa, s_a, None, qw, s_w, bias=bias, out_dtype=torch.bfloat16, out=out)
    torch.cuda.synchronize()
    ms = []
    for _ in range(max(5, args.steps)):
        flush.zero_()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        q8.q8_gemm_epilogue(qa, s_a, None, qw, s_w, bias=bias, out_dtype=torch.bfloat16, out=out)
        e1.record()
        torch.cuda.synchronize()
        ms.append(e0.elapsed_time(e1))
    mean = statistics.mean(ms)
    return {"ms": round(mean, 4), "TFLOP/s": round(ops / (mean * 1e-3) / 1e12, 1),
            "kernel": q8.q8_gemm_pick(qa.shape[0], N, qa.shape[1])}


def measure_f16a(q8, a, qw, s_w, y, flush, args, hbm_peak, tc_peak, ops):
    """The headline step with the activation codes stored as fp16 values: q8_quantize_act_f16
    (read A, 4 M K bytes; write codes, 2 M K) then q8_gemm_f16a (the pair kernel loading the fp16
    codes by TMA into its operand stages), L2 flushed before each step."""
    import torch
    M, K = a.shape
    qa16 = torch.empty((M, K), dtype=torch.float16, device=a.device)
    s_a = torch.empty(M, dtype=torch.float32, device=a.device)

    def quant():
        q8.q8_quantize_act_f16(a, per_row=True, symmetric=True, qa16=qa16, s_a=s_a)

    def gemm():
        q8.q8_gemm_f16a(qa16, s_a, None, qw, s_w, out=y)

    for _ in range(max(3, args.warmup)):
        flush.zero_()
        quant()
        gemm()
    torch.cuda.synchronize()
    qms, gms = [], []
    for _ in range(max(5, args.steps)):
        flush.zero_()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        ev[0].record()
        quant()
        ev[1].record()
        gemm()
        ev[2].record()
        torch.cuda.synchronize()
        qms.append(ev[0].elapsed_time(ev[1]))
        gms.append(ev[1].elapsed_time(ev[2]))
    assert q8.q8_device_error() == 0
    q, g = statistics.mean(qms), statistics.mean(gms)
    qbytes = M * K * 6 + 4 * M
    gtf = ops / (g * 1e-3) / 1e12
    return {"workload": "same layer; codes as fp16 values", "step_ms": round(q + g, 4),
            "TOPS": round(ops / ((q + g) * 1e-3) / 1e12, 1),
            "quantizer": {"ms": round(q, 4), "GB/s": round(qbytes / (q * 1e-3) / 1e9, 1),
                          "frac_hbm": round(qbytes / (q * 1e-3) / 1e9 / hbm_peak, 4), "bytes": qbytes},
            "gemm": {"ms": round(g, 4), "TFLOP/s": round(gtf, 1), "frac": round(gtf / tc_peak, 4),
                     "kernel": "tcgen05_pair (fp16 A by TMA)"}}


def measure_rmsnorm_quantize(q8, a, qa, s_a, flush, args, hbm_peak):
    """The fused norm-and-quantize kernel on the headline activations, L2 flushed before
    each launch; algorithmic bytes: read A (4 M K) and gamma (4 K), write codes (M K) and
    scales (4 M)."""
    import torch
    M, K = a.shape
    gamma = torch.from_numpy(workloads.make_norm_weights(K, seed=4)).to(a.device)
    for _ in range(max(3, args.warmup)):
        flush.zero_()
        q8.q8_rmsnorm_quantize_act(a, gamma, 1e-6, qa=qa, s_a=s_a)
    torch.cuda.synchronize()
    ms = []
    for _ in range(max(10, args.steps)):
        flush.zero_()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        q8.q8_rmsnorm_quantize_act(a, gamma, 1e-6, qa=qa, s_a=s_a)
        e1.record()
        torch.cuda.synchronize()
        ms.append(e0.elapsed_time(e1))
    mean = statistics.mean(ms)
    nbytes = 5 * M * K + 4 * M + 4 * K
    return {"workload": f"{HEADLINE} activations [{M},{K}], gamma [{K}], eps 1e-6", "ms": round(mean, 4),
            "GB/s": round(nbytes / (mean * 1e-3) / 1e9, 1), "frac_hbm": round(nbytes / (mean * 1e-3) / 1e9 / hbm_peak, 4),
            "bytes": nbytes}


def measure_config(q8, name, device, args, hbm_peak, tc_peak, flush):
    """One workload's step exactly as the headline is timed: q8_quantize_act then q8_gemm_dequant on
    inputs resident in HBM, the 256 MiB L2 flush before every step, CUDA events around each kernel
    on the launching stream. The flush (68 us of device time) lets the host queue the step's two
    launches before the device reaches them, so the events see device time, not launch gaps."""
    import torch
    wl, a, w = layer_inputs(name, device)
    M, N, K = wl.M, wl.N, wl.K
    apr, wpr, sym = wl.act_granularity == "row", wl.w_granularity == "row", wl.act_symmetric
    qw, s_w = q8.q8_quantize_weight(w, per_row=wpr)
    colsum = None if sym else q8.q8_colsum(qw)
    del w
    qa = torch.empty((M, K), dtype=torch.int8, device=device)
    s_a = torch.empty(M if apr else 1, dtype=torch.float32, device=device)
    z_a = None if sym else torch.empty(M if apr else 1, dtype=torch.int32, device=device)
    y = torch.empty((M, N), dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream()
    kernel = q8.q8_gemm_pick(M, N, K)
    ws = gemm_workspace(q8, M, N, K, device)
    ws16 = ws.view(torch.float16)[:M * K].view(M, K) if ws is not None else None

    def quantize():   # as the headline: with a workspace, the int8 codes and their fp16 copy in one pass
        if ws16 is not None:
            q8.q8_quantize_act_dual(a, per_row=apr, symmetric=sym, qa=qa, qa16=ws16, s_a=s_a, z_a=z_a)
        else:
            q8.q8_quantize_act(a, per_row=apr, symmetric=sym, qa=qa, s_a=s_a, z_a=z_a)

    def gemm():
        if ws16 is not None:
            q8.q8_gemm_f16a(ws16, s_a, z_a, qw, s_w, colsum, out=y)
        else:
            q8.q8_gemm_dequant(qa, s_a, z_a, qw, s_w, colsum, y=y)

    for _ in range(max(3, args.warmup)):
        flush.zero_()
        quantize()
        gemm()
    torch.cuda.synchronize()
    n = max(20, args.steps)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n)]
    for i in range(n):
        flush.zero_()
        evs[i][0].record(stream)
        quantize()
        evs[i][1].record(stream)
        gemm()
        evs[i][2].record(stream)
    torch.cuda.synchronize()
    assert q8.q8_device_error() == 0
    qms = [e[0].elapsed_time(e[1]) for e in evs]
    gms = [e[1].elapsed_time(e[2]) for e in evs]
    sms = [q + g for q, g in zip(qms, gms)]
    q, g, st = statistics.mean(qms), statistics.mean(gms), statistics.mean(sms)
    ops = 2.0 * M * N * K
    qbytes, gbytes = step_bytes(wl)
    if ws16 is not None:   # the fp16 copy: written by the quantizer, read by the GEMM instead of the int8 codes
        qbytes += 2 * M * K
        gbytes += M * K
    gtf = ops / (g * 1e-3) / 1e12
    bound = {"tiny": "latency", "decode": "hbm"}.get(name, "tensor")
    if bound == "tensor":
        roof = {"bound": "tensor", "kernel": f"gemm_{kernel}", "achieved": round(gtf, 1), "peak": tc_peak,
                "unit": "TFLOP/s", "frac": round(gtf / tc_peak, 4)}
    elif bound == "hbm":
        gbs = gbytes / (g * 1e-3) / 1e9
        roof = {"bound": "hbm", "kernel": f"gemm_{kernel}", "achieved": round(gbs, 1), "peak": hbm_peak,
                "unit": "GB/s", "frac": round(gbs / hbm_peak, 4)}
    else:
        roof = {"bound": "latency", "kernel": f"gemm_{kernel}", "achieved": round(g * 1e3, 2), "unit": "us",
                "peak": None, "frac": None, "note": "launch-latency bound: reported, no roofline fraction"}
    roof.update({"algorithmic_bytes_per_launch": gbytes, "ms_per_launch": round(g, 4)})
    return {
        "workload": f"{name}: A fp32 [{M},{K}] per-{'token' if apr else 'tensor'} "
                    f"{'sym' if sym else 'asym'} x W int8 [{N},{K}] per-{'channel' if wpr else 'tensor'} sym",
        "M": M, "N": N, "K": K, "gemm_kernel": kernel, "workspace_bytes": 0 if ws is None else ws.numel(), "steps": n,
        "ms_per_step": round(st, 4), "step_ms": {"min": round(min(sms), 4), "median": round(statistics.median(sms), 4)},
        "TOPS": round(ops / (st * 1e-3) / 1e12, 3),
        "quantizer": {"ms": round(q, 4), "GB/s": round(qbytes / (q * 1e-3) / 1e9, 1),
                      "frac_hbm": round(qbytes / (q * 1e-3) / 1e9 / hbm_peak, 4), "bytes": qbytes},
        "gemm": {"ms": round(g, 4), "TFLOP/s": round(gtf, 2)},
        "roofline": roof,
    }


def oracle_timing(name, threads, rows=None, budget_s=None):
    """The oracle as it stands on `threads` host cores: quantize the rows of A (the workload's
    granularity and symmetry) and run the integer GEMM and epilogue against the offline-quantized
    weights (C, int64 accumulation, OpenMP over output rows). All rows, or a row sample sized from a
    short probe to take about budget_s seconds."""
    import oracle
    wl = workloads.WORKLOADS[name]
    a_all, w = host_inputs(name)
    apr, wpr, sym = wl.act_granularity == "row", wl.w_granularity == "row", wl.act_symmetric
    qw, sw = oracle.quantize_sym(w, wpr)

    def run(r0, r):
        a = a_all[r0:r0 + r]
        t = time.perf_counter()
        if sym:
            qa, sa = oracle.quantize_sym(a, apr)
            za = None
        else:
            qa, sa, za = oracle.quantize_asym(a, apr)
        _, st = oracle.linear_codes(qa, sa, za, qw, sw, apr, wpr, threads=threads)
        assert st == oracle.OK
        return time.perf_counter() - t

    if rows is None and budget_s is not None and apr:
        probe = max(1, threads)
        dt = run(0, probe)
        rows = int(max(probe, min(wl.M, probe * budget_s / max(dt, 1e-3))))
        rows = max(probe, rows // probe * probe)
    rows = wl.M if (rows is None or not apr) else min(rows, wl.M)
    dt = run(0, rows)
    if dt < 0.2:   # short runs are repeated (about 0.2 s in all) and averaged
        reps = int(0.2 / max(dt, 1e-4)) + 1
        dt = sum(run(0, rows) for _ in range(reps)) / reps
    ops = 2.0 * rows * wl.N * wl.K
    whole = "all" if rows == wl.M else f"{rows} of {wl.M}"
    return {"value": round(ops / dt / 1e12, 6), "unit": "TOPS", "cores": threads, "kind": "oracle",
            "sample": f"{whole} token rows of {name} (quantize the rows, int64 dot products against all "
                      f"{wl.N} channels, K={wl.K}, epilogue), {dt:.3f} s", "seconds": round(dt, 3)}


def config_cpu(name, cores):
    """Oracle timings of one workload: threaded over all host cores (full runs where they take a few
    seconds, a row sample of the large prefill), and single-core runs of the tiny, prefill2k and
    decode workloads."""
    out = {}
    if name == HEADLINE:
        out["threaded"] = oracle_timing(name, cores, budget_s=8.0)
    else:
        out["threaded"] = oracle_timing(name, cores)
    if name in ("tiny", "prefill2k", "decode"):
        out["single_core"] = oracle_timing(name, 1)
    return out


def measure_sustained(q8, quantize, gemm, flush, args, local, ops, seconds):
    """The headline step back to back for about `seconds` (each step: the L2 flush, then the
    quantizer and the GEMM between CUDA events), with the SM clock sampled through NVML: the rate a
    layer keeps up once the power limit has pulled the clock down, against the sustained bf16 peak."""
    import torch
    stream = torch.cuda.current_stream()
    probe = []
    for _ in range(5):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        flush.zero_()
        quantize()
        gemm()
        e1.record(stream)
        torch.cuda.synchronize()
        probe.append(e0.elapsed_time(e1))
    n = int(max(50, seconds * 1e3 / statistics.median(probe)))
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n)]
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        w0 = time.perf_counter()
        for i in range(n):
            flush.zero_()
            evs[i][0].record(stream)
            quantize()
            evs[i][1].record(stream)
            gemm()
            evs[i][2].record(stream)
        torch.cuda.synchronize()
        w1 = time.perf_counter()
    assert q8.q8_device_error() == 0
    qms = [e[0].elapsed_time(e[1]) for e in evs]
    gms = [e[1].elapsed_time(e[2]) for e in evs]
    last = n // 2                                   # the second half: after the clock has settled
    st = statistics.mean(q + g for q, g in zip(qms[last:], gms[last:]))
    g = statistics.mean(gms[last:])
    peak, kind = sustained_peak()
    gtf = ops / (g * 1e-3) / 1e12
    c = clocks.summary()
    return {"steps": n, "seconds": round(w1 - w0, 2), "ms_per_step": round(st, 4),
            "TOPS": round(ops / (st * 1e-3) / 1e12, 1), "gemm_ms": round(g, 4), "gemm_TFLOP/s": round(gtf, 1),
            "frac": round(gtf / peak, 4), "peak": peak, "peak_source": f"{kind} bf16 dense sustained",
            "first_half_ms_per_step": round(statistics.mean(q + g for q, g in zip(qms[:last], gms[:last])), 4),
            "sm_mhz_median": c["sm_mhz"], "sm_max_mhz": c["sm_max_mhz"], "reasons": c["reasons"],
            "clock_samples": c["samples"], "timing": "mean over the second half of the steps"}


# ------------------------------------------------------------------ the oracle (CPU baseline / reference arm)

class OracleSample:
    """The headline workload's inputs, with W quantized offline, for timing the oracle on row samples."""

    def __init__(self):
        import oracle
        self.oracle = oracle
        self.wl = workloads.WORKLOADS[HEADLINE]
        self.a = workloads.make_activations(self.wl)
        self.qw, self.sw = oracle.quantize_sym(workloads.make_weights(self.wl), True)
        self.cores = len(os.sched_getaffinity(0))

    def step(self, rows: int, start: int = 0):
        o = self.oracle
        a = self.a[start:start + rows]
        qa, sa = o.quantize_sym(a, True)
        y, st = o.linear_codes(qa, sa, None, self.qw, self.sw, True, True, threads=self.cores)
        assert st == o.OK
        return y

    def ops(self, rows):
        return 2.0 * rows * self.wl.N * self.wl.K


def cpu_baseline(budget_s: float = 15.0):
    s = OracleSample()
    rows = max(1, s.cores)
    t = time.perf_counter()
    s.step(rows)
    dt = time.perf_counter() - t
    rows = int(max(1, min(s.wl.M, rows * budget_s / max(dt, 1e-3))))
    rows = max(s.cores, (rows // s.cores) * s.cores)
    t = time.perf_counter()
    s.step(rows, start=rows)
    dt = time.perf_counter() - t
    return {"value": round(s.ops(rows) / dt / 1e12, 6), "unit": "TOPS", "cores": s.cores, "kind": "oracle",
            "sample": f"{rows} of {s.wl.M} token rows of {HEADLINE} (quantize rows + int64 dot products "
                      f"against all {s.wl.N} channels, K={s.wl.K}), {dt:.1f} s"}


def run_reference(args, world, rank):
    if rank != 0:
        return
    s = OracleSample()
    rows = s.cores
    t = time.perf_counter()
    s.step(rows)
    dt = time.perf_counter() - t
    per_step_target = min(8.0, 150.0 / max(1, args.steps + args.warmup))
    rows = int(max(s.cores, min(s.wl.M // 2, rows * per_step_target / max(dt, 1e-3))))
    for i in range(args.warmup):
        s.step(rows, start=(i * rows) % (s.wl.M - rows))
    times = []
    for i in range(args.steps):
        t = time.perf_counter()
        s.step(rows, start=((i + args.warmup) * rows) % (s.wl.M - rows))
        times.append(time.perf_counter() - t)
    ms = statistics.mean(times) * 1e3
    value = s.ops(rows) / (ms * 1e-3) / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TOPS", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "int8", "data": "synthetic",
        "config": {"workload": f"{HEADLINE} (row sample per step: {rows} tokens)", "M": s.wl.M, "N": s.wl.N,
                   "K": s.wl.K},
        "cpu_baseline": {"value": round(value, 6), "unit": "TOPS", "cores": s.cores, "kind": "oracle",
                         "sample": f"{rows} token rows per step"},
        "e2e": {"value": round(value, 6), "unit": "TOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end measurement")
    ap.add_argument("--no-decode", action="store_true", help="skip the decode-shaped workload")
    ap.add_argument("--no-configs", action="store_true", help="skip the tiny / prefill2k / relu4k workloads")
    ap.add_argument("--no-sustained", action="store_true", help="skip the seconds-long sustained run")
    ap.add_argument("--sustained-s", type=float, default=2.5, help="length of the sustained run (s)")
    ap.add_argument("--w4-only", action="store_true",
                    help="only the W4A8 (int4 weight) measurements (one JSON object, for profiling)")
    ap.add_argument("--mx-only", action="store_true",
                    help="only the block-scaled weight measurements (one JSON object, for profiling)")
    ap.add_argument("--rms-only", action="store_true",
                    help="only the fused RMSNorm + quantize measurement (one JSON object, for profiling)")
    ap.add_argument("--decode-only", action="store_true",
                    help="only the decode-shaped workload (one JSON object, for profiling)")
    ap.add_argument("--f16a-only", action="store_true",
                    help="only the headline step with fp16-valued activation codes (one JSON object, for profiling)")
    args = ap.parse_args()
    if args.impl == "reference":
        world = int(os.environ.get("WORLD_SIZE", "1"))
        rank = int(os.environ.get("RANK", "0"))
        run_reference(args, world, rank)
        return
    world, rank, local = dist_setup()
    if args.w4_only:
        import torch
        import int8_quantized_gemm_gb300 as q8
        from int8_quantized_gemm_gb300 import build
        build.build()
        q8.load()
        device = torch.device("cuda", local)
        torch.cuda.set_device(device)
        flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
        wl = workloads.WORKLOADS[HEADLINE]
        a = torch.from_numpy(workloads.make_activations(wl)).to(device)
        qa, s_a, _ = q8.q8_quantize_act(a)
        del a
        ws = gemm_workspace(q8, wl.M, wl.N, wl.K, device)
        print(json.dumps(measure_w4a8(q8, device, qa, s_a, flush, args, peaks()[0], 2.0 * wl.M * wl.N * wl.K, ws)))
        return
    if args.mx_only:
        import torch
        import int8_quantized_gemm_gb300 as q8
        from int8_quantized_gemm_gb300 import build
        build.build()
        q8.load()
        device = torch.device("cuda", local)
        torch.cuda.set_device(device)
        flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
        wl = workloads.WORKLOADS[HEADLINE]
        a = torch.from_numpy(workloads.make_activations(wl)).to(device)
        qa, s_a, _ = q8.q8_quantize_act(a)
        del a
        ws = gemm_workspace(q8, wl.M, wl.N, wl.K, device)
        print(json.dumps(measure_mx(q8, device, qa, s_a, flush, args, peaks()[0], 2.0 * wl.M * wl.N * wl.K, ws)))
        return
    if args.rms_only:
        import torch
        import int8_quantized_gemm_gb300 as q8
        from int8_quantized_gemm_gb300 import build
        build.build()
        q8.load()
        device = torch.device("cuda", local)
        torch.cuda.set_device(device)
        flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
        wl = workloads.WORKLOADS[HEADLINE]
        a = torch.from_numpy(workloads.make_activations(wl)).to(device)
        qa = torch.empty((wl.M, wl.K), dtype=torch.int8, device=device)
        s_a = torch.empty(wl.M, dtype=torch.float32, device=device)
        print(json.dumps(measure_rmsnorm_quantize(q8, a, qa, s_a, flush, args, peaks()[0])))
        return
    if args.decode_only:
        import torch
        import int8_quantized_gemm_gb300 as q8
        from int8_quantized_gemm_gb300 import build
        build.build()
        q8.load()
        device = torch.device("cuda", local)
        torch.cuda.set_device(device)
        flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
        print(json.dumps(measure_decode(q8, device, args, peaks()[0], flush, kernels=("decode", "decode_tc"))))
        return
    if args.f16a_only:
        import torch
        import int8_quantized_gemm_gb300 as q8
        from int8_quantized_gemm_gb300 import build
        build.build()
        q8.load()
        device = torch.device("cuda", local)
        torch.cuda.set_device(device)
        hbm_peak, tc_peak, _ = peaks()
        wl, a, w = layer_inputs(HEADLINE, device)
        qw, s_w = q8.q8_quantize_weight(w, per_row=wl.w_granularity == "row")
        del w
        y = torch.empty((wl.M, wl.N), dtype=torch.float32, device=device)
        flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
        print(json.dumps(measure_f16a(q8, a, qw, s_w, y, flush, args, hbm_peak, tc_peak,
                                      2.0 * wl.M * wl.N * wl.K)))
        return
    run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
