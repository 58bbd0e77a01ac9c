#!/usr/bin/env python
"""Benchmark of the tensor-parallel MLP hot path on GB300.

One step = one pass of the whole path over one batch: the column-parallel
GEMM with the fused activation (all T shards), the row-parallel GEMM and the
all-reduce-sum, on the prefill workload (M = 2048 tokens, H = 4096,
F = 16384, T = 4, erf-GeLU, bf16 inputs, float32 accumulation).  Prints one
JSON line.  Under torchrun each rank runs an independent replica on its own
GPU (the path has no cross-GPU exchange: all shards live on one GPU), so the
scaling is weak and the value is the sum over ranks.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "TP-sharded MLP fwd TFLOP/s and % BF16 peak; shard-sum/decode HBM GB/s %"
WORKLOAD = "prefill_gelu_m2048_h4096_f16384_t4"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
PROFILE = os.path.join(ROOT, "profiles", "colpar_gemm_gelu_prefill_m2048_h4096_f16384_t4.md")
GEMM_SOURCES = [os.path.join(ROOT, "linear_sharding_gb300", "csrc", f)
                for f in ("tp_gemm_impl.cuh", "tp_gemm.cu", "tp_device.cuh", "tp_internal.h")]


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=("ours", "reference"), default="ours")
    p.add_argument("--variant", choices=("auto", "partials", "tmem_acc"), default="auto")
    p.add_argument("--extras", choices=("none", "all"), default="all",
                   help="secondary measurements at N=1 (all): decode, training, shard-sum, the "
                        "attention projections and the large SwiGLU prefill with every all-reduce "
                        "variant, the attention core and the transformer block")
    p.add_argument("--cpu-rows", type=int, default=64, help="rows of the oracle CPU-baseline sample")
    p.add_argument("--sustain-s", type=float, default=1.2,
                   help="seconds of back-to-back steps in the sustained leg (0: leave it out)")
    p.add_argument("--case", choices=("prefill", "decode", "shard_sum", "train", "block", "attention",
                                      "mlp", "oproj"),
                   default="prefill",
                   help="prefill: the headline step (default); decode / shard_sum: time only the "
                        "memory-bound decode MLP (H=8192, F=28672, T=8, SwiGLU, --decode-m tokens) "
                        "or the standalone shard-sum (T=8, n=8192*8192); train: the backward of the "
                        "prefill MLP; block: one transformer block (M=4096, 32x128 heads, T=8, "
                        "SwiGLU F=4H, causal); attention: the block's fused causal attention core "
                        "(M=4096, 32 heads of 128); mlp: tp_mlp_forward on --mlp-workload with "
                        "--variant; oproj: the row-parallel output projection of the attention "
                        "projections (M=4096, H=4096, T=8) with --variant; for profiling")
    p.add_argument("--mlp-workload", choices=("prefill_gelu", "prefill_swiglu_large"),
                   default="prefill_gelu",
                   help="--case mlp: M=2048 H=4096 F=16384 T=4 GeLU, or M=8192 H=8192 F=28672 T=8 "
                        "SwiGLU")
    p.add_argument("--decode-m", type=int, default=16)
    return p.parse_args(argv)


# ---- distributed plumbing (replicas) ------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return world, rank, local


def dist_init(world: int, backend: str):
    if world > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group(backend=backend)


def _reduce(value: float, op: str, device) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)
    return float(t.item())


def reduce_max(value: float, device="cpu") -> float:
    return _reduce(value, "max", device)


def reduce_sum(value: float, device="cpu") -> float:
    return _reduce(value, "sum", device)


def barrier(device=None):
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def aggregate(elapsed_s: float, units_per_rank: float, device="cpu"):
    """Whole-job throughput of replicas: the units all ranks processed over
    the slowest rank's time.  Returns (units/s, max elapsed)."""
    t = reduce_max(elapsed_s, device)
    units = reduce_sum(units_per_rank, device)
    return units / t, t


# ---- clocks ------------------------------------------------------------------

CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while work runs
    (the fallback when NVML cannot be loaded in-process)."""

    def __init__(self, gpu_index: int, period_ms: int = 20):
        self.path = tempfile.mktemp(prefix="clocks_", suffix=".csv")
        self.cmd = ["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits",
                    "-i", str(gpu_index), "-lms", str(period_ms)]
        self.proc = None

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(self.cmd, stdout=self.fh, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        return self

    def mark(self) -> float:
        return time.time()

    def window(self, t0: float, t1: float) -> dict:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no per-region samples (nvidia-smi)"]}

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) == 9:
                    rows.append(parts)
        os.unlink(self.path)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        samples = []
        for r in rows:
            try:
                sm, mx, pw = float(r[1]), float(r[2]), float(r[3])
            except ValueError:
                continue
            reasons = {name for name, flag in zip(names, r[5:9]) if flag.lower().startswith("active")}
            samples.append((0.0, sm, mx, pw, reasons))
        return summarize_clocks(samples)


# NVML clock-event reason bits (nvml.h, nvmlClocksEventReason*)
NVML_REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}


def summarize_clocks(samples) -> dict:
    """Median SM clock under load (samples drawing >= 30 % of the peak power
    seen), the maximum SM clock and every throttle reason seen."""
    if not samples:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
    pw_max = max(s[3] for s in samples)
    loaded = sorted(s[1] for s in samples if s[3] >= 0.3 * pw_max) or sorted(s[1] for s in samples)
    reasons = set()
    for s in samples:
        reasons |= s[4]
    return {"sm_mhz": loaded[len(loaded) // 2], "sm_max_mhz": max(s[2] for s in samples),
            "reasons": sorted(reasons), "samples": len(samples), "power_w_max": round(pw_max, 1)}


class NvmlClockSampler:
    """In-process NVML polling (ctypes, read-only queries) of the SM clock,
    power and clock-event reasons every `period_s`, from a thread, so that
    even a few-millisecond timed region gets samples.  window(t0, t1) returns
    the summary of the samples taken between two mark() times; stop() the
    summary of all, after one last sample."""

    def __init__(self, gpu_index: int, period_s: float = 0.002):
        import ctypes
        import threading
        self.ct = ctypes
        self.nvml = ctypes.CDLL("libnvidia-ml.so.1")
        if self.nvml.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.dev = ctypes.c_void_p()
        if self.nvml.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(gpu_index), ctypes.byref(self.dev)) != 0:
            raise OSError("no NVML device handle")
        self.reason_fn = getattr(self.nvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.nvml.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint()
        self.nvml.nvmlDeviceGetMaxClockInfo(self.dev, 1, ctypes.byref(mx))  # NVML_CLOCK_SM
        self.max_mhz = float(mx.value)
        self.period = period_s
        self.samples = []
        self.stop_ev = threading.Event()
        self.thread = threading.Thread(target=self._run, daemon=True)

    def _sample(self):
        ct = self.ct
        clk, pw, rs = ct.c_uint(), ct.c_uint(), ct.c_ulonglong()
        if self.nvml.nvmlDeviceGetClockInfo(self.dev, 1, ct.byref(clk)) != 0:
            return
        self.nvml.nvmlDeviceGetPowerUsage(self.dev, ct.byref(pw))
        self.reason_fn(self.dev, ct.byref(rs))
        reasons = {name for bit, name in NVML_REASONS.items() if rs.value & bit}
        self.samples.append((time.time(), float(clk.value), self.max_mhz, pw.value / 1e3, reasons))

    def _run(self):
        while not self.stop_ev.is_set():
            self._sample()
            time.sleep(self.period)

    def start(self):
        self.thread.start()
        return self

    def mark(self) -> float:
        return time.time()

    def window(self, t0: float, t1: float) -> dict:
        snap = list(self.samples)
        sel = [s for s in snap if t0 <= s[0] <= t1]
        note = None
        if not sel:  # a region shorter than the polling period: the first sample after it
            sel = [s for s in snap if s[0] >= t1][:1]
            note = "no sample inside the region; first sample after it"
        out = summarize_clocks(sel)
        if note:
            out["note"] = note
        return out

    def stop(self) -> dict:
        self.stop_ev.set()
        self.thread.join(timeout=5)
        self._sample()
        try:
            self.nvml.nvmlShutdown()
        except Exception:
            pass
        return summarize_clocks(self.samples)


def clock_sampler(gpu_index: int):
    try:
        return NvmlClockSampler(gpu_index).start()
    except (OSError, AttributeError):
        return ClockSampler(gpu_index).start()


def physical_gpu_index(local_rank: int) -> int:
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        ids = [v.strip() for v in vis.split(",") if v.strip()]
        if local_rank < len(ids) and ids[local_rank].isdigit():
            return int(ids[local_rank])
    return local_rank


# ---- roofline bookkeeping ------------------------------------------------------

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def gemm_source_sha() -> str:
    h = hashlib.sha256()
    for p in GEMM_SOURCES:
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic():
    """DRAM bytes per launch of the column-parallel GEMM from the committed ncu
    summary, or None if absent or taken on different kernel source."""
    try:
        text = open(PROFILE).read()
    except OSError:
        return None
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    sha = re.search(r"source_sha:\s*([0-9a-f]+)", text)
    if not m or not sha or sha.group(1) != gemm_source_sha():
        return None
    return float(m.group(1))


# ---- our implementation ---------------------------------------------------------

def _dev(a, device):
    import numpy as np
    import torch
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def cpu_baseline(w: dict, rows: int) -> dict:
    """The fp64 oracle as it stands, on a seeded sample of rows of the same
    workload, on this host's cores."""
    import numpy as np
    import oracle
    from synth import mlp_inputs
    oracle.build()
    d = mlp_inputs(M=w["M"], H=w["H"], F=w["F"], act=w["act"], dtype=w["dtype"], seed=0)
    sample = np.sort(np.random.default_rng(1).choice(w["M"], size=rows, replace=False))
    t0 = time.perf_counter()
    oracle.mlp_sharded(d["X"], d["W1"], d["W2"], w["T"], w["act"], rows=sample)
    dt = time.perf_counter() - t0
    flops = 4.0 * rows * w["H"] * w["F"]
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": oracle.max_threads(),
            "kind": "oracle",
            "sample": f"{rows} of {w['M']} rows (seeded), sharded fp64 oracle, {dt:.2f} s; "
                      f"full M extrapolates to {dt * w['M'] / rows:.0f} s"}


def run_ours(args) -> dict | None:
    import numpy as np
    import torch

    import linear_sharding_gb300 as tp
    from synth import WORKLOADS, mlp_inputs

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist_init(world, "nccl")
    tp.load_library()

    peaks, peak_src = measured_peaks()
    if peak_src == "measured":
        # the AUTO planners weigh partial traffic with this box's measured rates
        tp.tp_set_machine_balance(peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9))

    w = WORKLOADS[WORKLOAD]
    M, H, F, T, act = w["M"], w["H"], w["F"], w["T"], w["act"]
    d = mlp_inputs(M=M, H=H, F=F, act=act, dtype="bf16", seed=rank)
    s = tp.tp_shard_weights(_dev(d["W1"], device), _dev(d["W2"], device), T, act)
    X = _dev(d["X"], device)
    Y = torch.empty((T, M, F // T), dtype=torch.bfloat16, device=device)
    Z = torch.empty((M, H), dtype=torch.float32, device=device)
    ws_col = tp.tp_colpar_workspace_bytes(s, M)
    ws_row = tp.tp_rowpar_workspace_bytes(s, M, args.variant)
    wcol = torch.empty(max(ws_col, 1), dtype=torch.uint8, device=device)
    wrow = torch.empty(max(ws_row, 1), dtype=torch.uint8, device=device)
    launches_per_step = 1 + 1 + (1 if ws_row > 0 else 0)
    stream = torch.cuda.current_stream()
    flops_step = 4.0 * M * H * F

    def step():
        tp.tp_colpar_forward(s, X, Y, workspace=wcol)
        tp.tp_rowpar_forward(s, Y, args.variant, Z, workspace=wrow)

    clocks = clock_sampler(physical_gpu_index(local))
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if tp.tp_last_device_status() != 0:
        raise RuntimeError("device status error during warm-up")

    # ---- headline: K back-to-back steps (burst), events at the two ends only ----
    K = args.steps
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(device)
    torch.cuda.synchronize()
    c0 = clocks.mark()
    start.record(stream)
    for _ in range(K):
        step()
    end.record(stream)
    torch.cuda.synchronize()
    c1 = clocks.mark()
    barrier(device)
    clk = clocks.window(c0, c1)
    status = tp.tp_last_device_status()
    if status != 0:
        raise RuntimeError(f"device status {status} in the timed region")
    elapsed = start.elapsed_time(end) / 1e3
    value, t_max = aggregate(elapsed, flops_step * K, device)

    # ---- the next K steps with each GEMM between events, for the roofline: an event recorded
    # between two kernels keeps the second from starting its set-up while the first finishes
    # (programmatic dependent launch), so these steps run a little slower than the headline's ----
    e0 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    e1 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    e2 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    barrier(device)
    torch.cuda.synchronize()
    for i in range(K):
        e0[i].record(stream)
        tp.tp_colpar_forward(s, X, Y, workspace=wcol)
        e1[i].record(stream)
        tp.tp_rowpar_forward(s, Y, args.variant, Z, workspace=wrow)
        e2[i].record(stream)
    torch.cuda.synchronize()
    barrier(device)
    if tp.tp_last_device_status() != 0:
        raise RuntimeError("device status error in the per-kernel timing")
    col_ms = sum(e0[i].elapsed_time(e1[i]) for i in range(K)) / K
    row_ms = sum(e1[i].elapsed_time(e2[i]) for i in range(K)) / K
    ev_value, ev_t = aggregate(e0[0].elapsed_time(e2[K - 1]) / 1e3, flops_step * K, device)

    # ---- the same steps with L2 flushed before each (a 256 MiB write) ----
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)
    f0 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    f1 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    barrier(device)
    torch.cuda.synchronize()
    for i in range(K):
        flush.zero_()
        f0[i].record(stream)
        step()
        f1[i].record(stream)
    torch.cuda.synchronize()
    flushed_each = sorted(f0[i].elapsed_time(f1[i]) for i in range(K))
    flushed_s = sum(flushed_each) / 1e3
    flushed_value, flushed_t = aggregate(flushed_s, flops_step * K, device)
    # the median step (the measurement plan's "median of >= 20" with the flush between reps),
    # the slowest rank's, with every rank's flop
    flushed_med_ms = (flushed_each[(K - 1) // 2] + flushed_each[K // 2]) / 2.0
    flushed_med_value, flushed_med_s = aggregate(flushed_med_ms / 1e3, flops_step, device)
    del flush

    # end to end through the public host-buffer call: pinned X in, Z out.  Two
    # requests in flight on two streams (each with its own host and device
    # buffers), so one step's copies run under the other's compute; every
    # step's own copies stay inside the timed region.
    n_inflight = 2
    Xh = [torch.from_numpy(np.ascontiguousarray(d["X"]).view(np.int16)).view(torch.bfloat16).pin_memory()
          for _ in range(n_inflight)]
    Zh = [torch.empty((M, H), dtype=torch.float32).pin_memory() for _ in range(n_inflight)]
    wsh = [torch.empty(tp.tp_mlp_host_workspace_bytes(s, M, args.variant), dtype=torch.uint8, device=device)
           for _ in range(n_inflight)]
    streams = [torch.cuda.Stream(device=device) for _ in range(n_inflight)]
    for k in range(args.warmup):
        i = k % n_inflight
        tp.tp_mlp_forward_host(s, Xh[i], Zh[i], wsh[i], args.variant, stream=streams[i])
    barrier(device)
    torch.cuda.synchronize()
    hs, he = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    hs.record(stream)
    for st_ in streams:
        st_.wait_event(hs)
    for k in range(K):
        i = k % n_inflight
        tp.tp_mlp_forward_host(s, Xh[i], Zh[i], wsh[i], args.variant, stream=streams[i])
    for st_ in streams:
        ev = torch.cuda.Event()
        ev.record(st_)
        stream.wait_event(ev)
    he.record(stream)
    torch.cuda.synchronize()
    barrier(device)
    if not torch.equal(Zh[0], Zh[1]) or not torch.isfinite(Zh[0]).all():
        raise RuntimeError("end-to-end results differ between the two in-flight buffers")
    e2e_value, _ = aggregate(hs.elapsed_time(he) / 1e3, flops_step * K, device)

    # ---- sustained: >= 1 s of back-to-back steps, against the sustained peak (last, so that
    # the burst legs above run on a GPU that has not yet reached its power cap) ----
    n_sus = max(K, int(math.ceil(args.sustain_s / max(elapsed / K, 1e-6)))) if args.sustain_s > 0 else 0
    ss0, ss1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(device)
    torch.cuda.synchronize()
    c2 = clocks.mark()
    ss0.record(stream)
    for _ in range(n_sus):
        step()
    ss1.record(stream)
    torch.cuda.synchronize()
    c3 = clocks.mark()
    barrier(device)
    sus_t_local = ss0.elapsed_time(ss1) / 1e3 if n_sus else 1.0
    sus_value, sus_t = aggregate(sus_t_local, flops_step * n_sus, device)
    clk_sus = clocks.window(c2, c3)

    clk_all = clocks.stop()

    # the sustained peak once the region is long or ran under the power cap (the default
    # 2000 steps reach it within their 0.6 s); the burst peak for a short burst
    sustained = elapsed > 1.0 or (elapsed > 0.1 and "sw_power_cap" in clk.get("reasons", []))
    peak = peaks["bf16_tflops_sustained" if sustained else "bf16_tflops"]
    achieved = 2.0 * M * H * F / (col_ms / 1e3) / 1e12
    traffic = profiled_traffic()
    line = {
        "metric": METRIC,
        "value": round(value / 1e12, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(t_max * 1e3 / K, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) X, N(0,1/fan_in) weights, bf16)",
        "config": {"workload": WORKLOAD, "M": M, "H": H, "F": F, "T": T, "act": "erf-gelu",
                   "variant": args.variant, "accumulate": "fp32", "output": "fp32",
                   "parallelism": f"{world} independent replica(s); T={T} shards per GPU",
                   "l2": "inputs larger than L2 (256 MiB of weights read per step); the same steps "
                         "with a 256 MiB L2 flush before each are reported as l2_flushed"},
        "pct_bf16_peak": round(100.0 * value / 1e12 / world / peak, 1),
        "roofline": {"kernel": "tp_gemm_pair_kernel<EPI_GELU_BF16> (column-parallel GEMM + GeLU, "
                               "CTA-pair 256x256 tiles)",
                     "bound": "tensor", "achieved": round(achieved, 1),
                     "peak": peak, "unit": "TFLOP/s", "frac": round(achieved / peak, 3),
                     "peak_source": f"{peak_src} ({'sustained' if sustained else 'burst'})",
                     "traffic": traffic, "avg_launch_ms": round(col_ms, 5)},
        "rowpar_ms": round(row_ms, 5),
        "with_kernel_events": {"value": round(ev_value / 1e12, 2), "unit": "TFLOP/s",
                               "ms_per_step": round(ev_t * 1e3 / K, 5), "steps": K,
                               "note": "the K steps after the headline, each GEMM between events "
                                       "(the roofline's per-kernel times); the events stop each "
                                       "kernel's set-up from overlapping the one before"},
        "l2_flushed": {"value": round(flushed_value / 1e12, 2), "unit": "TFLOP/s",
                       "ms_per_step": round(flushed_t * 1e3 / K, 5), "steps": K,
                       "median_ms_per_step": round(flushed_med_s * 1e3, 5),
                       "median_value": round(flushed_med_value / 1e12, 2),
                       "flush": "256 MiB write before every step, outside the step's events"},
        "sustained": {"value": round(sus_value / 1e12, 2), "unit": "TFLOP/s", "steps": n_sus,
                      "seconds": round(sus_t, 3), "peak": peaks["bf16_tflops_sustained"],
                      "frac": round(sus_value / 1e12 / world / peaks["bf16_tflops_sustained"], 3),
                      "peak_source": f"{peak_src} (sustained)", "clocks": clk_sus} if n_sus else None,
        "e2e": {"value": round(e2e_value / 1e12, 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": M * H * 2, "d2h_bytes_per_step": M * H * 4,
                "api": "tp_mlp_forward_host", "in_flight": n_inflight},
        "gpu_launches": launches_per_step * K,
        "clocks": clk,
        "clocks_whole_run": clk_all,
        "context": {"ring_allreduce_bytes_per_rank_if_T_gpus": tp.ring_allreduce_bytes(M * H, T, 4)},
    }
    if world == 1 and rank == 0:
        if args.extras != "none":
            line["extras"] = extras(args, tp, device, peaks)
        line["cpu_baseline"] = cpu_baseline(w, args.cpu_rows)
    s.close()
    return line if rank == 0 else None


def _time_calls(fn, reps: int, warm: int = 3) -> float:
    import torch
    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        fn()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / 1e3 / reps


def _auto_slots(ws_bytes: int, fixed_bytes: int, M: int, H: int) -> int:
    """Accumulation slots of the row-parallel GEMM behind a workspace size:
    the float32 partials take slots x M x H x 4 bytes beyond `fixed_bytes`
    (1 slot: one TMEM accumulator over all shards, no partials)."""
    extra = ws_bytes - fixed_bytes
    return max(1, int(round(extra / (M * H * 4)))) if extra > 0 else 1


def _r256(n: int) -> int:
    return (n + 255) // 256 * 256


def extras(args, tp, device, peaks) -> dict:
    """Secondary measurements (N = 1): the memory-bound decode shapes and the
    standalone shard-sum against HBM bandwidth; the training step; the
    attention projections and the large SwiGLU prefill with each all-reduce
    variant (float32 partials + shard-sum, one TMEM accumulator over all
    shards, and the planner's AUTO pick, named) against tensor peak; the
    attention core and one transformer block.  Inputs for these timing-only
    runs are drawn on the device with a seeded generator (same distributions
    as the parity workloads)."""
    import torch
    from synth import WORKLOADS
    out = {}
    hbm = peaks["hbm_gbs"]
    gen = torch.Generator(device=device)
    gen.manual_seed(0)

    def randn(shape, std, dtype=torch.bfloat16):
        return (torch.randn(shape, generator=gen, device=device) * std).to(dtype)

    w = WORKLOADS["decode_swiglu_h8192_f28672_t8"]
    H, F, T = w["H"], w["F"], w["T"]
    W1 = randn((H, 2 * F), 1 / math.sqrt(H))
    W2 = randn((F, H), 1 / math.sqrt(F))
    s = tp.tp_shard_weights(W1, W2, T, "swiglu")
    del W1, W2
    dec = {}
    for M in w["decode_m"]:
        X = randn((M, H), 1.0)
        Z = torch.empty((M, H), dtype=torch.float32, device=device)
        ws = torch.empty(max(tp.tp_mlp_workspace_bytes(s, M, "auto"), 1), dtype=torch.uint8, device=device)
        t = _time_calls(lambda: tp.tp_mlp_forward(s, X, "auto", Z, ws), 50)
        byts = 3 * H * F * 2 + M * H * (2 + 4)
        dec[f"M{M}"] = {"us": round(t * 1e6, 1), "GB/s": round(byts / t / 1e9, 1),
                        "frac_hbm": round(byts / t / 1e9 / hbm, 3)}
        # the same step captured once into a CUDA graph and replayed (a decode loop's form)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            tp.tp_mlp_forward(s, X, "auto", Z, ws)
        tg = _time_calls(graph.replay, 50)
        dec[f"M{M}"].update({"graph_us": round(tg * 1e6, 1), "graph_frac_hbm": round(byts / tg / 1e9 / hbm, 3)})
        del graph
    s.close()
    torch.cuda.empty_cache()
    out["decode_swiglu_h8192_f28672_t8"] = dec

    # training: forward that keeps its activations + backward, prefill GeLU workload
    w = WORKLOADS[WORKLOAD]
    M, H, F, T = w["M"], w["H"], w["F"], w["T"]
    W1, W2 = randn((H, F), 1 / math.sqrt(H)), randn((F, H), 1 / math.sqrt(F))
    s = tp.tp_shard_weights(W1, W2, T, "gelu")
    tp.tp_shards_enable_backward(s, W1, W2)
    del W1, W2
    X, dZ = randn((M, H), 1.0), randn((M, H), 1.0)
    _, Hs, Ps = tp.tp_mlp_forward_train(s, X)
    t_fwd = _time_calls(lambda: tp.tp_mlp_forward_train(s, X), 20)
    t_bwd = _time_calls(lambda: tp.tp_mlp_backward(s, X, Hs, Ps, dZ), 20)
    out["training_prefill_gelu_m2048_h4096_f16384_t4"] = {
        "forward_ms": round(t_fwd * 1e3, 4), "backward_ms": round(t_bwd * 1e3, 4),
        "forward_TFLOP/s": round(4 * M * H * F / t_fwd / 1e12, 1),
        "backward_TFLOP/s": round(8 * M * H * F / t_bwd / 1e12, 1),
        "step_TFLOP/s": round(12 * M * H * F / (t_fwd + t_bwd) / 1e12, 1),
        "note": "timed through the Python binding, output buffers allocated per call"}
    s.close()
    del X, dZ, Hs, Ps
    torch.cuda.empty_cache()

    ss = {}
    for name, T, n in (("prefill_gelu", 4, 2048 * 4096), ("attn_proj", 8, 4096 * 4096),
                       ("prefill_swiglu_large", 8, 8192 * 8192)):
        P = [torch.randn(n, generator=gen, device=device) for _ in range(T)]
        Zs = torch.empty(n, dtype=torch.float32, device=device)
        t = _time_calls(lambda: tp.tp_partial_sum(P, Zs), 20)
        byts = (T + 1) * n * 4
        ss[f"{name}_T{T}_n{n}"] = {"us": round(t * 1e6, 1), "GB/s": round(byts / t / 1e9, 1),
                                   "frac_hbm": round(byts / t / 1e9 / hbm, 3)}
        del P, Zs
        torch.cuda.empty_cache()
    out["shard_sum"] = ss
    out["hbm_peak_gbs"] = hbm
    burst = peaks["bf16_tflops"]

    w = WORKLOADS["attn_proj_m4096_h4096_32x128_t8"]
    M, H, T, nh, hd = w["M"], w["H"], w["T"], w["n_heads"], w["head_dim"]
    s = tp.tp_shard_weights_qkv(randn((H, 3 * H), 1 / math.sqrt(H)), randn((H, H), 1 / math.sqrt(H)),
                                nh, hd, T)
    X, A = randn((M, H), 1.0), randn((M, H), 1.0)
    QKV = torch.empty((T, M, 3 * H // T), dtype=torch.bfloat16, device=device)
    Z = torch.empty((M, H), dtype=torch.float32, device=device)
    res = {}
    variants = ("auto", "partials", "tmem_acc")
    wss = {v: torch.empty(max(tp.tp_attn_proj_workspace_bytes(s, M, v), 1), dtype=torch.uint8, device=device)
           for v in variants}
    # the variants take turns, three rounds, and each keeps its median: the GPU's clock under its
    # power cap drifts over a run, and this keeps that drift off any one variant
    tq, to = {v: [] for v in variants}, {v: [] for v in variants}
    for _ in range(3):
        for v in variants:
            tq[v].append(_time_calls(lambda: tp.tp_attn_proj_forward(s, X=X, variant=v, QKV=QKV), 10))
            to[v].append(_time_calls(lambda: tp.tp_attn_proj_forward(s, A=A, variant=v, Z=Z,
                                                                     workspace=wss[v]), 10))
    for v in variants:
        t_qkv, t_o = sorted(tq[v])[1], sorted(to[v])[1]
        res[v] = {"qkv_TFLOP/s": round(2 * M * H * 3 * H / t_qkv / 1e12, 1),
                  "oproj_TFLOP/s": round(2 * M * H * H / t_o / 1e12, 1),
                  "us_qkv": round(t_qkv * 1e6, 1), "us_oproj": round(t_o * 1e6, 1),
                  "oproj_frac_burst": round(2 * M * H * H / t_o / 1e12 / burst, 3)}
    res["auto_oproj_slots"] = _auto_slots(tp.tp_attn_proj_workspace_bytes(s, M, "auto"), 0, M, H)
    out["attn_proj_m4096_h4096_32x128_t8"] = res
    s.close()
    del wss, X, A, QKV, Z
    torch.cuda.empty_cache()

    # the block's fused causal attention core alone (4096 tokens, 32 heads of 128)
    M, nh, hd = 4096, 32, 128
    Qa, Ka, Va = (randn((nh, M, hd), 1.0) for _ in range(3))
    Oa = torch.empty((M, nh * hd), dtype=torch.bfloat16, device=device)
    wsa = torch.empty(tp.tp_attention_workspace_bytes(M, nh, hd), dtype=torch.uint8, device=device)
    # 200 calls (20 ms) after 20 untimed ones, so that the GPU's clock has settled after the
    # large GEMMs before it
    t = _time_calls(lambda: tp.tp_attention_forward(Qa, Ka, Va, True, Oa, wsa), 200, warm=20)
    fl = 2 * 2 * nh * hd * M * (M + 1) / 2
    out["attention_m4096_32x128_causal"] = {"us": round(t * 1e6, 1), "TFLOP/s": round(fl / t / 1e12, 1),
                                             "frac_burst": round(fl / t / 1e12 / burst, 3)}
    del Qa, Ka, Va, Oa, wsa

    # one transformer block at the attention workload's shape, SwiGLU MLP with F = 4H
    M, H, T, nh, hd = 4096, 4096, 8, 32, 128
    F = 4 * H
    a = tp.tp_shard_weights_qkv(randn((H, 3 * H), 1 / math.sqrt(H)), randn((H, H), 1 / math.sqrt(H)),
                                nh, hd, T)
    m = tp.tp_shard_weights(randn((H, 2 * F), 1 / math.sqrt(H)), randn((F, H), 1 / math.sqrt(F)), T,
                            "swiglu")
    X = randn((M, H), 1.0)
    ob = torch.empty((M, H), dtype=torch.float32, device=device)
    ws = torch.empty(tp.tp_block_workspace_bytes(a, m, M, "auto"), dtype=torch.uint8, device=device)
    t = _time_calls(lambda: tp.tp_block_forward(a, m, X, True, "auto", ob, None, ws), 10)
    # algorithmic flop: projections, causal attention (the half below the diagonal), MLP
    fl = 2 * M * H * 3 * H + 2 * 2 * nh * hd * M * (M + 1) / 2 + 2 * M * H * H + 6 * M * H * F
    out["block_m4096_h4096_32x128_t8_swiglu_f16384"] = {"ms": round(t * 1e3, 3),
                                                         "TFLOP/s": round(fl / t / 1e12, 1)}
    a.close()
    m.close()
    del ws, ob, X
    torch.cuda.empty_cache()

    w = WORKLOADS["prefill_swiglu_m8192_h8192_f28672_t8_outliers"]
    M, H, F, T = w["M"], w["H"], w["F"], w["T"]
    s = tp.tp_shard_weights(randn((H, 2 * F), 1 / math.sqrt(H)), randn((F, H), 1 / math.sqrt(F)), T,
                            "swiglu")
    X = randn((M, H), 1.0)
    Z = torch.empty((M, H), dtype=torch.float32, device=device)
    res = {}
    variants = ("auto", "partials", "tmem_acc")
    times = {v: [] for v in variants}
    for _ in range(3):  # variants take turns (see the attention projections above)
        for v in variants:
            ws = torch.empty(max(tp.tp_mlp_workspace_bytes(s, M, v), 1), dtype=torch.uint8, device=device)
            times[v].append(_time_calls(lambda: tp.tp_mlp_forward(s, X, v, Z, ws), 4, warm=2))
            del ws
    for v in variants:
        t = sorted(times[v])[1]
        res[v] = {"ms": round(t * 1e3, 3), "TFLOP/s": round(6 * M * H * F / t / 1e12, 1),
                  "frac_burst": round(6 * M * H * F / t / 1e12 / burst, 3)}
    res["auto_slots"] = _auto_slots(tp.tp_mlp_workspace_bytes(s, M, "auto"), _r256(M * F * 2), M, H)
    out["prefill_swiglu_m8192_h8192_f28672_t8"] = res
    s.close()
    torch.cuda.empty_cache()
    return out


# ---- reference arm: the oracle on the host cores ----------------------------------

def run_reference(args) -> dict | None:
    import numpy as np

    import oracle
    from synth import WORKLOADS, mlp_inputs
    world, rank, _ = dist_env()
    if rank != 0:
        return None
    oracle.build()
    w = WORKLOADS[WORKLOAD]
    M, H, F, T, act = w["M"], w["H"], w["F"], w["T"], w["act"]
    d = mlp_inputs(M=M, H=H, F=F, act=act, dtype="bf16", seed=0)
    rows_per_step = 16
    rng = np.random.default_rng(2)

    def step():
        rows = np.sort(rng.choice(M, size=rows_per_step, replace=False))
        oracle.mlp_sharded(d["X"], d["W1"], d["W2"], T, act, rows=rows)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    flops = 4.0 * rows_per_step * H * F * args.steps
    value = flops / dt / 1e12
    cores = oracle.max_threads()
    sample = f"{rows_per_step} seeded rows of {M} per step (sharded fp64 oracle)"
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3 / args.steps, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded, same inputs as the GPU arm)",
        "config": {"workload": WORKLOAD, "M": M, "H": H, "F": F, "T": T, "act": "erf-gelu",
                   "sample_rows_per_step": rows_per_step},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def run_case(args) -> dict:
    """One memory-bound case on its own (N = 1): the decode MLP or the
    standalone shard-sum, timed over --steps calls after --warmup calls."""
    import torch

    import linear_sharding_gb300 as tp
    from synth import WORKLOADS
    torch.cuda.set_device(0)
    device = torch.device("cuda", 0)
    tp.load_library()
    peaks, peak_src = measured_peaks()
    if peak_src == "measured":
        tp.tp_set_machine_balance(peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9))
    gen = torch.Generator(device=device)
    gen.manual_seed(0)

    def randn(shape, std, dtype=torch.bfloat16):
        return (torch.randn(shape, generator=gen, device=device) * std).to(dtype)

    if args.case == "decode":
        w = WORKLOADS["decode_swiglu_h8192_f28672_t8"]
        H, F, T, M = w["H"], w["F"], w["T"], args.decode_m
        s = tp.tp_shard_weights(randn((H, 2 * F), 1 / math.sqrt(H)), randn((F, H), 1 / math.sqrt(F)), T,
                                "swiglu")
        X = randn((M, H), 1.0)
        Z = torch.empty((M, H), dtype=torch.float32, device=device)
        ws = torch.empty(max(tp.tp_mlp_workspace_bytes(s, M, args.variant), 1), dtype=torch.uint8,
                         device=device)
        fn = lambda: tp.tp_mlp_forward(s, X, args.variant, Z, ws)  # noqa: E731
        byts = 3 * H * F * 2 + M * H * (2 + 4)
        cfg = {"workload": "decode_swiglu_h8192_f28672_t8", "M": M, "H": H, "F": F, "T": T,
               "variant": args.variant}
    elif args.case == "mlp":
        name = (WORKLOAD if args.mlp_workload == "prefill_gelu"
                else "prefill_swiglu_m8192_h8192_f28672_t8_outliers")
        w = WORKLOADS[name]
        M, H, F, T, act = w["M"], w["H"], w["F"], w["T"], w["act"]
        ncols = 2 * F if act == "swiglu" else F
        s = tp.tp_shard_weights(randn((H, ncols), 1 / math.sqrt(H)), randn((F, H), 1 / math.sqrt(F)), T, act)
        X = randn((M, H), 1.0)
        Z = torch.empty((M, H), dtype=torch.float32, device=device)
        ws = torch.empty(max(tp.tp_mlp_workspace_bytes(s, M, args.variant), 1), dtype=torch.uint8,
                         device=device)
        fn = lambda: tp.tp_mlp_forward(s, X, args.variant, Z, ws)  # noqa: E731
        t = _time_calls(fn, args.steps, warm=args.warmup)
        if tp.tp_last_device_status() != 0:
            raise RuntimeError("device status error")
        fl = (6 if act == "swiglu" else 4) * M * H * F
        return {"metric": "MLP forward TFLOP/s", "value": round(fl / t / 1e12, 1), "unit": "TFLOP/s",
                "ms_per_call": round(t * 1e3, 4), "steps": args.steps, "warmup": args.warmup,
                "config": {"workload": name, "variant": args.variant}}
    elif args.case == "oproj":
        w = WORKLOADS["attn_proj_m4096_h4096_32x128_t8"]
        M, H, T, nh, hd = w["M"], w["H"], w["T"], w["n_heads"], w["head_dim"]
        s = tp.tp_shard_weights_qkv(randn((H, 3 * H), 1 / math.sqrt(H)), randn((H, H), 1 / math.sqrt(H)),
                                    nh, hd, T)
        A = randn((M, H), 1.0)
        Z = torch.empty((M, H), dtype=torch.float32, device=device)
        ws = torch.empty(max(tp.tp_attn_proj_workspace_bytes(s, M, args.variant), 1), dtype=torch.uint8,
                         device=device)
        fn = lambda: tp.tp_attn_proj_forward(s, A=A, variant=args.variant, Z=Z, workspace=ws)  # noqa: E731
        t = _time_calls(fn, args.steps, warm=args.warmup)
        if tp.tp_last_device_status() != 0:
            raise RuntimeError("device status error")
        return {"metric": "O-projection TFLOP/s", "value": round(2 * M * H * H / t / 1e12, 1),
                "unit": "TFLOP/s", "us_per_call": round(t * 1e6, 2), "steps": args.steps,
                "warmup": args.warmup,
                "config": {"workload": "attn_proj_m4096_h4096_32x128_t8 (O-projection)",
                           "variant": args.variant}}
    elif args.case == "train":
        w = WORKLOADS[WORKLOAD]
        M, H, F, T = w["M"], w["H"], w["F"], w["T"]
        W1, W2 = randn((H, F), 1 / math.sqrt(H)), randn((F, H), 1 / math.sqrt(F))
        s = tp.tp_shard_weights(W1, W2, T, "gelu")
        tp.tp_shards_enable_backward(s, W1, W2)
        X, dZ = randn((M, H), 1.0), randn((M, H), 1.0)
        _, Hs, Ps = tp.tp_mlp_forward_train(s, X)
        fn = lambda: tp.tp_mlp_backward(s, X, Hs, Ps, dZ)  # noqa: E731
        t = _time_calls(fn, args.steps, warm=args.warmup)
        return {"metric": "backward TFLOP/s", "value": round(8 * M * H * F / t / 1e12, 1),
                "unit": "TFLOP/s", "ms_per_call": round(t * 1e3, 4), "steps": args.steps,
                "warmup": args.warmup, "config": {"workload": WORKLOAD, "M": M, "H": H, "F": F, "T": T}}
    elif args.case == "block":
        M, H, T, nh, hd = 4096, 4096, 8, 32, 128
        F = 4 * H
        a = tp.tp_shard_weights_qkv(randn((H, 3 * H), 1 / math.sqrt(H)), randn((H, H), 1 / math.sqrt(H)),
                                    nh, hd, T)
        m = tp.tp_shard_weights(randn((H, 2 * F), 1 / math.sqrt(H)), randn((F, H), 1 / math.sqrt(F)), T,
                                "swiglu")
        X = randn((M, H), 1.0)
        ob = torch.empty((M, H), dtype=torch.float32, device=device)
        ws = torch.empty(tp.tp_block_workspace_bytes(a, m, M, args.variant), dtype=torch.uint8, device=device)
        fn = lambda: tp.tp_block_forward(a, m, X, True, args.variant, ob, None, ws)  # noqa: E731
        t = _time_calls(fn, args.steps, warm=args.warmup)
        fl = 2 * M * H * 3 * H + 2 * 2 * nh * hd * M * (M + 1) / 2 + 2 * M * H * H + 6 * M * H * F
        return {"metric": "transformer block TFLOP/s", "value": round(fl / t / 1e12, 1), "unit": "TFLOP/s",
                "ms_per_call": round(t * 1e3, 4), "steps": args.steps, "warmup": args.warmup,
                "config": {"workload": "block_m4096_h4096_32x128_t8_swiglu_f16384_causal"}}
    elif args.case == "attention":
        M, nh, hd = 4096, 32, 128
        Q, K, V = (randn((nh, M, hd), 1.0) for _ in range(3))
        O = torch.empty((M, nh * hd), dtype=torch.bfloat16, device=device)
        ws = torch.empty(tp.tp_attention_workspace_bytes(M, nh, hd), dtype=torch.uint8, device=device)
        fn = lambda: tp.tp_attention_forward(Q, K, V, True, O, ws)  # noqa: E731
        t = _time_calls(fn, args.steps, warm=args.warmup)
        if tp.tp_last_device_status() != 0:
            raise RuntimeError("device status error")
        fl = 2 * 2 * nh * hd * M * (M + 1) / 2  # Q K^T and P V over the allowed (causal) pairs
        return {"metric": "attention TFLOP/s", "value": round(fl / t / 1e12, 1), "unit": "TFLOP/s",
                "ms_per_call": round(t * 1e3, 4), "steps": args.steps, "warmup": args.warmup,
                "config": {"workload": "attention_m4096_32x128_causal"}}
    else:
        T, n = 8, 8192 * 8192
        P = [torch.randn(n, generator=gen, device=device) for _ in range(T)]
        Z = torch.empty(n, dtype=torch.float32, device=device)
        fn = lambda: tp.tp_partial_sum(P, Z)  # noqa: E731
        byts = (T + 1) * n * 4
        cfg = {"workload": "shard_sum_t8_n67108864", "T": T, "n": n}
    t = _time_calls(fn, args.steps, warm=args.warmup)
    if tp.tp_last_device_status() != 0:
        raise RuntimeError("device status error")
    gbs = byts / t / 1e9
    return {"metric": f"{args.case} HBM GB/s", "value": round(gbs, 1), "unit": "GB/s",
            "us_per_call": round(t * 1e6, 2), "frac_hbm": round(gbs / peaks["hbm_gbs"], 3),
            "peak_source": peak_src, "steps": args.steps, "warmup": args.warmup, "config": cfg,
            "algorithmic_bytes": byts, "l2": "inputs larger than L2"}


def main(argv=None):
    args = parse_args(argv)
    if args.steps < 1 or args.warmup < 0:
        raise SystemExit("--steps >= 1 and --warmup >= 0")
    if args.case != "prefill" and args.impl == "ours":
        print(json.dumps(run_case(args)), flush=True)
        return
    line = run_reference(args) if args.impl == "reference" else run_ours(args)
    if line is not None:
        print(json.dumps(line), flush=True)
    try:
        import torch.distributed as dist
        if dist.is_available() and dist.is_initialized():
            dist.destroy_process_group()
    except Exception:
        pass


if __name__ == "__main__":
    main()
