#!/usr/bin/env python
"""Benchmark of the fused attention hot path: one step = forward + backward of
the workload (default: B=4, H=16, N=8192, d=128, non-causal, bf16), inputs
resident in HBM, timed with CUDA events.  Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload headline|causal|gqa|varlen|fp8|sweep-d<64|128|256>-n<1024|4096|16384>[-causal]]

--impl reference times the fp64 CPU oracle (a deliberately slow, plain
statement of the same computation) on the host cores: each step is the forward
and backward of one (batch, head) slice of the same workload.

Multi-GPU (torchrun, one rank per GPU): every rank runs its own independent
copy of the workload (attention heads shard with no exchange), so scaling is
weak and `value` is the total over ranks divided by the slowest rank's time.
"""
from __future__ import annotations

import argparse
import csv
import datetime
import hashlib
import io
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attention TFLOPs/s fwd & bwd (bf16, d=128) at 1 GB300; fraction of 2.25 PF BF16 peak"
NOMINAL_BF16_TFLOPS = 2250.0


def sweep_name(d: int, N: int, causal: bool) -> str:
    return f"sweep-d{d}-n{N}" + ("-causal" if causal else "")


SWEEP_NAMES = [sweep_name(d, N, c) for d in (64, 128, 256) for N in (1024, 4096, 16384) for c in (False, True)]


def workload(name: str):
    from exact_attention_blackwell_gb300 import inputs

    if name.startswith("sweep-"):  # one point of the head-dim sweep (B*N = 32768 tokens, H = 16)
        return {sweep_name(w.d, w.N, w.causal): w for w in inputs.sweep()}[name]
    return {"headline": inputs.headline, "causal": inputs.causal_outliers, "gqa": inputs.long_gqa,
            "varlen": inputs.packed_causal}[name]()


def env_int(k, default):
    try:
        return int(os.environ.get(k, default))
    except ValueError:
        return default


# ------------------------------------------------------------------ clocks
class NvmlClockSampler:
    """In-process, read-only NVML sampling of the SM clock and clock-event
    reasons, every 4 ms on a background thread (the driver's libnvidia-ml is
    called through ctypes; nothing is set).  Only samples whose host time falls
    inside the timed window (mark()) are summarised, so even a 0.1 s timed
    region has its own record."""

    PERIOD_S = 0.004
    NVML_CLOCK_SM = 1
    # clock-event reason bits (nvml.h)
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}

    def __init__(self, gpu_index: int):
        import ctypes
        import threading

        self._ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit_v2 failed")
        self.handle = ctypes.c_void_p()
        if self.lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(gpu_index), ctypes.byref(self.handle)) != 0:
            raise OSError("nvmlDeviceGetHandleByIndex_v2 failed")
        self._reasons_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(self.lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
        self.samples = []
        self.window = None
        self._stop = threading.Event()
        self._thread = threading.Thread(target=self._run, daemon=True)
        u = ctypes.c_uint()
        self.max_mhz = float(u.value) if self.lib.nvmlDeviceGetMaxClockInfo(
            self.handle, ctypes.c_int(self.NVML_CLOCK_SM), ctypes.byref(u)) == 0 else None

    def _read(self):
        ct = self._ct
        clk, rs = ct.c_uint(), ct.c_ulonglong()
        if self.lib.nvmlDeviceGetClockInfo(self.handle, ct.c_int(self.NVML_CLOCK_SM), ct.byref(clk)) != 0:
            return None
        reasons = rs.value if self._reasons_fn(self.handle, ct.byref(rs)) == 0 else 0
        return time.time(), float(clk.value), reasons

    def _run(self):
        while not self._stop.is_set():
            s = self._read()
            if s is not None:
                self.samples.append(s)
            time.sleep(self.PERIOD_S)

    def start(self):
        self._thread.start()

    def mark(self, t0: float, t1: float):
        """Host wall-clock bounds (time.time()) of the timed region."""
        self.window = (t0, t1)

    def stop(self):
        self._stop.set()
        self._thread.join(timeout=2)
        inside = [s for s in self.samples if self.window and self.window[0] <= s[0] <= self.window[1]]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["no samples inside the timed region"],
                    "source": "NVML in-process"}
        sm = [s[1] for s in inside]
        reasons = sorted({name for s in inside for bit, name in self.REASONS.items() if s[2] & bit})
        return {"sm_mhz": statistics.median(sm), "sm_min_mhz": min(sm), "sm_max_mhz": self.max_mhz,
                "samples": len(sm), "window": "timed region", "reasons": reasons,
                "source": f"NVML in-process, every {self.PERIOD_S * 1e3:.0f} ms"}


class SmiClockSampler:
    """nvidia-smi sampling of SM clock, power and throttle reasons (used when
    the NVML library cannot be loaded).

    Sampling starts before the warm-up (nvidia-smi takes a moment to start);
    only the readings whose timestamps fall inside the timed window count.
    """

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.window = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None

    def mark(self, t0: float, t1: float):
        """Host wall-clock bounds (time.time()) of the timed region."""
        self.window = (t0, t1)

    @staticmethod
    def _stamp(text: str):
        try:
            return datetime.datetime.strptime(text.strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
        except ValueError:
            return None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for row in csv.reader(io.StringIO(out)):
            if len(row) < 10:
                continue
            try:
                rows.append((self._stamp(row[0]), float(row[2]), float(row[3]), float(row[4]), row[6:10]))
            except ValueError:
                continue
        inside = [r for r in rows if self.window and r[0] is not None and self.window[0] <= r[0] <= self.window[1]]
        used = inside if len(inside) >= 3 else rows
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for _, c, cmax, pw, flags in used:
            sm.append(c)
            smax.append(cmax)
            power.append(pw)
            for n, v in zip(names, flags):
                if v.strip().lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "power_w_max": max(power),
                "power_w_median": statistics.median(power), "samples": len(sm), "source": "nvidia-smi -lms 50",
                "window": "timed region" if used is inside else "whole run (too few samples inside the timed region)",
                "reasons": sorted(reasons)}


def ClockSampler(gpu_index: int):
    """NVML in-process sampler where the driver library loads, else nvidia-smi."""
    try:
        return NvmlClockSampler(gpu_index)
    except (OSError, AttributeError):
        return SmiClockSampler(gpu_index)


# ------------------------------------------------------------------ peaks and profiles
# The roofline's denominator: each timed region lasts well under a second and
# its SM clock stays near the maximum, the conditions of the burst GEMM figure;
# the sustained figure (seconds of back-to-back GEMMs at the 1.4 kW cap, SM
# clock ~1450 MHz) is reported beside it as frac_of_sustained.
PEAK_NOTE = "cuBLAS bf16 burst (timed region under a second, SM clock near max)"


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            j = json.load(f)
        return {"sustained": float(j["bf16_tflops_sustained"]), "burst": float(j["bf16_tflops"]),
                "hbm_gbs": float(j["hbm_gbs"]), "source": "measured (MEASURED_PEAKS.json)"}
    except (OSError, KeyError, ValueError):
        return {"sustained": 1700.0, "burst": 1900.0, "hbm_gbs": 6800.0, "source": "fallback (no measured file)"}


def kernel_source_hash(files) -> str:
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "exact_attention_blackwell_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(summary: str, src_hash: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", summary)
    try:
        text = open(path).read()
    except OSError:
        return None
    m_b = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    m_h = re.search(r"source_sha:\s*([0-9a-f]+)", text)
    if not m_b or not m_h or m_h.group(1) != src_hash:
        return None
    return float(m_b.group(1))


def oracle_tiny_one_thread() -> float:
    """Seconds of one fwd + bwd of the tiny case (B1 H2 N128 d64) by the oracle on one thread."""
    import oracle
    from exact_attention_blackwell_gb300 import inputs

    w = inputs.tiny()
    x = inputs.make_inputs(w)
    all_threads = oracle.num_threads()
    oracle.set_threads(1)
    try:
        t0 = time.perf_counter()
        oracle.attention_fwd(x["q"], x["k"], x["v"], w.sm_scale, w.causal)
        oracle.attention_bwd(x["q"], x["k"], x["v"], x["dO"], w.sm_scale, w.causal)
        return time.perf_counter() - t0
    finally:
        oracle.set_threads(all_threads)


# ------------------------------------------------------------------ reference arm (CPU oracle)
def cpu_oracle_step(x, w, head: int):
    """fwd + bwd of one (b, h) slice with the fp64 oracle; returns seconds."""
    import oracle

    b, h = divmod(head % (w.B * w.H), w.H)
    kh = h // (w.H // w.Hkv)
    q = x["q"][b:b + 1, :, h:h + 1]
    k = x["k"][b:b + 1, :, kh:kh + 1]
    v = x["v"][b:b + 1, :, kh:kh + 1]
    dO = x["dO"][b:b + 1, :, h:h + 1] if x["dO"] is not None else None
    t0 = time.perf_counter()
    oracle.attention_fwd(q, k, v, w.sm_scale, w.causal)
    if w.backward:
        oracle.attention_bwd(q, k, v, dO, w.sm_scale, w.causal)
    return time.perf_counter() - t0


def head_flops(w) -> float:
    f = 4.0 * w.N * w.N * w.d / (2 if w.causal else 1)
    return f * (3.5 if w.backward else 1.0)


def run_reference(args):
    import oracle
    from exact_attention_blackwell_gb300 import inputs

    rank = env_int("RANK", 0)
    if rank != 0:
        return 0
    oracle.build()
    w = workload(args.workload)
    if args.workload == "varlen":
        return run_reference_varlen(args, w)
    x = inputs.make_inputs(w, with_dO=w.backward)
    for s in range(args.warmup):
        cpu_oracle_step(x, w, s)
    t = 0.0
    for s in range(args.steps):
        t += cpu_oracle_step(x, w, args.warmup + s)
    value = head_flops(w) * args.steps / t / 1e12
    cores = oracle.num_threads()
    sample = f"one (batch, head) slice per step ({w.N} query rows x {w.N} keys, d={w.d}), fwd+bwd, fp64"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(w),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_reference_varlen(args, w):
    """Oracle arm of the packed workload: each step is the shortest sequence's fwd+bwd (all heads)."""
    import oracle
    from exact_attention_blackwell_gb300 import inputs

    x = inputs.make_packed_inputs(w)
    n = min(w.lens)
    a = w.cu_seqlens()[list(w.lens).index(n)]
    sl = lambda t: t[None, a:a + n]
    t = 0.0
    for s in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        oracle.attention_fwd(sl(x["q"]), sl(x["k"]), sl(x["v"]), w.sm_scale, w.causal)
        oracle.attention_bwd(sl(x["q"]), sl(x["k"]), sl(x["v"]), sl(x["dO"]), w.sm_scale, w.causal)
        if s >= args.warmup:
            t += time.perf_counter() - t0
    f = 3.5 * 4.0 * w.H * n * n * w.d / 2
    value = f * args.steps / t / 1e12
    sample = f"the shortest sequence ({n} rows, all {w.H} heads) per step, fwd+bwd, fp64"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name + " fwd+bwd", "B": w.B, "total": w.total, "max_seqlen": w.max_seqlen},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}), flush=True)
    return 0


def config_of(w):
    return {"workload": w.name + (" fwd+bwd" if w.backward else " fwd"), "B": w.B, "H": w.H, "Hkv": w.Hkv,
            "N": w.N, "d": w.d, "causal": w.causal,
            "l2": "inputs larger than L2 (no flush between steps)", "parallelism": "independent heads per GPU"}


# ------------------------------------------------------------------ our arm
def run_ours(args):
    import torch

    import exact_attention_blackwell_gb300 as fa
    from exact_attention_blackwell_gb300 import inputs, sharding

    world = env_int("WORLD_SIZE", 1)
    rank = env_int("RANK", 0)
    local = env_int("LOCAL_RANK", 0)
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    fa.lib()  # fails loudly if the CUDA library is missing

    w = workload(args.workload)
    if args.batch:
        w = inputs.Workload(w.name.replace(f"B{w.B}", f"B{args.batch}"), args.batch, w.H, w.Hkv, w.N, w.d, w.causal,
                            w.seed, w.outliers, w.backward)
    B, H, Hkv, N, d = w.B, w.H, w.Hkv, w.N, w.d
    scale, causal = w.sm_scale, w.causal
    xw = inputs.Workload(w.name, B, H, Hkv, N, d, causal, sharding.rank_seed(w.seed, rank), w.outliers, w.backward)
    x_cpu = inputs.make_inputs(xw, with_dO=w.backward)
    dev = torch.device("cuda", local)
    q, k, v = (x_cpu[n].to(dev) for n in ("q", "k", "v"))
    dO = x_cpu["dO"].to(dev) if w.backward else None
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    if w.backward:
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        ws_bytes = fa.fa_bwd_workspace_bytes(B, H, Hkv, N, d)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    sptr = stream.cuda_stream

    def check(st, what):
        if st != fa.FA_OK:
            raise fa.FaError(st, what)

    ev = lambda: torch.cuda.Event(enable_timing=True)
    fwd_ev, dkdv_ev, dq_ev = [], [], []

    def timed(events, record, fn):
        if not record:
            return fn()
        e0, e1 = ev(), ev()
        e0.record(stream)
        r = fn()
        e1.record(stream)
        events.append((e0, e1))
        return r

    def step(record=False):
        check(timed(fwd_ev, record, lambda: fa.fa_fwd(q, k, v, o, lse, B, H, Hkv, N, d, scale, causal, sptr)),
              "fa_fwd")
        if not w.backward:
            return
        check(fa.fa_bwd_prepare(o, lse, dO, B, H, Hkv, N, d, ws, ws_bytes, sptr), "fa_bwd_prepare")
        check(timed(dkdv_ev, record, lambda: fa.fa_bwd_dkdv(q, k, v, dO, dk, dv, B, H, Hkv, N, d, scale, causal, ws,
                                                            ws_bytes, sptr)), "fa_bwd_dkdv")
        check(timed(dq_ev, record, lambda: fa.fa_bwd_dq(q, k, v, dO, dq, B, H, Hkv, N, d, scale, causal, ws,
                                                        ws_bytes, sptr)), "fa_bwd_dq")

    launches_per_step = 4 if w.backward else 1
    sampler = ClockSampler(local)
    sampler.start()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if fa.fa_last_device_status(sptr) != fa.FA_OK:
        raise RuntimeError("device status reports a timed-out wait during warm-up")
    if dist:
        dist.barrier()
    torch.cuda.synchronize()

    t_start, t_end = ev(), ev()
    wall0 = time.time()
    t_start.record(stream)
    for _ in range(args.steps):
        step(record=True)
    t_end.record(stream)
    torch.cuda.synchronize()
    sampler.mark(wall0, time.time())
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    clocks = sampler.stop()
    total_ms = sharding.max_over_ranks(t_start.elapsed_time(t_end), dist, dev)
    if fa.fa_last_device_status(sptr) != fa.FA_OK:
        raise RuntimeError("device status reports a timed-out wait")
    if not torch.isfinite(o).all() or (w.backward and not torch.isfinite(dq.float()).all()):
        raise RuntimeError("non-finite outputs")

    fwd_f = w.fwd_flops()
    bwd_f = w.bwd_flops() if w.backward else 0.0
    step_f = fwd_f + bwd_f
    ms_step = total_ms / args.steps
    value = sharding.whole_job_tflops(step_f, args.steps, total_ms, world)
    fwd_ms = statistics.mean(a.elapsed_time(b) for a, b in fwd_ev)
    peaks = measured_peaks()
    out = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) rounded to bf16)",
           "config": dict(config_of(w), input_sha256=inputs.input_sha256(x_cpu)[:16]),
           "frac_of_2250_tflops": value / world / NOMINAL_BF16_TFLOPS,
           "fwd_tflops": fwd_f / (fwd_ms * 1e-3) / 1e12, "fwd_ms": fwd_ms}
    # the metric's own flop counts (backward = 2.5 x forward) against the measured burst peak:
    # unlike roofline.frac (executed flops of one kernel) these charge the recomputed GEMMs
    out["fwd_frac_of_burst"] = out["fwd_tflops"] / peaks["burst"]
    if w.backward:
        dkdv_ms = statistics.mean(a.elapsed_time(b) for a, b in dkdv_ev)
        dq_ms = statistics.mean(a.elapsed_time(b) for a, b in dq_ev)
        out["bwd_ms"] = ms_step - fwd_ms
        out["bwd_tflops"] = bwd_f / ((ms_step - fwd_ms) * 1e-3) / 1e12
        out["bwd_frac_of_burst"] = out["bwd_tflops"] / peaks["burst"]
        out["dkdv_ms"], out["dq_ms"] = dkdv_ms, dq_ms
        # executed GEMM flops of each backward kernel: dK/dV recomputes S^T and dP^T
        # (4 GEMMs of 2 N^2 d per head), dQ recomputes S and dP (3 GEMMs)
        gemm = fwd_f / 2  # one N x N x d GEMM pass over all heads, causal halving included
        # head dim 256 runs on CTA pairs; head dim 128 too for sequences longer than
        # 2048 rows (4096 causal: FA_DKDV_PAIR_MIN_N[_CAUSAL] in fa_bwd.cu)
        pair128 = d == 128 and N > (4096 if causal else 2048)
        dkdv_name = "bwd_dkdv256_pair_kernel" if d == 256 else "bwd_dkdv_pair_kernel" if pair128 else "bwd_dkdv_kernel"
        dq_name = "bwd_dq256_pair_kernel" if d == 256 else "bwd_dq_kernel"
        kern = (dkdv_name, dkdv_ms, 4 * gemm, "fa_bwd.cu") if dkdv_ms >= dq_ms else \
            (dq_name, dq_ms, 3 * gemm, "fa_bwd.cu")
        name, kms, kflops, _ = kern
        src = kernel_source_hash(["fa_bwd.cu", "ptx.cuh", "exp2_poly.cuh", "fa_internal.h"])
        achieved = kflops / (kms * 1e-3) / 1e12
        out["roofline"] = {
            "bound": "tensor", "kernel": name, "achieved": achieved,
            "peak": peaks["burst"], "unit": "TFLOP/s", "frac": achieved / peaks["burst"],
            "frac_of_sustained": achieved / peaks["sustained"],
            "peak_source": peaks["source"] + ", " + PEAK_NOTE,
            "flops_per_launch": kflops, "launch_ms": kms,
            # the committed figures are per launch of the workload's own size
            "traffic": None if args.batch else profiled_traffic(f"{name}_{args.workload}.md", src),
        }
    else:
        src = kernel_source_hash(["fa_fwd.cu", "ptx.cuh", "exp2_poly.cuh", "fa_internal.h"])
        achieved = fwd_f / (fwd_ms * 1e-3) / 1e12
        out["roofline"] = {
            "bound": "tensor", "kernel": "fa_fwd_kernel", "achieved": achieved, "peak": peaks["burst"],
            "unit": "TFLOP/s", "frac": achieved / peaks["burst"], "frac_of_sustained": achieved / peaks["sustained"],
            "peak_source": peaks["source"] + ", " + PEAK_NOTE,
            "flops_per_launch": fwd_f, "launch_ms": fwd_ms,
            "traffic": None if args.batch else profiled_traffic(f"fa_fwd_kernel_{args.workload}.md", src),
        }
    out["gpu_launches"] = launches_per_step * args.steps
    out["clocks"] = clocks

    # ---- end to end through the C ABI with host buffers: H2D inputs, D2H outputs every step
    if args.no_e2e:
        if rank == 0:
            print(json.dumps(out), flush=True)
        if dist:
            dist.destroy_process_group()
        return 0
    # Pipelined over three streams, as a caller feeding a stream of batches would
    # run it: step i's uploads (stream s_in) overlap step i-1's kernels (s_cmp)
    # and step i-2's downloads (s_out); two device buffer sets alternate.  Every
    # step still moves its full inputs host -> device and outputs device -> host.
    names = ("q", "k", "v") + (("dO",) if w.backward else ())
    pin = {n: x_cpu[n].pin_memory() for n in names}
    first_in = {"q": q, "k": k, "v": v, "dO": dO}
    first_out = [o, lse] + ([dq, dk, dv] if w.backward else [])
    sets = [({n: first_in[n] for n in names}, first_out),
            ({n: torch.empty_like(first_in[n]) for n in names}, [torch.empty_like(t) for t in first_out])]
    outs_h = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in first_out]
    s_in, s_cmp, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def kernels(ins, outs, sp):
        check(fa.fa_fwd(ins["q"], ins["k"], ins["v"], outs[0], outs[1], B, H, Hkv, N, d, scale, causal, sp), "fa_fwd")
        if w.backward:
            check(fa.fa_bwd_prepare(outs[0], outs[1], ins["dO"], B, H, Hkv, N, d, ws, ws_bytes, sp), "fa_bwd_prepare")
            check(fa.fa_bwd_dkdv(ins["q"], ins["k"], ins["v"], ins["dO"], outs[3], outs[4], B, H, Hkv, N, d, scale,
                                 causal, ws, ws_bytes, sp), "fa_bwd_dkdv")
            check(fa.fa_bwd_dq(ins["q"], ins["k"], ins["v"], ins["dO"], outs[2], B, H, Hkv, N, d, scale, causal, ws,
                               ws_bytes, sp), "fa_bwd_dq")

    def pipeline(n_steps, e_start=None, e_end=None):
        in_done, cmp_done, out_done = [], [], []
        if e_start is not None:
            e_start.record(s_in)
        for i in range(n_steps):
            ins, outs = sets[i % 2]
            if i >= 2:
                s_in.wait_event(cmp_done[i - 2])  # step i-2 has finished reading this input set
            with torch.cuda.stream(s_in):
                for n in names:
                    ins[n].copy_(pin[n], non_blocking=True)
            in_done.append(torch.cuda.Event())
            in_done[-1].record(s_in)
            s_cmp.wait_event(in_done[i])
            if i >= 2:
                s_cmp.wait_event(out_done[i - 2])  # step i-2's outputs in this set are on the host
            kernels(ins, outs, s_cmp.cuda_stream)
            cmp_done.append(torch.cuda.Event())
            cmp_done[-1].record(s_cmp)
            s_out.wait_event(cmp_done[i])
            with torch.cuda.stream(s_out):
                for hd, dd in zip(outs_h, outs):
                    hd.copy_(dd, non_blocking=True)
            out_done.append(torch.cuda.Event())
            out_done[-1].record(s_out)
        if e_end is not None:
            for e in out_done + cmp_done:
                s_out.wait_event(e)
            e_end.record(s_out)

    e2e_steps = max(3, args.steps // 2)
    torch.cuda.synchronize()
    pipeline(3)
    torch.cuda.synchronize()
    e0, e1 = ev(), ev()
    pipeline(e2e_steps, e0, e1)
    torch.cuda.synchronize()
    if fa.fa_last_device_status(sptr) != fa.FA_OK:
        raise RuntimeError("device status reports a timed-out wait (end-to-end leg)")
    e2e_ms = sharding.max_over_ranks(e0.elapsed_time(e1), dist, dev)
    out["e2e"] = {"value": sharding.whole_job_tflops(step_f, e2e_steps, e2e_ms, world), "unit": "TFLOP/s",
                  "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in pin.values()),
                  "d2h_bytes_per_step": sum(t.numel() * t.element_size() for t in outs_h),
                  "ms_per_step": e2e_ms / e2e_steps,
                  "schedule": "three streams: uploads of step i, kernels of step i-1, downloads of step i-2 overlap; "
                              "two device buffer sets"}
    if not torch.equal(outs_h[0], first_out[0].cpu()) and not torch.equal(outs_h[0], sets[1][1][0].cpu()):
        raise RuntimeError("end-to-end output differs from the device result")

    # ---- CPU oracle on the host cores (rank 0, single GPU only), a bounded sample
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle

        oracle.build()
        t = cpu_oracle_step(x_cpu, w, 0)
        tiny_1t = oracle_tiny_one_thread()
        out["cpu_baseline"] = {"value": head_flops(w) / t / 1e12, "unit": "TFLOP/s", "cores": oracle.num_threads(),
                               "tiny_one_thread_seconds": tiny_1t,
                               "kind": "oracle", "seconds": t,
                               "sample": f"(batch 0, head 0) slice: {N} query rows x {N} keys, d={d}, "
                                         f"{'fwd+bwd' if w.backward else 'fwd'}, fp64",
                               # every (batch, head) slice costs the same: B * H slices make the whole step
                               "full_problem_seconds_extrapolated": t * B * H,
                               "extrapolation": f"measured slice time x {B * H} (batch, head) slices; not measured"}
    if rank == 0:
        print(json.dumps(out), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


# ------------------------------------------------------------------ one problem split over the ranks
def run_sharded(args):
    """--shard: one problem of the workload split over the ranks by (batch, kv head)
    groups, GQA groups whole, no data-path collective (strong scaling: the total work
    is fixed as the rank count grows).  Each rank solves its pieces with the same
    entry points as the default run."""
    import torch

    import exact_attention_blackwell_gb300 as fa
    from exact_attention_blackwell_gb300 import inputs, sharding

    world, rank, local = env_int("WORLD_SIZE", 1), env_int("RANK", 0), env_int("LOCAL_RANK", 0)
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    fa.lib()
    w = workload(args.workload)
    g = w.H // w.Hkv
    x = inputs.make_inputs(w, with_dO=w.backward)  # the same problem on every rank
    dev = torch.device("cuda", local)
    pieces = []
    for pc in sharding.head_pieces(w.B, w.Hkv, world, rank):
        b0, b1, kh0, kh1 = pc
        t = {n: sharding.slice_piece(x[n], pc, g).to(dev) for n in (("q", "dO") if w.backward else ("q",))}
        t.update({n: sharding.slice_piece(x[n], pc).to(dev) for n in ("k", "v")})
        B, H, Hkv = b1 - b0, (kh1 - kh0) * g, kh1 - kh0
        t["o"] = torch.empty_like(t["q"])
        t["lse"] = torch.empty((B, H, w.N), dtype=torch.float32, device=dev)
        if w.backward:
            t["dq"], t["dk"], t["dv"] = torch.empty_like(t["q"]), torch.empty_like(t["k"]), torch.empty_like(t["v"])
            nb = fa.fa_bwd_workspace_bytes(B, H, Hkv, w.N, w.d)
            t["ws"], t["nb"] = torch.empty(nb, dtype=torch.uint8, device=dev), nb
        pieces.append((B, H, Hkv, t))
    stream = torch.cuda.current_stream()
    sptr = stream.cuda_stream

    def step():
        for B, H, Hkv, t in pieces:
            st = fa.fa_fwd(t["q"], t["k"], t["v"], t["o"], t["lse"], B, H, Hkv, w.N, w.d, w.sm_scale, w.causal, sptr)
            if st == fa.FA_OK and w.backward:
                st = fa.fa_bwd(t["q"], t["k"], t["v"], t["o"], t["lse"], t["dO"], t["dq"], t["dk"], t["dv"], B, H, Hkv,
                               w.N, w.d, w.sm_scale, w.causal, t["ws"], t["nb"], sptr)
            if st != fa.FA_OK:
                raise fa.FaError(st, "sharded step")

    sampler = ClockSampler(local)
    sampler.start()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    wall0 = time.time()
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    sampler.mark(wall0, time.time())
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    clocks = sampler.stop()
    total_ms = sharding.max_over_ranks(e0.elapsed_time(e1), dist, dev)
    if fa.fa_last_device_status(sptr) != fa.FA_OK:
        raise RuntimeError("device status reports a timed-out wait")
    problem_f = w.fwd_flops() + (w.bwd_flops() if w.backward else 0.0)
    value = problem_f * args.steps / (total_ms * 1e-3) / 1e12  # the whole problem, once per step, over all ranks
    launches = len(pieces) * (4 if w.backward else 1) * args.steps
    if rank == 0:
        print(json.dumps({
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True, "scaling": "strong",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) rounded to bf16)",
            "config": dict(config_of(w), parallelism=f"{w.B * w.Hkv} (batch, kv head) groups split over {world} GPUs"),
            "gpu_launches_rank0": launches, "pieces_rank0": [list(pc) for pc in sharding.head_pieces(w.B, w.Hkv, world, 0)],
            "clocks": clocks}), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


# ------------------------------------------------------------------ FP8 forward
def run_fp8(args):
    """One step = fa_fwd_fp8 (rotation + e4m3 quantization launches + the FP8 forward) on the headline shape."""
    import torch

    import exact_attention_blackwell_gb300 as fa
    from exact_attention_blackwell_gb300 import inputs

    torch.cuda.set_device(0)
    fa.lib()
    w = inputs.headline()
    x = inputs.make_inputs(w, with_dO=False)
    dev = torch.device("cuda", 0)
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    B, H, Hkv, N, d = w.B, w.H, w.Hkv, w.N, w.d
    g = torch.Generator().manual_seed(w.seed)
    signs = torch.where(torch.rand(d, generator=g) < 0.5, -1.0, 1.0).to(torch.float32).to(dev)
    o, lse = torch.empty_like(q), torch.empty((B, H, N), dtype=torch.float32, device=dev)
    nb = fa.fa_fwd_fp8_workspace_bytes(B, H, Hkv, N, d)
    ws = torch.empty(nb, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    sptr = stream.cuda_stream

    def step():
        st = fa.fa_fwd_fp8(q, k, v, signs, o, lse, B, H, Hkv, N, d, w.sm_scale, w.causal, ws, nb, sptr)
        if st != fa.FA_OK:
            raise fa.FaError(st, "fa_fwd_fp8")

    sampler = ClockSampler(0)
    sampler.start()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    wall0 = time.time()
    t0.record(stream)
    for _ in range(args.steps):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    sampler.mark(wall0, time.time())
    clocks = sampler.stop()
    if fa.fa_last_device_status(sptr) != fa.FA_OK:
        raise RuntimeError("device status reports a timed-out wait")
    ms = t0.elapsed_time(t1) / args.steps
    f = w.fwd_flops()
    value = f / (ms * 1e-3) / 1e12
    peaks = measured_peaks()
    fp8_peak = 2.0 * peaks["burst"]  # the nominal fp8 : bf16 dense ratio of the part is 2
    print(json.dumps({
        "metric": "attention forward TFLOPs/s, FP8 (e4m3) with incoherent processing, d=128, 1 GB300",
        "value": value, "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "e4m3", "data": "synthetic",
        "config": {"workload": w.name + " fwd, fp8 (rotation and quantization launches included)", "B": B, "H": H,
                   "Hkv": Hkv, "N": N, "d": d, "causal": w.causal,
                   "l2": "inputs larger than L2 (no flush between steps)"},
        "roofline": {"bound": "tensor", "kernel": "fa_fwd_fp8 (3 launches)", "achieved": value, "peak": fp8_peak,
                     "unit": "TFLOP/s", "frac": value / fp8_peak,
                     "peak_source": peaks["source"] + ", " + PEAK_NOTE + ", x 2 (nominal fp8 / bf16 ratio)",
                     "traffic": None},
        "gpu_launches": 3 * args.steps, "clocks": clocks}), flush=True)
    return 0


# ------------------------------------------------------------------ packed variable-length batch
def run_varlen(args):
    """One step = fa_fwd_varlen + fa_bwd_varlen on a packed causal batch (single GPU)."""
    import torch

    import exact_attention_blackwell_gb300 as fa
    from exact_attention_blackwell_gb300 import inputs

    if env_int("WORLD_SIZE", 1) > 1:
        raise SystemExit("--workload varlen runs on one GPU")
    torch.cuda.set_device(0)
    fa.lib()
    w = inputs.packed_causal()
    x_cpu = inputs.make_packed_inputs(w)
    dev = torch.device("cuda", 0)
    q, k, v, dO = (x_cpu[n].to(dev) for n in ("q", "k", "v", "dO"))
    cu = x_cpu["cu_seqlens"].to(dev)
    B, T, L, H, Hkv, d = w.B, w.total, w.max_seqlen, w.H, w.Hkv, w.d
    o, lse = torch.empty_like(q), torch.empty((H, T), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    nb = fa.fa_bwd_workspace_bytes(B, H, Hkv, L, d)
    ws = torch.empty(nb, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    sptr = stream.cuda_stream
    ev = lambda: torch.cuda.Event(enable_timing=True)
    fwd_ev, bwd_ev = [], []

    def step(record=False):
        e = [ev() for _ in range(3)] if record else None
        if record:
            e[0].record(stream)
        st = fa.fa_fwd_varlen(q, k, v, o, lse, cu, B, L, T, H, Hkv, d, w.sm_scale, w.causal, sptr)
        if st != fa.FA_OK:
            raise fa.FaError(st, "fa_fwd_varlen")
        if record:
            e[1].record(stream)
        st = fa.fa_bwd_varlen(q, k, v, o, lse, dO, dq, dk, dv, cu, B, L, T, H, Hkv, d, w.sm_scale, w.causal, ws, nb,
                              sptr)
        if st != fa.FA_OK:
            raise fa.FaError(st, "fa_bwd_varlen")
        if record:
            e[2].record(stream)
            fwd_ev.append((e[0], e[1]))
            bwd_ev.append((e[1], e[2]))

    sampler = ClockSampler(0)
    sampler.start()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    t0, t1 = ev(), ev()
    wall0 = time.time()
    t0.record(stream)
    for _ in range(args.steps):
        step(record=True)
    t1.record(stream)
    torch.cuda.synchronize()
    sampler.mark(wall0, time.time())
    clocks = sampler.stop()
    if fa.fa_last_device_status(sptr) != fa.FA_OK:
        raise RuntimeError("device status reports a timed-out wait")
    total_ms = t0.elapsed_time(t1)
    fwd_f, bwd_f = w.fwd_flops(), w.bwd_flops()
    fwd_ms = statistics.mean(a.elapsed_time(b) for a, b in fwd_ev)
    bwd_ms = statistics.mean(a.elapsed_time(b) for a, b in bwd_ev)
    value = (fwd_f + bwd_f) * args.steps / (total_ms * 1e-3) / 1e12
    peaks = measured_peaks()
    # the backward's three launches execute 7 GEMMs of the forward's 2 (S and dP recomputed)
    achieved = 3.5 * fwd_f / (bwd_ms * 1e-3) / 1e12
    out = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) rounded to bf16)",
           "config": {"workload": w.name + " fwd+bwd", "B": B, "total": T, "max_seqlen": L, "H": H, "Hkv": Hkv,
                      "d": d, "causal": w.causal, "lens": list(w.lens),
                      "l2": "inputs larger than L2 (no flush between steps)", "parallelism": "one GPU"},
           "frac_of_2250_tflops": value / NOMINAL_BF16_TFLOPS,
           "fwd_tflops": fwd_f / (fwd_ms * 1e-3) / 1e12, "fwd_ms": fwd_ms,
           "bwd_tflops": bwd_f / (bwd_ms * 1e-3) / 1e12, "bwd_ms": bwd_ms,
           "roofline": {"bound": "tensor", "kernel": "backward (pre + dK/dV + dQ launches)", "achieved": achieved,
                        "peak": peaks["burst"], "unit": "TFLOP/s", "frac": achieved / peaks["burst"],
                        "frac_of_sustained": achieved / peaks["sustained"],
                        "peak_source": peaks["source"] + ", " + PEAK_NOTE,
                        "flops_per_launch": 3.5 * fwd_f, "launch_ms": bwd_ms, "traffic": None},
           "gpu_launches": 4 * args.steps, "clocks": clocks}
    if not args.no_e2e:
        # The same schedule as the fixed-length workloads: step i's uploads (s_in)
        # overlap step i-1's kernels (s_cmp) and step i-2's downloads (s_out) over
        # two device buffer sets; the kernels of all steps run in order on s_cmp,
        # so they share one workspace.
        names = ("q", "k", "v", "dO")
        pin = {n: x_cpu[n].pin_memory() for n in names}
        first_in = {"q": q, "k": k, "v": v, "dO": dO}
        first_out = [o, lse, dq, dk, dv]
        sets = [(first_in, first_out),
                ({n: torch.empty_like(first_in[n]) for n in names}, [torch.empty_like(t) for t in first_out])]
        outs_h = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in first_out]
        s_in, s_cmp, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)

        def kernels(ins, outs, sp):
            st = fa.fa_fwd_varlen(ins["q"], ins["k"], ins["v"], outs[0], outs[1], cu, B, L, T, H, Hkv, d, w.sm_scale,
                                  w.causal, sp)
            if st != fa.FA_OK:
                raise fa.FaError(st, "fa_fwd_varlen")
            st = fa.fa_bwd_varlen(ins["q"], ins["k"], ins["v"], outs[0], outs[1], ins["dO"], outs[2], outs[3],
                                  outs[4], cu, B, L, T, H, Hkv, d, w.sm_scale, w.causal, ws, nb, sp)
            if st != fa.FA_OK:
                raise fa.FaError(st, "fa_bwd_varlen")

        def pipeline(n_steps, e_start=None, e_end=None):
            in_done, cmp_done, out_done = [], [], []
            if e_start is not None:
                e_start.record(s_in)
            for i in range(n_steps):
                ins, outs = sets[i % 2]
                if i >= 2:
                    s_in.wait_event(cmp_done[i - 2])  # step i-2 has finished reading this input set
                with torch.cuda.stream(s_in):
                    for n in names:
                        ins[n].copy_(pin[n], non_blocking=True)
                in_done.append(torch.cuda.Event())
                in_done[-1].record(s_in)
                s_cmp.wait_event(in_done[i])
                if i >= 2:
                    s_cmp.wait_event(out_done[i - 2])  # step i-2's outputs in this set are on the host
                kernels(ins, outs, s_cmp.cuda_stream)
                cmp_done.append(torch.cuda.Event())
                cmp_done[-1].record(s_cmp)
                s_out.wait_event(cmp_done[i])
                with torch.cuda.stream(s_out):
                    for hd, dd in zip(outs_h, outs):
                        hd.copy_(dd, non_blocking=True)
                out_done.append(torch.cuda.Event())
                out_done[-1].record(s_out)
            if e_end is not None:
                for e in out_done + cmp_done:
                    s_out.wait_event(e)
                e_end.record(s_out)

        n_e2e = max(3, args.steps // 2)
        torch.cuda.synchronize()
        pipeline(3)
        torch.cuda.synchronize()
        e0, e1 = ev(), ev()
        pipeline(n_e2e, e0, e1)
        torch.cuda.synchronize()
        if fa.fa_last_device_status(sptr) != fa.FA_OK:
            raise RuntimeError("device status reports a timed-out wait (end-to-end leg)")
        ms = e0.elapsed_time(e1)
        out["e2e"] = {"value": (fwd_f + bwd_f) * n_e2e / (ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                      "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in pin.values()),
                      "d2h_bytes_per_step": sum(t.numel() * t.element_size() for t in outs_h), "ms_per_step": ms / n_e2e,
                      "schedule": "three streams: uploads of step i, kernels of step i-1, downloads of step i-2 "
                                  "overlap; two device buffer sets"}
        if not torch.equal(outs_h[0], first_out[0].cpu()) and not torch.equal(outs_h[0], sets[1][1][0].cpu()):
            raise RuntimeError("end-to-end output differs from the device result")
    if not args.no_cpu_baseline:
        import oracle

        oracle.build()
        n = min(w.lens)
        a = w.cu_seqlens()[list(w.lens).index(n)]
        sl = lambda t: t[None, a:a + n]
        t_start = time.perf_counter()
        oracle.attention_fwd(sl(x_cpu["q"]), sl(x_cpu["k"]), sl(x_cpu["v"]), w.sm_scale, w.causal)
        oracle.attention_bwd(sl(x_cpu["q"]), sl(x_cpu["k"]), sl(x_cpu["v"]), sl(x_cpu["dO"]), w.sm_scale, w.causal)
        t = time.perf_counter() - t_start
        f = 3.5 * 4.0 * H * n * n * d / 2
        out["cpu_baseline"] = {"value": f / t / 1e12, "unit": "TFLOP/s", "cores": oracle.num_threads(),
                               "kind": "oracle", "seconds": t,
                               "sample": f"the shortest sequence ({n} rows, all {H} heads), fwd+bwd, fp64"}
    print(json.dumps(out), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: 100 for our arm, 20 for the CPU oracle arm)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=["headline", "causal", "gqa", "varlen", "fp8"] + SWEEP_NAMES,
                    default="headline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--shard", action="store_true",
                    help="split one problem over the ranks by (batch, kv head) groups (strong scaling)")
    ap.add_argument("--batch", type=int, default=None,
                    help="override the workload's batch (smaller cases of the same kernels, e.g. for profiling)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)  # at least three untimed warm-up steps, whatever is asked
    if args.workload in ("varlen", "fp8") and args.impl == "ours":
        if args.steps is None:
            args.steps = 100
        return run_varlen(args) if args.workload == "varlen" else run_fp8(args)
    if args.workload == "fp8":
        print(json.dumps({"impl": "reference", "unavailable": "the fp8 line has no oracle arm; use the headline workload"}))
        return 0
    if args.steps is None:
        # our arm: about 0.6 s of timed work on the headline workload, long enough for the
        # clock record; the oracle arm: one (batch, head) slice per step, a few seconds each
        args.steps = 20 if args.impl == "reference" else 100
    if args.shard and args.impl == "ours":
        return run_sharded(args)
    return run_reference(args) if args.impl == "reference" else run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
