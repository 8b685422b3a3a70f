#!/usr/bin/env python3
"""Benchmark of the quantized attention forward on GB300.

One step = one pass of the whole hot path over one batch: quantise Q/K/V
(INT8 per 32-token block, E4M3 per V channel) and run the fused attention
kernel, through the C ABI (``sage_attn_fwd``).  The metric is the pages'
attention throughput, TOPS = 4*B*H*S^2*D / step time.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                  [--impl ours|reference] [--graph] [--lse|--fused-q|--smooth-k]

``--graph`` replays each step from a ``sage_plan`` (the call recorded once
as a CUDA graph, with ``--fused-q`` or ``--smooth-k`` that variant) instead
of calling ``sage_attn_fwd``; the kernels and their
output are the same, only the per-call host work goes.

N > 1 runs N independent replicas, one process per GPU (the method has no
exchange step in one call): under torchrun each rank is one replica; run
directly, bench.py starts the N rank processes itself.  The line reports the
whole-job throughput over the maximum time of the ranks.  ``--impl reference`` times the CPU
oracle (the only stand-in for a reference implementation: none exists for
this hardware) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
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

METRIC = "quantized attention TOPS (4*B*H*S^2*D/s)"
UNIT = "TOPS"
DTYPE = "int8+e4m3"          # INT8 QK^T (exact, FP32 accumulate), E4M3 PV (FP32 accumulate)
DEFAULT_WORKLOAD = "b2_s16384_h24_outlier"
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "attention_traffic.json")
ATTN_SOURCES = [os.path.join(ROOT, "quantized_attention_diffusion_gb300", "csrc", f)
                for f in ("attention.cu", "sm103_ptx.cuh")]


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="approximate CPU time budget of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--lse", action="store_true",
                    help="time sage_attn_fwd_lse (also writes the per-row log-sum-exp)")
    ap.add_argument("--fused-q", action="store_true",
                    help="time sage_attn_fwd_fused_q (Q quantised inside the attention kernel)")
    ap.add_argument("--smooth-k", action="store_true",
                    help="time sage_attn_fwd_smooth_k (K loses its per-channel mean before quantisation)")
    ap.add_argument("--graph", action="store_true",
                    help="replay each step from a sage_plan (the call recorded once as a CUDA graph)")
    ap.add_argument("--no-e2e", action="store_true",
                    help="skip the host-buffer leg (for short profiling runs; the line then has no e2e figure)")
    ap.add_argument("--launcher-selftest", action="store_true",
                    help="CPU check of the replica launcher and rank plumbing (gloo): no GPU, no metric")
    return ap.parse_args()


# ------------------------------------------------------------ processes --

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


class Group:
    """Barrier and max-reduce across ranks (no data-path collective)."""

    def __init__(self, world, rank, local, use_cuda):
        self.world, self.rank = world, rank
        self.dist = None
        if world > 1:
            import torch.distributed as dist
            os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
            dist.init_process_group("nccl" if use_cuda else "gloo")
            self.dist = dist

    def barrier(self):
        if self.dist:
            self.dist.barrier()

    def max(self, x: float) -> float:
        if not self.dist:
            return x
        import torch
        dev = torch.device("cuda", torch.cuda.current_device()) if torch.cuda.is_available() else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.dist.all_reduce(t, op=self.dist.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.dist:
            self.dist.destroy_process_group()


def free_port() -> int:
    import socket
    with socket.socket() as sock:
        sock.bind(("127.0.0.1", 0))
        return sock.getsockname()[1]


def launch_replicas(n: int, argv) -> int:
    """Run this script as n rank processes (RANK = LOCAL_RANK = 0..n-1,
    WORLD_SIZE = n, rendezvous on 127.0.0.1), one GPU each; rank 0's output
    passes through.  Returns the worst exit code."""
    port = str(free_port())
    procs = []
    for r in range(n):
        env = dict(os.environ, RANK=str(r), LOCAL_RANK=str(r), WORLD_SIZE=str(n),
                   LOCAL_WORLD_SIZE=str(n), MASTER_ADDR="127.0.0.1", MASTER_PORT=port)
        out = None if r == 0 else subprocess.DEVNULL
        procs.append(subprocess.Popen([sys.executable, os.path.abspath(__file__), *argv], env=env, stdout=out))
    codes = [p.wait() for p in procs]
    return max(codes, key=abs)


def job_tops(world: int, ops_per_call: float, calls_per_rank: int, ms_max: float) -> float:
    """Whole-job throughput of weak-scaled replicas: every rank runs the
    same number of calls; the slowest rank's time bounds the job."""
    return world * ops_per_call * calls_per_rank / (ms_max * 1e-3) / 1e12


# --------------------------------------------------------------- clocks --

class ClockSampler:
    """SM clock, power and clock-event reasons of one GPU, read through NVML
    (read-only queries) every `period_s` by a background thread; `stop`
    keeps the samples taken inside [t0, t1], the host times that bracket
    the timed region.  Falls back to `nvidia-smi -lms 20` without NVML."""

    # nvmlClocksEventReasons bits
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, cuda_index: int, period_s: float = 0.005):
        self.cuda_index, self.period = cuda_index, period_s
        self.samples, self.source = [], None
        self.thread = self.proc = None
        self.stop_flag = False

    def _nvml_handle(self):
        import ctypes
        nvml = ctypes.CDLL("libnvidia-ml.so.1")
        if nvml.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        h = ctypes.c_void_p()
        uuid = None
        try:
            import torch
            uuid = str(torch.cuda.get_device_properties(self.cuda_index).uuid)
        except Exception:
            pass
        ok = -1
        if uuid:
            uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
            ok = nvml.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(h))
        if ok != 0:
            ok = nvml.nvmlDeviceGetHandleByIndex_v2(self.cuda_index, ctypes.byref(h))
        if ok != 0:
            raise OSError("no NVML handle")
        return nvml, h

    def start(self):
        import threading
        try:
            nvml, h = self._nvml_handle()
        except OSError:
            return self._start_smi()
        import ctypes
        reasons_fn = getattr(nvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            nvml.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint(0)
        nvml.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx))
        self.max_mhz = float(mx.value)
        self.source = "nvml"

        def run():
            sm, pw, rs = ctypes.c_uint(0), ctypes.c_uint(0), ctypes.c_ulonglong(0)
            while not self.stop_flag:
                t = time.perf_counter()
                if nvml.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(sm)) == 0:
                    nvml.nvmlDeviceGetPowerUsage(h, ctypes.byref(pw))
                    reasons_fn(h, ctypes.byref(rs))
                    self.samples.append((t, float(sm.value), pw.value / 1000.0, int(rs.value)))
                time.sleep(self.period)

        self.thread = threading.Thread(target=run, daemon=True)
        self.thread.start()

    def _start_smi(self):
        fields = "clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active"
        try:
            self.file = tempfile.TemporaryFile(mode="w+")
            self.t_smi0 = time.perf_counter()
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.cuda_index), f"--query-gpu={fields}",
                 "--format=csv,noheader,nounits", "-lms", "20"], stdout=self.file, stderr=subprocess.DEVNULL)
            self.source = "nvidia-smi"
        except OSError:
            self.proc = None

    def stop(self, t0: float, t1: float):
        if self.thread is not None:
            self.stop_flag = True
            self.thread.join(timeout=5)
            rows = [(sm, pw, rs) for t, sm, pw, rs in self.samples if t0 <= t <= t1]
            smax = self.max_mhz
        elif self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.file.seek(0)
            rows, smax = [], None
            for line in self.file.read().splitlines():
                f = [x.strip() for x in line.split(",")]
                try:
                    rows.append((float(f[0]), float(f[2]), int(f[3], 16)))
                    smax = float(f[1])
                except (ValueError, IndexError):
                    continue
        else:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no clock source"]}
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": smax, "reasons": ["no samples"], "source": self.source}
        reasons = sorted({name for _, _, rs in rows for bit, name in self.REASONS.items() if rs & bit})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": smax, "reasons": reasons,
                "samples": len(rows), "sm_mhz_min": min(r[0] for r in rows),
                "power_w_max": max(r[1] for r in rows), "source": self.source,
                "period_ms": round(self.period * 1e3, 1) if self.source == "nvml" else 20}


# ---------------------------------------------------------------- peaks --

def tensor_peak():
    """Dense peaks of the attention kernel's mixed contraction (TFLOP/s).

    QK^T runs at the fp16/bf16 tensor rate P (the measured cuBLAS bf16
    figure), PV on E4M3 at 2P (the ratio our tcgen05 probe measured per MMA:
    M=128, N=256, kind::f16 with K=16 and kind::f8f6f4 with K=32 both take
    128 SM clocks).  Half the ops run at each rate, so the combined peak is
    4 / (2/P + 2/(2P)) = 4P/3.  The headline uses the burst P (a kernel timed
    on its own, at the clock it ran at); the sustained P (a seconds-long,
    power-capped GEMM loop) is returned too.
    Returns (burst, sustained, bf16 burst, hbm GB/s, source)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    src = "fallback"
    p_burst, p_sust, hbm = 1900.0, 1700.0, 6800.0
    try:
        with open(path) as f:
            m = json.load(f)
        p_burst = float(m["bf16_tflops"])
        p_sust = float(m.get("bf16_tflops_sustained", p_burst))
        hbm = float(m["hbm_gbs"])
        src = "measured"
    except (OSError, KeyError, ValueError):
        pass
    return 4.0 * p_burst / 3.0, 4.0 * p_sust / 3.0, p_burst, hbm, src


# tcgen05 dense rate per SM and clock at M=128: 8192 fp16 flop (our probe:
# N=256, K=16 in 128 clocks), E4M3 twice that; GB300 has 152 SMs.
FP16_FLOP_PER_CLK_SM = 8192
N_SMS = 152
# ex2.approx results per clock per SM: one warp instruction per 4 clocks per
# sub-partition (the attention kernel's XU counter matches its ex2 count at
# that rate); the softmax takes one per score element.
EX2_PER_CLK_SM = 32
MAX_SM_MHZ = 2070


def attention_traffic():
    """dram bytes per attention launch from the committed ncu summary, or
    None if the kernel source changed since it was captured."""
    try:
        with open(PROFILE_TRAFFIC) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    h = hashlib.sha256()
    for p in ATTN_SOURCES:
        with open(p, "rb") as f:
            h.update(f.read())
    if rec.get("source_sha256") != h.hexdigest():
        return None
    return rec.get("dram_bytes_per_launch_full")


# -------------------------------------------------------- oracle timing --

def cpu_model() -> str:
    """The host CPU's model name (x86 /proc/cpuinfo, else lscpu, which also
    names Arm cores), for the oracle's timing record."""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return platform.machine() or "unknown"


def oracle_sample(w, q, k, v, seconds: float, steps: int = 1):
    """Time the CPU oracle on a bounded sample: one (batch, head) of the
    workload, quantised whole, and as many of its query rows as fit in
    `seconds` per step.  Returns (TOPS, sample text, cores, s_per_step)."""
    import numpy as np

    import oracle
    from quantized_attention_diffusion_gb300.workloads import bf16_bits

    b, h = 0, 0
    sl = [np.ascontiguousarray(bf16_bits(t[b:b + 1, :, h:h + 1, :])) for t in (q, k, v)]

    def run(n_rows):
        t0 = time.perf_counter()
        quant = oracle.quantize(*sl)
        rows = np.stack([np.zeros(n_rows), np.zeros(n_rows),
                         np.linspace(0, w.S - 1, n_rows).round()], axis=1).astype(np.int32)
        oracle.attend_rows(quant, w.S, w.softmax_scale, rows, Skv=w.skv)
        return time.perf_counter() - t0

    n_cal = 64
    t_cal = run(n_cal)
    t_quant = max(1e-3, run(1))
    per_row = max(1e-7, (t_cal - t_quant) / (n_cal - 1))
    n_rows = int(max(8, min(w.S, (seconds - t_quant) / per_row)))
    times = [run(n_rows) for _ in range(steps)]
    t = statistics.median(times) if steps > 1 else times[0]
    ops = 4.0 * n_rows * w.skv * w.D
    sample = (f"one (b,h) of {w.name}: quantise its {w.S} query and {w.skv} key/value tokens, "
              f"then attention for {n_rows} of its query rows ({ops:.3g} ops)")
    return ops / t / 1e12, sample, oracle.num_threads(), ops, times


# ------------------------------------------------------------------ ours --

def run_ours(args, group, local):
    import torch

    import quantized_attention_diffusion_gb300 as qad
    from quantized_attention_diffusion_gb300.workloads import WORKLOADS, make_workload

    w = WORKLOADS[args.workload]
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    qad.load_library()
    q_h, k_h, v_h = make_workload(w)                       # CPU, seeded
    q, k, v = (t.to(dev) for t in (q_h, k_h, v_h))
    cpu_sample = [t[:1, :, :1].clone() for t in (q_h, k_h, v_h)]   # one (b, h) for the oracle leg
    out = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.S), dtype=torch.float32, device=dev) if args.lse else None
    K, W = args.steps, args.warmup

    def step(qq, kk, vv, oo, ll=None):
        if w.Skv is not None:
            qad.attn_fwd_cross(qq, kk, vv, w.softmax_scale, out=oo, lse=ll)
        elif args.lse:
            qad.attn_fwd_lse(qq, kk, vv, w.softmax_scale, out=oo, lse=ll)
        else:
            qad.attn_fwd(qq, kk, vv, w.softmax_scale, out=oo, fused_q=args.fused_q, smooth_k=args.smooth_k)

    if args.lse + args.fused_q + args.smooth_k > 1 or ((args.fused_q or args.smooth_k) and w.Skv is not None):
        raise SystemExit("--lse, --fused-q and --smooth-k select one call each; the last two are self-attention")
    plans = {}

    def plan_step(qq, kk, vv, oo, ll=None):
        key = (qq.data_ptr(), oo.data_ptr())
        if key not in plans:                                 # recorded once per buffer set, before timing
            plans[key] = qad.Plan(qq, kk, vv, w.softmax_scale, out=oo, lse=ll, smooth_k=args.smooth_k,
                                  fused_q=args.fused_q)
        plans[key].launch()

    run = plan_step if args.graph else step
    for _ in range(W):
        run(q, k, v, out, lse)
    torch.cuda.synchronize()

    # per-step events around the attention kernel (materialise handles first)
    before = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    after = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    for e in before + after:
        e.record()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    sampler = ClockSampler(local)
    group.barrier()
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.1)
    t0 = time.perf_counter()
    start.record()
    for i in range(K):
        if not args.graph:
            qad.set_attention_events(before[i], after[i])
        run(q, k, v, out, lse)
    end.record()
    torch.cuda.synchronize()
    t1 = time.perf_counter()
    qad.set_attention_events()
    group.barrier()
    clocks = sampler.stop(t0, t1)
    ms = start.elapsed_time(end)
    if args.graph:
        # A graph records no timing hook: the attention kernel's own duration
        # comes from the same kernels launched by direct calls, K more steps.
        for i in range(K):
            qad.set_attention_events(before[i], after[i])
            step(q, k, v, out, lse)
        torch.cuda.synchronize()
        qad.set_attention_events()
    attn_ms = statistics.mean(b.elapsed_time(a) for b, a in zip(before, after))
    ms_max = group.max(ms)
    attn_ms_max = group.max(attn_ms)
    value = job_tops(group.world, w.ops, K, ms_max)

    # End to end through the public API with host buffers: every step copies
    # its Q/K/V from pinned host memory to the device, runs the step and
    # copies its output back to pinned host memory.  Device buffers are
    # double-buffered and the copies run on their own streams, so step i+1's
    # upload and step i-1's download overlap step i's compute, as a serving
    # loop would; all K2 steps' copies are inside the timed region.  The first
    # step's upload and the last step's download overlap nothing (about 4 ms at
    # 2 x 16384 x 24 on a ~200 GB/s host link), so the leg runs at least 40
    # steps to show the loop's steady rate rather than its fill and drain.
    K2 = max(40, min(K, 200))
    e2e_value = None
    if not args.no_e2e:
        host_in = [t.pin_memory() for t in (q_h, k_h, v_h)]
        host_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        host_lse = torch.empty(lse.shape, dtype=lse.dtype).pin_memory() if args.lse else None
        del q_h, k_h, v_h
        bufs = [[torch.empty_like(t) for t in (q, k, v)] for _ in range(2)]
        outs = [torch.empty_like(out) for _ in range(2)]
        lses = [torch.empty_like(lse) for _ in range(2)] if args.lse else [None, None]
        comp = torch.cuda.current_stream(dev)
        up, down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

        def e2e(n):
            h2d = [torch.cuda.Event() for _ in range(n)]
            done = [torch.cuda.Event() for _ in range(n)]
            d2h = [torch.cuda.Event() for _ in range(n)]
            for i in range(n + 1):
                if i < n:
                    with torch.cuda.stream(up):
                        if i >= 2:
                            up.wait_event(done[i - 2])          # buffer i%2 is free again
                        for dst, src in zip(bufs[i % 2], host_in):
                            dst.copy_(src, non_blocking=True)
                        h2d[i].record(up)
                if i >= 1:
                    b = (i - 1) % 2
                    comp.wait_event(h2d[i - 1])
                    if i - 1 >= 2:
                        comp.wait_event(d2h[i - 3])             # output buffer b was read back
                    run(*bufs[b], outs[b], lses[b])
                    done[i - 1].record(comp)
                    with torch.cuda.stream(down):
                        down.wait_event(done[i - 1])
                        host_out.copy_(outs[b], non_blocking=True)
                        if args.lse:
                            host_lse.copy_(lses[b], non_blocking=True)
                        d2h[i - 1].record(down)
            comp.wait_event(d2h[n - 1])

        e2e(2)
        torch.cuda.synchronize()
        group.barrier()
        s2, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s2.record(up)
        comp.wait_event(s2)
        e2e(K2)
        e2.record(comp)
        torch.cuda.synchronize()
        group.barrier()
        e2e_ms = group.max(s2.elapsed_time(e2))
        e2e_value = job_tops(group.world, w.ops, K2, e2e_ms)
    in_bytes = (q.numel() + k.numel() + v.numel()) * q.element_size()
    out_bytes = out.numel() * out.element_size() + (lse.numel() * 4 if args.lse else 0)

    peak, peak_sust, p_bf16, hbm, src = tensor_peak()
    achieved = w.ops / (attn_ms_max * 1e-3) / 1e12
    clock_peak = None
    if clocks.get("sm_mhz"):
        clock_peak = 4.0 / 3.0 * FP16_FLOP_PER_CLK_SM * N_SMS * clocks["sm_mhz"] * 1e6 / 1e12
    exps = w.B * w.H * w.S * w.skv
    xu_ms = exps / (EX2_PER_CLK_SM * N_SMS * (clocks.get("sm_mhz") or MAX_SM_MHZ) * 1e6) * 1e3
    # The quantisation pass: 3 B per element of each tensor it quantises
    # (2 B of bf16 read, 1 B of code written); with fused Q, Q is quantised
    # inside the attention kernel, and K smoothing reads K once more.
    e_q, e_kv = w.B * w.S * w.H * w.D, w.B * w.skv * w.H * w.D
    q_bytes = (0 if args.fused_q else 3 * e_q) + 6 * e_kv + (2 * e_kv if args.smooth_k else 0)
    quant_ms = ms_max / K - attn_ms_max
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": UNIT,
        "n_gpus": group.world,
        "steps": K,
        "warmup": W,
        "ms_per_step": round(ms_max / K, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": DTYPE,
        "data": "synthetic (seeded; shapes and distributions of the pages' diffusion workloads)",
        "config": {
            "workload": w.name, "B": w.B, "S": w.S, "Skv": w.skv, "H": w.H, "D": w.D, "recipe": w.recipe,
            "seed": w.seed, "softmax_scale": w.softmax_scale, "path": ("sage_attn_fwd_cross" if w.Skv is not None else "sage_attn_fwd_lse" if args.lse
                     else "sage_attn_fwd_fused_q" if args.fused_q
                     else "sage_attn_fwd_smooth_k" if args.smooth_k else "sage_attn_fwd") + (" (quantise + attention + LSE)" if args.lse
                                               else " (quantise + attention)")
                    + (", replayed from a sage_plan CUDA graph" if args.graph else ""),
            "l2": f"inputs larger than L2 ({in_bytes / 1e6:.0f} MB read per step, L2 129 MB)",
            "parallelism": "replicas" if group.world > 1 else "single GPU",
        },
        "e2e": {"value": round(e2e_value, 2), "unit": UNIT, "h2d_bytes_per_step": in_bytes,
                "d2h_bytes_per_step": out_bytes, "steps": K2,
                "note": "pinned host Q/K/V -> device, sage_attn_fwd, output -> pinned host, every step; "
                        "copies of neighbouring steps overlap compute on separate streams; the first upload "
                        "and the last download (pipeline fill and drain) are inside the timed region"}
        if e2e_value is not None else {"skipped": "--no-e2e"},
        "gpu_launches": qad.attn_fwd_launches(w.B, w.S, w.H, Skv=w.Skv, smooth_k=args.smooth_k) * K,
        "roofline": {
            "bound": "tensor", "achieved": round(achieved, 1), "peak": round(peak, 1), "unit": "TFLOP/s",
            "frac": round(achieved / peak, 4), "traffic": attention_traffic(),
            "kernel": "sage_attn_kernel", "attention_ms_per_launch": round(attn_ms_max, 4),
            "peak_basis": f"{src} cuBLAS bf16 burst {p_bf16} TFLOP/s (of measured) for QK^T at the fp16 rate, "
                          f"2x for E4M3 PV (per-MMA ratio measured by a tcgen05 probe): 4P/3",
            "peak_sustained": round(peak_sust, 1), "frac_vs_sustained": round(achieved / peak_sust, 4),
            "peak_at_sampled_clock": round(clock_peak, 1) if clock_peak else None,
            "frac_vs_sampled_clock": round(achieved / clock_peak, 4) if clock_peak else None,
            "secondary": {"xu": {"exp2_per_launch": exps, "floor_ms": round(xu_ms, 4),
                                 "frac": round(xu_ms / attn_ms_max, 4),
                                 "basis": f"one ex2.approx per score element, {N_SMS} SMs x {EX2_PER_CLK_SM} "
                                          f"per clock at the sampled SM clock"}},
        },
        "quantise": {
            "ms_per_step": round(quant_ms, 4), "algorithmic_bytes": q_bytes,
            "achieved_gbs": round(q_bytes / (quant_ms * 1e-3) / 1e9, 1) if quant_ms > 0 else None,
            "peak_gbs": round(hbm, 1),
            "frac": round(q_bytes / (quant_ms * 1e-3) / 1e9 / hbm, 4) if quant_ms > 0 else None,
            "note": "step time outside the attention kernel: the quantisation launches and the gaps between "
                    "launches; bytes are the pass's algorithmic 3 per element of each tensor it quantises",
        },
        "clocks": clocks,
    }
    if group.rank == 0 and group.world == 1 and not args.no_cpu_baseline:
        tops, sample, cores, _, _ = oracle_sample(w, *cpu_sample, args.cpu_seconds)
        line["cpu_baseline"] = {"value": round(tops, 6), "unit": UNIT, "cores": cores, "cpu": cpu_model(),
                                "kind": "oracle", "sample": sample}
    return line


# ------------------------------------------------------------- reference --

def run_reference(args):
    from quantized_attention_diffusion_gb300.workloads import WORKLOADS, make_workload

    w = WORKLOADS[args.workload]
    q, k, v = make_workload(w)
    K, W = args.steps, args.warmup
    per_step = max(0.05, min(2.0, 150.0 / max(1, K + W)))
    _, sample, cores, ops, times = oracle_sample(w, q, k, v, per_step, steps=K + W)
    timed = times[W:] if len(times) > W else times
    t = statistics.mean(timed)
    value = ops / t / 1e12
    return {
        "impl": "reference",
        "metric": METRIC, "value": round(value, 6), "unit": UNIT, "n_gpus": 1, "steps": K, "warmup": W,
        "ms_per_step": round(t * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": DTYPE,
        "data": "synthetic (seeded; shapes and distributions of the pages' diffusion workloads)",
        "config": {"workload": w.name, "B": w.B, "S": w.S, "Skv": w.skv, "H": w.H, "D": w.D, "recipe": w.recipe,
                   "seed": w.seed, "softmax_scale": w.softmax_scale,
                   "path": "CPU oracle (plain C, OpenMP) on a bounded sample per step"},
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": cores, "cpu": cpu_model(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def launcher_selftest(world, rank, local):
    """Rank plumbing on CPU (gloo): barrier, then the max of per-rank times;
    rank 0 prints what the real line's n_gpus and ms_max would be."""
    group = Group(world, rank, local, use_cuda=False)
    try:
        group.barrier()
        ms_max = group.max(10.0 + rank)
        group.barrier()
        if rank == 0:
            print(json.dumps({"launcher_selftest": True, "n_gpus": group.world, "ms_max": ms_max}), flush=True)
    finally:
        group.close()


def main():
    args = parse_args()
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ and args.impl == "ours":
        sys.exit(launch_replicas(args.gpus, sys.argv[1:]))
    world, rank, local = dist_env()
    if args.launcher_selftest:
        return launcher_selftest(world, rank, local)
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    import torch
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the attention path has no CPU fallback)")
    group = Group(world, rank, local, use_cuda=True)
    try:
        line = run_ours(args, group, local)
        if rank == 0:
            print(json.dumps(line), flush=True)
    finally:
        group.close()


if __name__ == "__main__":
    main()
