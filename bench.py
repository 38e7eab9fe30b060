#!/usr/bin/env python3
"""Throughput benchmark of libgemm.so on GB300: TFLOP/s = 2*M*N*K / time.

Default workload (one step = one call of the C ABI): FP16 TN GEMM with
M = N = K = 8192, A row-major, B column-major, C column-major, FP32
accumulation, entries N(0,1)*0.1 (seed 2).  The line also reports BF16 and
FP8-E4M3 at 8192^3 and the FP32 SIMT path at 4096^3, each against its dense
peak, every BF16/FP8 configuration shape and the pages' transformer and
skinny shapes (per_config), the end-to-end rate with host buffers, the kernel's roofline fraction,
the SM clocks seen while timing, the CPU oracle timed on a bounded sample, and
the main call's per-launch mean, median and min with L2 warm and flushed.

Timing: W untimed warm-up steps, then exactly K steps between a barrier and a
synchronize on each side, timed with CUDA events on the launching stream.
Steps rotate over three input sets (3 x 384 MiB, far above the 129 MB L2), so
no step finds its operands in L2; no flush kernel runs.  Under torchrun each
rank runs its own replica (weak scaling: the GEMM does not need a collective),
the time is the maximum over ranks and `value` counts every rank's work.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--no-per-config]
  python bench.py --ncu-case bf16:128x8192x8192[:half=3,workspace=0]
                  (launches for a profiler capture, with library options if given)
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GEMM TFLOP/s (2MNK/time) FP16 TN 8192³, BF16, FP8; % of GB300 dense peak"
UNIT = "TFLOP/s"
# Best FP16 TN 8192^3 figure on the pages: the tuned 192x224 kernel on an
# RX 9070 XT, FP16 accumulation ("FP16 GEMM Optimization on AMD RDNA 3 and
# RDNA 4", "Tuning Further", Table 17).  Another machine: context only.
PAGES_FP16_8192_TFLOPS = 142.30
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FP8_OVER_BF16 = 2.0  # nominal dense ratio (4.5 / 2.25 PFLOP/s)
SETS = 3
WORKSPACE_BYTES = 1 << 30   # the library workspace the bench registers (1 GiB)


# ---------------------------------------------------------------- helpers

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world: int, backend: str):
    import torch.distributed as dist

    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist if world > 1 else None


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(dist, value: float, device=None) -> float:
    """Largest `value` over all ranks (the job's time is its slowest rank's)."""
    if dist is None:
        return value
    import torch

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_tflops(flops_per_step: float, steps: int, world: int, max_ms: float) -> float:
    """Whole-job TFLOP/s: every rank's work over the slowest rank's time."""
    return flops_per_step * steps * world / (max_ms * 1e-3) / 1e12


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            p = json.load(fh)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi sampling (every 100 ms) around a timed region."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._reader = threading.Thread(target=self._read, daemon=True)
            self._reader.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, begin: bool):
        if begin:
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            rows.append((ts, parts))
        timed = self.t0 is not None and self.t1 is not None
        inside = [r for r in rows if timed and self.t0 - 0.05 <= r[0] <= self.t1 + 0.15]
        use = inside or rows
        sm = [float(p[2]) for _, p in use if p[2].replace(".", "").isdigit()]
        mx = [float(p[3]) for _, p in use if p[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, p in use for i in range(4) if p[6 + i] == "Active"})
        power = [float(p[4]) for _, p in use if p[4].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons,
                "samples": len(use), "samples_in_window": len(inside),
                "power_w_max": max(power) if power else None}


# ------------------------------------------------------- our implementation

def tn_sets(kind, M, N, K, seed, sigma, nsets, device, out_f32=False):
    """Seeded operands for a TN call, copied into `nsets` distinct buffer sets."""
    import torch

    import synthetic_inputs as si

    ops = si.tn_operands(kind, M, N, K, dist="normal", seed=seed, sigma=sigma)
    out_dt = torch.float32 if out_f32 else (torch.float16 if kind == "f16" else torch.bfloat16)
    sets = []
    for _ in range(nsets):
        a = ops["A"].to(device)
        b = ops["B"].to(device)
        c = torch.empty((N, M), dtype=out_dt, device=device)
        sets.append((a, b, c))
    return ops, sets


def tn_call(kind, M, N, K, scale_a, scale_b, stream_h, out_f32=False):
    from dense_gemm_tcgen05_gb300 import capi

    fns = {"f16": capi.gemm_f16_tn, "bf16": capi.gemm_bf16_tn}
    fp8 = capi.gemm_fp8_tn_f32 if out_f32 else capi.gemm_fp8_tn

    def call(a, b, c):
        if kind == "e4m3":
            st = fp8(M, N, K, a.data_ptr(), K, b.data_ptr(), K, scale_a, scale_b, c.data_ptr(), M,
                     stream_h)
        else:
            st = fns[kind](M, N, K, a.data_ptr(), K, b.data_ptr(), K, c.data_ptr(), M, stream_h)
        if st != 0:
            raise RuntimeError("gemm call failed: %s" % capi.status_text(st))

    return call


def timed_loop(call, sets, steps, warmup, stream, dist=None, sampler=None):
    """W warm-up steps, then K timed steps; returns (total_ms, mean_launch_ms)."""
    total, launches = timed_launches(call, sets, steps, warmup, stream, dist, sampler)
    return total, sum(launches) / len(launches)


def timed_launches(call, sets, steps, warmup, stream, dist=None, sampler=None):
    """W warm-up steps, then K timed steps; returns (total_ms, [ms per launch])."""
    import torch

    for i in range(warmup):
        call(*sets[i % len(sets)])
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    t_begin = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    barrier(dist)
    torch.cuda.synchronize()
    if sampler:
        sampler.mark(True)
    t_begin.record(stream)
    for i in range(steps):
        starts[i].record(stream)
        call(*sets[i % len(sets)])
        ends[i].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    if sampler:
        sampler.mark(False)
    barrier(dist)
    total = t_begin.elapsed_time(t_end)
    launches = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    return total, launches


def graph_time(call, sets, launches, stream, replays=9):
    """Mean ms per call of `launches` back-to-back calls, rotating over `sets`,
    captured in one CUDA graph and replayed (median of `replays`): the steady
    state of a stream of calls, without the host's launch cost and without
    events between the calls, which keep programmatic dependent launch from
    overlapping a call's prologue with the end of the one before."""
    import torch

    with torch.cuda.stream(stream):
        for i in range(3):
            call(*sets[i % len(sets)])
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(launches):
                call(*sets[i % len(sets)])
        g.replay()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        per = []
        for _ in range(replays):
            e0.record(stream)
            g.replay()
            e1.record(stream)
            e1.synchronize()
            per.append(e0.elapsed_time(e1) / launches)
    del g
    return statistics.median(per)


def spread(launches):
    """Mean, median, min and max of per-launch times (ms)."""
    ms = sorted(launches)
    return {"mean_ms": round(sum(ms) / len(ms), 4), "median_ms": round(statistics.median(ms), 4),
            "min_ms": round(ms[0], 4), "max_ms": round(ms[-1], 4), "launches": len(ms)}


def e2e_loop(kind, M, N, K, ops, steps, warmup, stream, stream_h):
    """End to end through the C ABI with host buffers: every step copies A and
    B from pinned host memory, runs the GEMM and copies C back to pinned host
    memory.  Steps are pipelined the way a throughput-bound caller would run
    them: two device buffer sets, host-to-device copies on one stream, the GEMM
    on `stream`, device-to-host copies on a third, so that the copies of steps
    i + 1 and i - 1 overlap the GEMM of step i; events order each buffer's reuse.
    The timed region runs from before the first step's input copy to after the
    last step's output copy.  Returns (pipelined ms per step, serial ms per step,
    host-to-device bytes per step, device-to-host bytes per step, copies-only ms
    per step); the serial figure runs copy, GEMM, copy back to back on one
    stream, for context.  The copies-only figure runs the same pipelined steps
    without the GEMM (the better of two runs): the host link's own limit on
    this loop, against which the end-to-end rate is read."""
    import torch

    ha = ops["A"].pin_memory()
    hb = ops["B"].pin_memory()
    out_dt = torch.float16 if kind == "f16" else torch.bfloat16
    hc = torch.empty((N, M), dtype=out_dt).pin_memory()
    da = [torch.empty_like(ha, device="cuda") for _ in range(2)]
    db = [torch.empty_like(hb, device="cuda") for _ in range(2)]
    dc = [torch.empty((N, M), dtype=out_dt, device="cuda") for _ in range(2)]
    call = tn_call(kind, M, N, K, ops["scale_a"], ops["scale_b"], stream_h)
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: [torch.cuda.Event() for _ in range(2)]  # noqa: E731
    in_done, gemm_done, out_done = ev(), ev(), ev()

    def step(i, gemm=True):
        j = i % 2
        if i >= 2:
            s_in.wait_event(gemm_done[j])      # the GEMM of step i - 2 has read slot j
        with torch.cuda.stream(s_in):
            da[j].copy_(ha, non_blocking=True)
            db[j].copy_(hb, non_blocking=True)
        in_done[j].record(s_in)
        stream.wait_event(in_done[j])
        if i >= 2:
            stream.wait_event(out_done[j])     # C of step i - 2 has left slot j
        if gemm:
            call(da[j], db[j], dc[j])
        gemm_done[j].record(stream)
        s_out.wait_event(gemm_done[j])
        with torch.cuda.stream(s_out):
            hc.copy_(dc[j], non_blocking=True)
        out_done[j].record(s_out)

    def serial_step():
        with torch.cuda.stream(stream):
            da[0].copy_(ha, non_blocking=True)
            db[0].copy_(hb, non_blocking=True)
            call(da[0], db[0], dc[0])
            hc.copy_(dc[0], non_blocking=True)

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(s_in)
    for i in range(steps):
        step(i)
    t1.record(s_out)                           # after the last copy back, which follows all
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / steps

    # The copies alone: the ceiling the pipelined steps approach.  A warm-up
    # step, then the better of two runs, since a short run can catch a slow
    # moment of the host link and would understate the ceiling.
    copy_ms = None
    for _ in range(2):
        step(0, gemm=False)
        torch.cuda.synchronize()
        t0.record(s_in)
        for i in range(steps):
            step(i, gemm=False)
        t1.record(s_out)
        torch.cuda.synchronize()
        c = t0.elapsed_time(t1) / steps
        copy_ms = c if copy_ms is None else min(copy_ms, c)

    for _ in range(warmup):
        serial_step()
    torch.cuda.synchronize()
    t0.record(stream)
    for _ in range(steps):
        serial_step()
    t1.record(stream)
    torch.cuda.synchronize()
    serial_ms = t0.elapsed_time(t1) / steps
    h2d = ha.numel() * ha.element_size() + hb.numel() * hb.element_size()
    d2h = hc.numel() * hc.element_size()
    return ms, serial_ms, h2d, d2h, copy_ms


def l2_modes(ops, M, N, K, stream, stream_h, launches=30, warmup=10):
    """Per-launch CUDA-event times of the main call in two L2 modes: "warm",
    the same operands at every launch, and "cold", a 512 MiB buffer (four
    times L2) written between launches, outside the events.  Mean, median
    and min per launch for each."""
    import torch

    a = ops["A"].to("cuda")
    b = ops["B"].to("cuda")
    c = torch.empty((N, M), dtype=torch.float16, device="cuda")
    call = tn_call("f16", M, N, K, 1.0, 1.0, stream_h)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    flops = 2.0 * M * N * K
    out = {"launches": launches, "flush_bytes": flush.numel()}
    for mode in ("warm", "cold"):
        events = []
        with torch.cuda.stream(stream):
            for i in range(warmup + launches):
                if mode == "cold":
                    flush.fill_(i & 0xFF)
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                call(a, b, c)
                e1.record(stream)
                if i >= warmup:
                    events.append((e0, e1))
        torch.cuda.synchronize()
        ms = sorted(e0.elapsed_time(e1) for e0, e1 in events)
        median = statistics.median(ms)
        out[mode] = {"mean_ms": round(sum(ms) / len(ms), 4), "median_ms": round(median, 4),
                     "min_ms": round(ms[0], 4),
                     "tflops_at_median": round(flops / (median * 1e-3) / 1e12, 1)}
    del a, b, c, flush
    torch.cuda.empty_cache()
    return out


def f32_bench(n, steps, warmup, stream, stream_h):
    import torch

    import synthetic_inputs as si
    from dense_gemm_tcgen05_gb300 import capi

    ops = si.f32_operands(n, n, n, dist="uniform", seed=1)
    sets = [(ops["A"].cuda(), ops["B"].cuda(), torch.empty((n, n), device="cuda"))
            for _ in range(SETS)]

    def call(a, b, c):
        st = capi.gemm_f32(n, n, n, a.data_ptr(), n, b.data_ptr(), n, c.data_ptr(), n, stream_h)
        if st != 0:
            raise RuntimeError(capi.status_text(st))

    with torch.cuda.stream(stream):
        total, launch = timed_loop(call, sets, steps, warmup, stream)
    return launch


def f32_bf16x6_bench(n, steps, warmup, stream, stream_h):
    """gemm_f32_bf16x6 on the FP32 leg's operands (U[-1,1], seed 1), with the
    splits in the bench's registered workspace; returns the mean per-call ms
    (two split launches and the GEMM)."""
    import torch

    import synthetic_inputs as si
    from dense_gemm_tcgen05_gb300 import capi

    ops = si.f32_operands(n, n, n, dist="uniform", seed=1)
    sets = [(ops["A"].cuda(), ops["B"].cuda(), torch.empty((n, n), device="cuda"))
            for _ in range(SETS)]
    # the bench's registered workspace holds the splits
    assert capi.gemm_f32_bf16x6_workspace_bytes(n, n, n) <= WORKSPACE_BYTES

    def call(a, b, c):
        st = capi.gemm_f32_bf16x6(n, n, n, a.data_ptr(), n, b.data_ptr(), n, c.data_ptr(), n,
                                  stream_h)
        if st != 0:
            raise RuntimeError(capi.status_text(st))

    with torch.cuda.stream(stream):
        total, launch = timed_loop(call, sets, steps, warmup, stream)
    return launch


def cublas_context(M, N, K, dtype, steps, stream):
    """torch.matmul (cuBLAS) on the same problem, for context only.  FP32 runs
    with TF32 off, i.e. on the CUDA cores like gemm_f32."""
    import torch

    a = torch.randn((M, K), device="cuda").to(dtype)
    b = torch.randn((N, K), device="cuda").to(dtype)
    tf32 = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = False
    try:
        return _time_matmul(a, b, M, N, K, steps, stream)
    finally:
        torch.backends.cuda.matmul.allow_tf32 = tf32


def _time_matmul(a, b, M, N, K, steps, stream):
    import torch

    with torch.cuda.stream(stream):
        for _ in range(3):
            torch.matmul(a, b.t())
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(steps):
            torch.matmul(a, b.t())
        t1.record(stream)
        torch.cuda.synchronize()
    return 2.0 * M * N * K / (t0.elapsed_time(t1) / steps * 1e-3) / 1e12


def sm_count():
    import torch

    return torch.cuda.get_device_properties(0).multi_processor_count


# A timed window shorter than this stays in the burst regime.  Back-to-back
# 8192^3 GEMMs reach the power cap within ~0.1 s (a 0.67 s window of 1000
# launches ran at 1424 MHz with sw_power_cap set), the regime the measured
# sustained peak was taken in.
SUSTAINED_MIN_WINDOW_MS = 250.0


def tensor_peak(window_ms: float, clocks, burst: float, sustained: float):
    """The tensor peak a timed window is held against, and why: the sustained
    figure only when the window lasted seconds AND the clock sampler saw the
    power cap inside it; otherwise the burst figure."""
    reasons = (clocks or {}).get("reasons") or []
    capped = "sw_power_cap" in reasons
    if window_ms >= SUSTAINED_MIN_WINDOW_MS and capped:
        return sustained, "sustained", ("window %.0f ms >= %.0f ms with sw_power_cap seen"
                                        % (window_ms, SUSTAINED_MIN_WINDOW_MS))
    why = ("window %.0f ms < %.0f ms" % (window_ms, SUSTAINED_MIN_WINDOW_MS)
           if window_ms < SUSTAINED_MIN_WINDOW_MS else "no sw_power_cap seen in the window")
    return burst, "burst", why


def fp32_alu_peak_tflops(sms: int, mhz: float) -> float:
    """FFMA peak: SMs x 128 FP32 lanes x 2 flops x clock."""
    return sms * 128 * 2 * mhz * 1e6 / 1e12


def _oracle_sample_rate(oracle, si, kind, M, N, K, a, b, seed, budget_s):
    """Times the oracle on a growing number of random output elements until
    one timing takes `budget_s`; returns (TFLOP/s, elements, seconds)."""
    count = 512
    elapsed = 0.0
    while True:
        ms, ns = si.sample_positions(M, N, count, seed=seed, edges=False)
        t0 = time.perf_counter()
        oracle.gemm_tn_sampled(kind, K, a, K, b, K, ms, ns)
        elapsed = time.perf_counter() - t0
        if elapsed >= budget_s or count >= 1 << 26:
            break
        count = int(count * min(16.0, max(2.0, budget_s / max(elapsed, 1e-3))))
    return 2.0 * K * count / elapsed / 1e12, count, elapsed


def cpu_baseline(kind="f16", M=8192, N=8192, K=8192, seed=2, sigma=0.1, budget_s=12.0,
                 one_core_budget_s=3.0):
    """The oracle, as it stands, on a bounded sample of the workload: random
    output elements of the same problem, each one K-long FP64 dot product.
    Timed on all the cores OpenMP uses, then on one core."""
    import oracle
    import synthetic_inputs as si

    ops = si.tn_operands(kind, M, N, K, dist="normal", seed=seed, sigma=sigma)
    a, b = si.codes(ops["A"]), si.codes(ops["B"])
    cores = oracle.num_threads()
    tflops, count, elapsed = _oracle_sample_rate(oracle, si, kind, M, N, K, a, b, seed, budget_s)
    oracle.set_num_threads(1)
    try:
        one, count1, elapsed1 = _oracle_sample_rate(oracle, si, kind, M, N, K, a, b, seed,
                                                    one_core_budget_s)
    finally:
        oracle.set_num_threads(cores)
    return {"value": tflops, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": "%d random output elements of the %s TN %dx%dx%d problem (each a %d-long "
                      "FP64 dot product), %.1f s" % (count, kind, M, N, K, K, elapsed),
            "one_core": {"value": one, "unit": UNIT, "cores": 1,
                         "sample": "%d elements, %.1f s" % (count1, elapsed1)}}


def run_ours(args):
    import torch

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dist = init_dist(world, "nccl")
    from dense_gemm_tcgen05_gb300 import build as libbuild
    from dense_gemm_tcgen05_gb300 import capi

    if rank == 0 or world == 1:
        libbuild.build()
    barrier(dist)
    capi.lib()
    peaks, peak_src = load_peaks()
    burst = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    sustained = float(peaks.get("bf16_tflops_sustained",
                                FALLBACK_PEAKS["bf16_tflops_sustained"]))
    stream = torch.cuda.Stream()
    stream_h = stream.cuda_stream
    # The library's recommended setup: one caller-owned workspace, registered
    # once (split-K for shapes that cannot fill the GPU, a last wave cut into K
    # pieces for long tiles, and the FP32 tensor-core leg's operand splits).
    from dense_gemm_tcgen05_gb300 import capi as _capi_ws
    workspace = torch.empty(WORKSPACE_BYTES, dtype=torch.uint8, device="cuda")
    if _capi_ws.gemm_set_workspace(workspace.data_ptr(), workspace.numel()) != 0:
        raise RuntimeError("could not register the workspace")
    M = N = K = 8192
    flops = 2.0 * M * N * K

    ops, sets = tn_sets("f16", M, N, K, seed=2, sigma=0.1, nsets=SETS, device="cuda")
    call = tn_call("f16", M, N, K, 1.0, 1.0, stream_h)
    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    with torch.cuda.stream(stream):
        total_ms, launch_ms = timed_loop(call, sets, args.steps, args.warmup, stream, dist,
                                         sampler)
    clocks = sampler.stop() if sampler else None
    max_ms = max_over_ranks(dist, total_ms, device="cuda")
    value = aggregate_tflops(flops, args.steps, world, max_ms)
    achieved = flops / (launch_ms * 1e-3) / 1e12
    del sets
    torch.cuda.empty_cache()

    result = None
    if rank == 0 and args.only_main:
        result = {"metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
                  "steps": args.steps, "warmup": args.warmup,
                  "ms_per_step": round(max_ms / args.steps, 5), "higher_is_better": True,
                  "scaling": "weak", "note": "--only-main: main workload only (profiling runs)",
                  "roofline": {"achieved": round(achieved, 1), "peak": burst}}
    elif rank == 0:
        per = {}
        sub_steps = max(10, min(args.steps, 50))
        for kind, peak in (("bf16", burst), ("e4m3", burst * FP8_OVER_BF16)):
            o, s = tn_sets(kind, M, N, K, seed=4 if kind == "e4m3" else 3,
                           sigma=1.0 if kind == "e4m3" else 0.05, nsets=SETS, device="cuda")
            c = tn_call(kind, M, N, K, o["scale_a"], o["scale_b"], stream_h)
            with torch.cuda.stream(stream):
                _, ls = timed_launches(c, s, sub_steps, 3, stream)
            lm = sum(ls) / len(ls)
            tf = flops / (lm * 1e-3) / 1e12
            per[kind + "_tn_8192"] = {"tflops": round(tf, 1), "peak": round(peak, 1),
                                      "frac": round(tf / peak, 4), **spread(ls)}
            del s
            torch.cuda.empty_cache()
        # FP16 accumulation (the FP16 page's measured mode), same problem
        from dense_gemm_tcgen05_gb300 import capi as _capi

        o16, s16 = tn_sets("f16", M, N, K, seed=2, sigma=0.1, nsets=SETS, device="cuda")

        def acc16(a, b, c):
            st = _capi.gemm_f16_tn_acc16(M, N, K, a.data_ptr(), K, b.data_ptr(), K, c.data_ptr(),
                                         M, stream_h)
            if st != 0:
                raise RuntimeError(_capi.status_text(st))

        with torch.cuda.stream(stream):
            _, lm = timed_loop(acc16, s16, sub_steps, 3, stream)
        tf = flops / (lm * 1e-3) / 1e12
        per["f16_acc16_tn_8192"] = {"tflops": round(tf, 1), "peak": round(burst, 1),
                                    "frac": round(tf / burst, 4),
                                    "over_pages_fp16_acc16": round(tf / PAGES_FP16_8192_TFLOPS, 1)}
        del s16
        torch.cuda.empty_cache()
        lm = f32_bench(4096, sub_steps, 3, stream, stream_h)
        tf = 2.0 * 4096 ** 3 / (lm * 1e-3) / 1e12
        clk = clocks.get("sm_max_mhz") if clocks and clocks.get("sm_max_mhz") else 2070.0
        fpk = fp32_alu_peak_tflops(sm_count(), clk)
        per["f32_simt_4096"] = {"tflops": round(tf, 2), "peak": round(fpk, 1),
                                "frac": round(tf / fpk, 4), "bound": "alu"}
        # The same FP32 product on the tensor cores (exact BF16 splits, six
        # piece products): effective FP32 rate, and the BF16 tensor rate the
        # GEMM runs at (6 x 2 n^3 over the whole call, splits included).
        lx = f32_bf16x6_bench(4096, sub_steps, 3, stream, stream_h)
        tfx = 2.0 * 4096 ** 3 / (lx * 1e-3) / 1e12
        per["f32_bf16x6_4096"] = {"tflops": round(tfx, 1), "tensor_tflops": round(6 * tfx, 1),
                                  "peak": round(burst, 1), "frac": round(6 * tfx / burst, 4),
                                  "bound": "tensor", "over_simt": round(tfx / tf, 2)}
        per["cublas_context_f32_4096"] = round(cublas_context(4096, 4096, 4096, torch.float32,
                                                              20, stream), 2)
        per["cublas_context_f16_8192"] = round(cublas_context(M, N, K, torch.float16, 20, stream), 1)
        per_cfg = None
        if not args.no_per_config:
            hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
            per_cfg = per_config(stream, stream_h, burst, hbm, workspace)

        e2e_steps = max(3, min(args.steps, 20))
        e_ms, serial_ms, h2d, d2h, copy_ms = e2e_loop("f16", M, N, K, ops, e2e_steps, 2, stream,
                                             stream_h)
        try:
            l2 = l2_modes(ops, M, N, K, stream, stream_h)
        except Exception as exc:  # an auxiliary figure must not cost the line itself
            l2 = {"error": "%s: %s" % (type(exc).__name__, exc)}
        traffic = load_traffic()
        peak, regime, why = tensor_peak(total_ms, clocks, burst, sustained)
        result = {
            "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(max_ms / args.steps, 5),
            "higher_is_better": True, "scaling": "weak",
            # The pages' FP16 8192^3 figure accumulates in FP16, this metric in
            # FP32, so it is not the same metric: context below, no ratio here.
            "vs_baseline": None,
            "dtype": "f16", "data": "synthetic",
            "config": {**workload_config(world), "accumulate": "f32",
                       "l2": "3 rotating input sets (1.1 GiB total) >> 129 MB L2, no flush",
                       "workspace_bytes": WORKSPACE_BYTES,
                       "pages_context": "best FP16 8192^3 on the pages: 142.30 TFLOP/s (RX 9070 "
                                        "XT, FP16 accumulation); compare per_dtype."
                                        "f16_acc16_tn_8192"},
            # The timed window's own clock record picks the peak: sustained only
            # for a window of seconds that ran under the power cap, else burst.
            "roofline": {"bound": "tensor", "achieved": round(achieved, 1), "peak": peak,
                         "unit": UNIT, "frac": round(achieved / peak, 4),
                         "traffic": traffic,
                         "peak_source": "%s bf16 %s (fp16 runs at the same tensor rate): %s"
                                        % (peak_src, regime, why),
                         "frac_of_burst": round(achieved / burst, 4),
                         "frac_of_sustained": round(achieved / sustained, 4)},
            "e2e": {"value": round(flops / (e_ms * 1e-3) / 1e12, 2), "unit": UNIT,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "steps": e2e_steps,
                    "how": "pinned host A, B -> device, gemm_f16_tn, C -> pinned host, every "
                           "step; copies of neighbouring steps overlap the GEMM (two buffer "
                           "sets, three streams)",
                    "serial_value": round(flops / (serial_ms * 1e-3) / 1e12, 2),
                    # the same pipelined loop with the GEMM left out: the host
                    # link's ceiling for this metric, and its rate in GB/s
                    "copies_only_value": round(flops / (copy_ms * 1e-3) / 1e12, 2),
                    "copies_only_gbs": round((h2d + d2h) / (copy_ms * 1e-3) / 1e9, 1),
                    "frac_of_copies_only": round(copy_ms / e_ms, 4)},
            "gpu_launches": args.steps,
            "clocks": clocks,
            "per_dtype": per,
            "per_config": per_cfg,
            "l2_modes": l2,
        }
        if not args.no_cpu_baseline:
            result["cpu_baseline"] = cpu_baseline()
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    return result


def compulsory_bytes(kind, M, N, K, out_f32=False) -> int:
    """Bytes a TN call must move at least: A and B read once, C written once."""
    es = 1 if kind == "e4m3" else 2
    return (M * K + N * K) * es + M * N * (4 if out_f32 else 2)


L2_BYTES = 129 * 10 ** 6   # GB300 L2 (129 MB)

# The shapes of the BF16 and FP8 configurations, the pages' own transformer
# shapes ("FP16 GEMM Optimization on AMD RDNA 3 and RDNA 4", "Where That
# Leaves Us", Table 16; "FP8 GEMM Optimization on AMD RDNA 4", "Results",
# Tables 1-4, which write FP32 C) and skinny shapes whose time is set by HBM
# ("Tuning Further").  (kind, (M, N, K), FP32 output, values (seed, sigma),
# HBM-bound).
PER_CONFIG = [
    ("bf16", (4096, 4096, 4096), False, (3, 0.05), False),
    ("bf16", (4096, 14336, 4096), False, (3, 0.05), False),
    ("bf16", (4096, 4096, 14336), False, (3, 0.05), False),
    ("bf16", (2047, 3001, 1023), False, (3, 0.05), False),
    ("bf16", (8191, 8191, 8191), False, (3, 0.05), False),
    ("e4m3", (8192, 8192, 8192), False, (4, 1.0), False),
    ("e4m3", (4096, 14336, 4096), False, (4, 1.0), False),
    ("e4m3", (16384, 4096, 4096), False, (4, 1.0), False),
    ("f16", (8192, 28672, 8192), False, (2, 0.1), False),
    ("e4m3", (8192, 8192, 8192), True, (4, 1.0), False),
    ("e4m3", (8192, 28672, 8192), True, (4, 1.0), False),
    ("e4m3", (8192, 10240, 8192), True, (4, 1.0), False),
    ("e4m3", (3072, 4096, 8192), True, (4, 1.0), False),
    ("bf16", (16, 8192, 8192), False, (3, 0.05), True),
    ("bf16", (128, 8192, 8192), False, (3, 0.05), True),
    ("bf16", (192, 8192, 8192), False, (3, 0.05), True),
    ("bf16", (256, 8192, 8192), False, (3, 0.05), True),
    ("bf16", (64, 14336, 4096), False, (3, 0.05), True),
    ("bf16", (1024, 1024, 8192), False, (3, 0.05), True),
    ("e4m3", (128, 8192, 8192), False, (4, 1.0), True),
]


def sets_beyond_l2(kind, M, N, K, out_f32=False):
    """Rotating input sets whose bytes together exceed twice the L2, so that
    no launch finds its operands there (at least 3)."""
    per = compulsory_bytes(kind, M, N, K, out_f32)
    return max(SETS, min(64, -(-2 * L2_BYTES // per)))


def per_config(stream, stream_h, burst, hbm, workspace, launches=20):
    """Every configuration shape above, timed with the bench's workspace
    registered (the library's recommended setup): `launches` back-to-back
    calls after 3 warm-ups over rotating input sets that exceed the L2.  Each
    entry: TFLOP/s at the mean launch, the fraction of the dtype's burst peak
    (FP8 = 2x BF16 by the nominal ratio), GB/s of compulsory bytes and the
    per-launch spread; the HBM-bound shapes add the fraction of the measured
    copy bandwidth, and the same calls replayed as a CUDA graph (graph_us,
    graph_gbs, hbm_frac_graph: the steady state of a stream of calls, where a
    call's prologue overlaps the end of the one before) with cuBLAS replayed
    the same way beside them (16-bit inputs: torch's linear, whose M x N
    row-major output is the transpose of this library's layout, and matmul
    into this library's layout).  The tight-leading-dimension
    BF16 shapes are timed again without a workspace (the load-based producer
    reads them in place)."""
    import torch

    from dense_gemm_tcgen05_gb300 import capi

    out = {}

    def one(kind, M, N, K, f32, seed, sigma, tag="", graph=False):
        nsets = sets_beyond_l2(kind, M, N, K, f32)
        o, s = tn_sets(kind, M, N, K, seed=seed, sigma=sigma, nsets=nsets, device="cuda",
                       out_f32=f32)
        c = tn_call(kind, M, N, K, o["scale_a"], o["scale_b"], stream_h, out_f32=f32)
        with torch.cuda.stream(stream):
            _, ls = timed_launches(c, s, launches, 3, stream)
        lm = sum(ls) / len(ls)
        tf = 2.0 * M * N * K / (lm * 1e-3) / 1e12
        peak = burst * (FP8_OVER_BF16 if kind == "e4m3" else 1.0)
        byts = compulsory_bytes(kind, M, N, K, f32)
        gbs = byts / (lm * 1e-3) / 1e9
        key = "%s%s_%dx%dx%d%s" % (kind, "_f32out" if f32 else "", M, N, K, tag)
        out[key] = {"tflops": round(tf, 1), "frac": round(tf / peak, 4), "gbs": round(gbs),
                    "sets": nsets, **spread(ls)}
        if graph:
            # The same calls as a replayed CUDA graph, and cuBLAS (torch's
            # linear on the same operands, 16-bit inputs) replayed the same
            # way, for context.
            gm = graph_time(c, s, 2 * len(s) * max(1, 10 // len(s)), stream)
            out[key]["graph_us"] = round(gm * 1e3, 2)
            out[key]["graph_gbs"] = round(byts / (gm * 1e-3) / 1e9)
            if kind != "e4m3" and not f32:
                # linear writes C as M x N row-major, the transpose of this
                # library's layout, and cuBLAS then picks its kernel for that
                # problem; matmul into the (N, M) buffer keeps this library's
                # layout (C = B A^T row-major, i.e. column-major M x N).
                def lin(a, b, _c):
                    torch.nn.functional.linear(a, b)

                def same_layout(a, b, c):
                    torch.matmul(b, a.t(), out=c)
                cm = graph_time(lin, s, 2 * len(s) * max(1, 10 // len(s)), stream)
                out[key]["cublas_graph_us"] = round(cm * 1e3, 2)
                out[key]["cublas_over_this"] = round(cm / gm, 3)
                cs = graph_time(same_layout, s, 2 * len(s) * max(1, 10 // len(s)), stream)
                out[key]["cublas_same_layout_graph_us"] = round(cs * 1e3, 2)
                out[key]["cublas_same_layout_over_this"] = round(cs / gm, 3)
        del s, o
        torch.cuda.empty_cache()
        return key, gbs

    for kind, (M, N, K), f32, (seed, sigma), hbm_bound in PER_CONFIG:
        key, gbs = one(kind, M, N, K, f32, seed, sigma, graph=hbm_bound)
        if hbm_bound:
            out[key]["hbm_frac"] = round(gbs / hbm, 3)
            out[key]["hbm_frac_graph"] = round(out[key]["graph_gbs"] / hbm, 3)
    capi.gemm_set_workspace(None, 0)
    try:
        for M, N, K in ((2047, 3001, 1023), (8191, 8191, 8191)):
            one("bf16", M, N, K, False, 3, 0.05, tag="_no_workspace")
    finally:
        if capi.gemm_set_workspace(workspace.data_ptr(), workspace.numel()) != 0:
            raise RuntimeError("could not register the workspace")
    return out


KERNEL_SOURCES = ("tc_gemm.cuh", "ptx.cuh", "raster.h", "common.h")


def kernel_source_hash() -> str:
    """SHA-256 over the tensor-core kernel's sources, to tell whether committed
    profiler counters still describe the kernel being timed."""
    import hashlib

    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "dense_gemm_tcgen05_gb300", "csrc", name), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def load_traffic():
    """DRAM bytes per launch of the main kernel from the committed ncu summary
    (profiles/tc_gemm_f16_8192.txt); None when there is none or when the
    kernel's sources changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "tc_gemm_f16_8192.txt")
    fields = {}
    try:
        for line in open(path):
            if ":" in line:
                k, v = line.split(":", 1)
                fields[k.strip()] = v.strip()
    except OSError:
        return None
    if fields.get("kernel_source_sha256") != kernel_source_hash():
        return None
    try:
        return int(float(fields["traffic_bytes_per_launch"]))
    except (KeyError, ValueError):
        return None


# -------------------------------------------------------- reference arm

def workload_config(world: int) -> dict:
    """The workload part of the line's config, the same on both arms."""
    return {"workload": "fp16_tn_8192x8192x8192", "M": 8192, "N": 8192, "K": 8192,
            "layout": "TN: A row-major, B column-major, C column-major (ld=M)",
            "values": "N(0,1)*0.1, seed 2",
            "parallelism": "replicas" if world > 1 else "single"}


def run_reference(args):
    """The oracle on the host cores, on the same metric and workload: each step
    is a bounded sample of the FP16 8192^3 problem."""
    world, rank, _ = dist_env()
    if rank != 0:
        return None
    import oracle
    import synthetic_inputs as si

    M = N = K = 8192
    ops = si.tn_operands("f16", M, N, K, dist="normal", seed=2, sigma=0.1)
    a, b = si.codes(ops["A"]), si.codes(ops["B"])
    per_step = 2048
    times = []
    for i in range(args.warmup + args.steps):
        ms, ns = si.sample_positions(M, N, per_step, seed=100 + i, edges=False)
        t0 = time.perf_counter()
        oracle.gemm_tn_sampled("f16", K, a, K, b, K, ms, ns)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(dt)
    total = sum(times)
    value = 2.0 * K * per_step * len(times) / total / 1e12
    sample = ("%d random output elements per step of the f16 TN 8192^3 problem (each an "
              "8192-long FP64 dot product)" % per_step)
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(total / len(times) * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {**workload_config(world), "accumulate": "f64 (the oracle)"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def parse_ncu_case(spec: str):
    """KIND:MxNxK[:name=value,...] -> (kind, M, N, K, options, workspace).  The
    optional third field sets library options (gemm_set_option) for the
    case; workspace=0 runs it without the bench workspace."""
    parts = spec.split(":")
    if len(parts) not in (2, 3):
        raise ValueError("expected KIND:MxNxK[:name=value,...], got %r" % spec)
    kind = parts[0]
    M, N, K = (int(x) for x in parts[1].lower().split("x"))
    options, workspace = {}, True
    if len(parts) == 3 and parts[2]:
        for item in parts[2].split(","):
            name, value = item.split("=")
            if name == "workspace":
                workspace = int(value) != 0
            else:
                options[name] = int(value)
    return kind, M, N, K, options, workspace


def ncu_case(spec: str):
    """A few launches of one TN shape for profiler captures: three rounds of
    this library's call followed by cuBLAS's (torch.matmul) on the same
    operands, with the bench workspace registered (unless the spec says
    workspace=0) and any options the spec names set for the case.  Nothing is
    timed; the line only names the case and the plan.  FP8 runs this
    library's call alone."""
    import torch

    from dense_gemm_tcgen05_gb300 import capi

    kind, M, N, K, options, use_ws = parse_ncu_case(spec)
    if kind == "f32":
        return ncu_case_f32(M, N, K)
    for name, value in options.items():
        if capi.gemm_set_option(name, value) != 0:
            raise ValueError("invalid option %s=%d" % (name, value))
    workspace = torch.empty(WORKSPACE_BYTES, dtype=torch.uint8, device="cuda") if use_ws else None
    if use_ws:
        assert capi.gemm_set_workspace(workspace.data_ptr(), workspace.numel()) == 0
    plan_kind = {"f16": "f16", "bf16": "bf16", "e4m3": "e4m3"}[kind]
    st, plan = capi.gemm_tn_plan(plan_kind, M, N, K,
                                 workspace_bytes=workspace.numel() if use_ws else 0,
                                 sms=torch.cuda.get_device_properties(0).multi_processor_count)
    _, sets = tn_sets(kind, M, N, K, 2, 0.1, 2, "cuda")
    stream = torch.cuda.Stream()
    call = tn_call(kind, M, N, K, 1.0, 1.0, stream.cuda_stream)
    with torch.cuda.stream(stream):
        for i in range(3):
            a, b, c = sets[i % 2]
            call(a, b, c)
            if kind != "e4m3":
                torch.matmul(b, a.T, out=c)      # C column-major = (B A^T) row-major
    torch.cuda.synchronize()
    if use_ws:
        assert capi.gemm_set_workspace(None, 0) == 0
    for name in options:
        capi.gemm_set_option(name, -1 if name == "pair" else 0)
    return {"ncu_case": spec, "launches_each": 3, "cublas": kind != "e4m3", "plan": plan}


def ncu_case_f32(M, N, K):
    """Three gemm_f32 calls (U[-1,1] operands, seed 1) and cuBLAS's FP32 GEMM
    (TF32 off) on the same operands after each, for profiler captures."""
    import torch

    import synthetic_inputs as si
    from dense_gemm_tcgen05_gb300 import capi

    ops = si.f32_operands(M, N, K, dist="uniform", seed=1)
    a, b = ops["A"].cuda(), ops["B"].cuda()
    c = torch.empty((M, N), device="cuda")
    stream = torch.cuda.Stream()
    tf32 = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = False
    try:
        with torch.cuda.stream(stream):
            for _ in range(3):
                st = capi.gemm_f32(M, N, K, a.data_ptr(), K, b.data_ptr(), N, c.data_ptr(), N,
                                   stream.cuda_stream)
                if st != 0:
                    raise RuntimeError(capi.status_text(st))
                torch.matmul(a, b, out=c)
        torch.cuda.synchronize()
    finally:
        torch.backends.cuda.matmul.allow_tf32 = tf32
    return {"ncu_case": "f32:%dx%dx%d" % (M, N, K), "launches_each": 3, "cublas": True}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the per-configuration shapes (BF16/FP8 configs, page shapes)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only-main", action="store_true",
                    help="time the main workload only (for profiler runs)")
    ap.add_argument("--ncu-case", metavar="KIND:MxNxK[:name=value,...]",
                    help="launch one shape (f16/bf16/e4m3 TN, or f32) three times, and cuBLAS "
                         "beside it, for ncu; the optional third field sets library options "
                         "(workspace=0: no workspace)")
    args = ap.parse_args(argv)
    if args.ncu_case:
        print(json.dumps(ncu_case(args.ncu_case)), flush=True)
        return
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        out = run_reference(args)
    else:
        out = run_ours(args)
    if out is not None:
        print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
