"""Benchmark: GFLOP/s and fraction of the FP32 CUDA-core roofline.

Headline (``value``): the exact-mode fp32 product C = A*B at m = n = k = 4096
(A, B ~ N(0, 1), row-major, contiguous), one om_gemm_f32_ws call per step
(the balanced schedule; om_gemm_f32 without scratch is reported beside it),
inputs resident in HBM, L2 flushed (a 512 MiB write) before every timed
call. Also reported per step set: fast mode on the same product, the
ResNet-50 stage-1 3x3 and 1x1 convolutions (exact and fast), the prefill
product and the grouped/strided/dilated convolution.

Roofline: the kernels are bound by the FP32 pipes (bound "alu"). The peak is
derived from unit counts and the maximum SM clock: SMs x 128 FP32 lanes x 2
flops x 2070 MHz (fast mode, one fused multiply-add per term); exact mode
issues a multiply and an add per term, so its ceiling is half of that.

``--impl reference`` times the CPU oracle (plain C loops of the definition)
on the host cores on a bounded row sample of the same product.

Multi-GPU (torchrun, N > 1): every rank runs its own replica of the workload
on its own GPU; there is no data exchange. value = work of all ranks / the
slowest rank's time (weak scaling).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

SM_MAX_MHZ = 2070.0
FP32_LANES_PER_SM = 128


TF32_PER_BF16 = 1.1 / 2.25  # nominal dense tf32 / bf16 tensor rates of the part


def measured_peaks() -> dict:
    """The measured bf16 tensor peak, else the documented fallback."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(path))
        return {"bf16_tflops": float(d["bf16_tflops"]), "hbm_gbs": float(d["hbm_gbs"]),
                "basis": "measured bf16 burst (MEASURED_PEAKS.json)"}
    except (OSError, ValueError, KeyError):
        return {"bf16_tflops": 1900.0, "hbm_gbs": 6800.0, "basis": "fallback bf16 1.9 PFLOP/s"}


def fp32_peak_tflops(sms: int, exact: bool) -> float:
    p = sms * FP32_LANES_PER_SM * 2 * SM_MAX_MHZ * 1e6 / 1e12
    return p / 2 if exact else p


# ----------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clock/throttle samples, each stamped with the host time it
    arrived; summary() keeps the samples taken inside a given time window."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.samples = []  # (host time, sm MHz, max MHz, set of active reasons)
        self.reader = None

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm, mx = float(parts[1]), float(parts[2])
            except ValueError:
                continue
            active = {n for n, v in zip(self.REASONS, parts[5:9]) if v.lower() == "active"}
            self.samples.append((time.time(), sm, mx, active))

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.reader = threading.Thread(target=self._read, daemon=True)
            self.reader.start()
            t0 = time.time()
            while not self.samples and time.time() - t0 < 5.0:
                time.sleep(0.05)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self.reader is not None:
                self.reader.join(timeout=5)

    def summary(self, t0: float, t1: float) -> dict:
        inside = [s for s in self.samples if t0 <= s[0] <= t1 + 0.15]
        basis = "inside the timed region"
        if not inside:
            after = [s for s in self.samples if s[0] >= t0]
            inside = after[:1]
            basis = "first sample after the timed region began (region shorter than the sampling period)"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        reasons = set()
        for s in inside:
            reasons |= s[3]
        return {"sm_mhz": float(np.median([s[1] for s in inside])),
                "sm_max_mhz": max(s[2] for s in inside), "reasons": sorted(reasons),
                "samples": len(inside), "basis": basis}


# ----------------------------------------------------------------- workloads
def gemm_workload():
    from implicit_gemm_convolution_gb300 import synth
    return synth.workload_gemm_4096()


# The sources each kernel's translation unit is built from.
KERNEL_SOURCES = {
    "sgemm_tiled_kernel": ("sgemm_tiled.cu", "simt_tile.cuh", "om_device.cuh", "om_internal.h",
                           "schedule_host.h"),
    "conv_implicit_kernel": ("conv_implicit.cu", "simt_tile.cuh", "om_device.cuh", "om_internal.h",
                             "schedule_host.h"),
    "gemm_tf32x3_kernel": ("gemm_tf32x3.cu", "om_device.cuh", "om_internal.h"),
    "conv_rows_kernel": ("conv_rows.cu", "om_device.cuh", "om_internal.h"),
    "gemv_kernel": ("gemv.cu", "om_device.cuh", "om_internal.h"),
    "conv_dw_tma_kernel": ("conv_direct.cu", "om_device.cuh", "om_internal.h"),
    "conv_group_kernel": ("conv_direct.cu", "om_device.cuh", "om_internal.h"),
}


def kernel_source_hash(kernel: str = "") -> str:
    """SHA-256 prefix of the kernel's sources (all of csrc/ if the kernel is
    not listed in KERNEL_SOURCES)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "implicit_gemm_convolution_gb300", "csrc")
    files = KERNEL_SOURCES.get(kernel) or sorted(
        f for f in os.listdir(csrc) if f.endswith((".cu", ".cuh", ".h")))
    for f in files:
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary
    (profiles/dram_traffic.txt), if it was taken on the current kernel
    sources; else None."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    try:
        lines = open(path).read().splitlines()
    except OSError:
        return None
    for line in lines:
        parts = line.split()
        if len(parts) == 4 and not line.startswith("#") and parts[0] == kernel and parts[1] == workload:
            return int(parts[3]) if parts[2] == kernel_source_hash(kernel) else None
    return None


class L2Flusher:
    def __init__(self, dev):
        import torch
        self.buf = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)

    def __call__(self):
        self.buf.fill_(1.0)


def time_calls(fn, steps: int, warmup: int, flush, stream) -> list[float]:
    """Per-call device time (ms) of fn on stream, L2 flushed before each call."""
    import torch
    for _ in range(warmup):
        flush()
        fn()
    torch.cuda.synchronize()
    times = []
    for _ in range(steps):
        flush()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        e1.synchronize()
        times.append(e0.elapsed_time(e1))
    return times


def time_reps(fn, flush, stream, min_ms: float = 80.0, reps: int = 3, warmup: int = 3,
              min_calls: int = 5) -> dict:
    """The repetition method of the pages' benchmark applied on the device:
    after warm-up calls, each repetition runs calls (L2 flushed before each,
    CUDA events around each on the launching stream) until their summed device
    time reaches min_ms; a repetition's figure is its mean per-call time, and
    the result is the median over the repetitions."""
    import torch
    for _ in range(warmup):
        flush()
        fn()
    torch.cuda.synchronize()
    means, calls = [], []
    for _ in range(reps):
        total, count = 0.0, 0
        while total < min_ms or count < min_calls:
            flush()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            e1.synchronize()
            total += e0.elapsed_time(e1)
            count += 1
        means.append(total / count)
        calls.append(count)
    return {"ms": float(np.median(means)), "rep_ms": [round(v, 5) for v in means],
            "calls_per_rep": calls}


def time_rotating(fns, stream, min_ms: float = 80.0, reps: int = 3, warmup: int = 3) -> dict:
    """Back-to-back calls cycling over fns, each working on its own copy of the
    operands, with no flush in between: the copies are sized so that between
    two calls on the same copy more data than the L2 holds passes through it,
    so no call finds its operands in L2 (the 'inputs larger than L2' rule).
    CUDA events bracket each batch on the launching stream, so launch latency
    overlaps the previous call as it does for a caller issuing calls in a row;
    a repetition's figure is batch time / calls, the result the median."""
    import torch
    n = len(fns)
    for i in range(max(warmup, n)):
        fns[i % n]()
    torch.cuda.synchronize()

    def batch(calls):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(calls):
            fns[i % n]()
        e1.record(stream)
        e1.synchronize()
        return e0.elapsed_time(e1)

    probe = batch(2 * n) / (2 * n)
    calls = max(2 * n, int(np.ceil(min_ms / max(probe, 1e-4) / n)) * n)
    means = [batch(calls) / calls for _ in range(reps)]
    return {"ms": float(np.median(means)), "rep_ms": [round(v, 5) for v in means],
            "calls_per_rep": [calls] * reps, "copies": n}


def rotation_copies(nbytes: float, l2_bytes: float) -> int:
    """Operand copies for time_rotating: the fewest with (copies - 1) x the
    call's bytes >= 1.5 x the L2 size."""
    return max(2, int(np.ceil(1.5 * l2_bytes / nbytes)) + 1)


def combine_ranks(ms_local: float, flops_per_rank: float, world: int, dist=None, device="cpu"):
    """Replicas only: every rank ran the same workload on its own GPU with no
    exchange. Returns (the slowest rank's ms per step, whole-job GFLOP/s =
    all ranks' flops / that time)."""
    ms = ms_local
    if world > 1 and dist is not None:
        import torch
        t = torch.tensor([ms_local], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    return ms, world * flops_per_rank / (ms * 1e-3) / 1e9


def run_ours(args, rank: int, world: int, local_rank: int):
    import torch
    import implicit_gemm_convolution_gb300 as om
    from implicit_gemm_convolution_gb300 import synth

    om.build()
    om.lib()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    flush = L2Flusher(dev)
    dist = None
    if world > 1:
        import torch.distributed as dist  # noqa: F811

    case = gemm_workload()
    m, n, k = case.m, case.n, case.k
    flops = 2.0 * m * n * k
    A = torch.from_numpy(case.A).to(dev)
    B = torch.from_numpy(case.B).to(dev)
    C = torch.empty((m, n), dtype=torch.float32, device=dev)

    ws = om.new_workspace(dev)

    def step_exact():
        st = om.gemm_raw(m, n, k, A.data_ptr(), k, B.data_ptr(), n, C.data_ptr(), n, "exact", stream,
                         workspace=ws)
        if st != 0:
            raise RuntimeError(f"om_gemm_f32 failed: {om.STATUS_NAMES.get(st, st)}")

    # ---- headline: K timed steps bracketed by barrier + synchronize
    for _ in range(args.warmup):
        flush()
        step_exact()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(local_rank)
    clocks.__enter__()
    region0 = time.time()
    t_wall0 = time.perf_counter()
    kernel_ms = []
    for _ in range(args.steps):
        flush()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        step_exact()
        e1.record(stream)
        e1.synchronize()
        kernel_ms.append(e0.elapsed_time(e1))
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall0
    region1 = time.time()
    clock_summary = clocks.summary(region0, region1)
    clocks.__exit__(None, None, None)
    ms_local = float(np.mean(kernel_ms))
    ms, value = combine_ranks(ms_local, flops, world, dist, dev)
    reps = time_reps(step_exact, flush, stream, args.rep_ms)
    if dist is not None:
        dist.barrier()
    achieved_tflops = flops / (ms_local * 1e-3) / 1e12
    peak_exact = fp32_peak_tflops(sms, exact=True)

    if rank != 0:
        return None

    # ---- end to end through the C ABI with host buffers (pinned), copies timed
    hA = torch.from_numpy(case.A).pin_memory()
    hB = torch.from_numpy(case.B).pin_memory()
    hC = torch.empty((m, n), dtype=torch.float32).pin_memory()
    dA = torch.empty_like(A)
    dB = torch.empty_like(B)

    def e2e_step():
        dA.copy_(hA, non_blocking=True)
        dB.copy_(hB, non_blocking=True)
        st = om.gemm_raw(m, n, k, dA.data_ptr(), k, dB.data_ptr(), n, C.data_ptr(), n, "exact",
                         stream, workspace=ws)
        if st != 0:
            raise RuntimeError("om_gemm_f32 failed")
        hC.copy_(C, non_blocking=True)

    serial_ms = float(np.mean(time_calls(e2e_step, max(2, args.steps // 2), 2, flush, stream)))

    # Pipelined over steps: two device buffer sets; step i's host-to-device
    # copies (one stream) and step i-1's result read-back (another) overlap
    # step i-1's / i's product. Every step still copies its inputs in and its
    # result out inside the timed region.
    h2d, d2h = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    sets = [(torch.empty_like(A), torch.empty_like(B), torch.empty_like(C),
             torch.empty((m, n), dtype=torch.float32).pin_memory()) for _ in range(2)]

    def run_pipelined(steps):
        free = [None, None]  # event: the set's last read-back finished
        for i in range(steps):
            dA_, dB_, C_, hC_ = sets[i % 2]
            if free[i % 2] is not None:
                h2d.wait_event(free[i % 2])
            with torch.cuda.stream(h2d):
                dA_.copy_(hA, non_blocking=True)
                dB_.copy_(hB, non_blocking=True)
            ready = torch.cuda.Event()
            ready.record(h2d)
            stream.wait_event(ready)
            st = om.gemm_raw(m, n, k, dA_.data_ptr(), k, dB_.data_ptr(), n, C_.data_ptr(), n,
                             "exact", stream, workspace=ws)
            if st != 0:
                raise RuntimeError("om_gemm_f32 failed")
            computed = torch.cuda.Event()
            computed.record(stream)
            d2h.wait_event(computed)
            with torch.cuda.stream(d2h):
                hC_.copy_(C_, non_blocking=True)
            free[i % 2] = torch.cuda.Event()
            free[i % 2].record(d2h)
        stream.wait_stream(h2d)
        stream.wait_stream(d2h)

    run_pipelined(3)
    torch.cuda.synchronize()
    e2e_steps = max(4, args.steps // 2)
    p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    p0.record(stream)
    run_pipelined(e2e_steps)
    p1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = p0.elapsed_time(p1) / e2e_steps
    e2e = {"value": round(flops / (e2e_ms * 1e-3) / 1e9, 1), "unit": "GFLOP/s",
           "h2d_bytes_per_step": int(hA.numel() * 4 + hB.numel() * 4),
           "d2h_bytes_per_step": int(hC.numel() * 4), "ms_per_step": round(e2e_ms, 4),
           "steps": e2e_steps,
           "how": "pinned host A, B in and C out every step, on two copy streams that overlap "
                  "the neighbouring steps' products (two device buffer sets)",
           "serial_ms_per_step": round(serial_ms, 4),
           "serial_value": round(flops / (serial_ms * 1e-3) / 1e9, 1)}

    # ---- per-mode and per-workload lines (same timing rules)
    extras = {}

    wsp = om.new_workspace(dev)
    l2_bytes = float(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or 129e6)

    def with_traffic(name, traffic):
        """DRAM bytes per launch of the line's kernel from the committed ncu
        capture of the same workload (None when that capture is older than the
        kernel's sources)."""
        if traffic is not None:
            extras[name]["traffic"] = recorded_traffic(*traffic)
            extras[name]["traffic_source"] = f"{traffic[0]} {traffic[1]}, profiles/dram_traffic.txt"

    def gemm_line(name, mode, case_, use_ws=False, hbm_bound=False, traffic=None):
        def make(Ad, Bd, Cd):
            def f():
                st = om.gemm_raw(case_.m, case_.n, case_.k, Ad.data_ptr(), case_.lda, Bd.data_ptr(),
                                 case_.ldb, Cd.data_ptr(), case_.ldc, mode, stream,
                                 workspace=wsp if use_ws else None)
                if st != 0:
                    raise RuntimeError(f"{name}: {om.STATUS_NAMES.get(st, st)}")
            return f
        ops = (torch.from_numpy(case_.A).to(dev), torch.from_numpy(case_.B).to(dev),
               torch.from_numpy(case_.C_init).to(dev))
        t0 = time.time()
        r = time_reps(make(*ops), flush, stream, args.rep_ms)
        t = r["ms"]
        fl = 2.0 * case_.m * case_.n * case_.k
        tf = fl / (t * 1e-3) / 1e12
        pk = fp32_peak_tflops(sms, exact=(mode == "exact"))
        extras[name] = {"ms": round(t, 4), "GFLOP/s": round(tf * 1e3, 1),
                        "roofline_frac": round(tf / pk, 4), "peak_tflops": round(pk, 2),
                        "rep_ms": r["rep_ms"], "calls_per_rep": r["calls_per_rep"]}
        nbytes = 4.0 * (case_.m * case_.k + case_.k * case_.n + case_.m * case_.n)
        copies = [ops] + [tuple(torch.empty_like(o).copy_(o) for o in ops)
                          for _ in range(rotation_copies(nbytes, l2_bytes) - 1)]
        rr = time_rotating([make(*o) for o in copies], stream, args.rep_ms)
        del copies
        if hbm_bound:
            extras[name].update(hbm_fields(nbytes, t, rr))
        else:
            extras[name].update(in_a_row_fields(fl, pk, nbytes, rr))
        with_traffic(name, traffic)
        extras[name]["clocks"] = line_clocks(t0)

    def hbm_fields(nbytes, t_flushed, rot):
        """Algorithmic bytes (each operand read once, the output written once)
        against the measured copy bandwidth, for HBM-bound kernels. The
        figure is taken from calls in a row rotating over operand copies
        larger than L2 (time_rotating); the per-call figure with L2 flushed
        before each call, which adds the launch latency and the write-back of
        the flush's dirty lines to every call, is kept beside it."""
        gbs = nbytes / (rot["ms"] * 1e-3) / 1e9
        hbm = measured_peaks()["hbm_gbs"]
        gbs_f = nbytes / (t_flushed * 1e-3) / 1e9
        return {"bound": "hbm", "ms_in_a_row": round(rot["ms"], 4), "GB/s": round(gbs, 1),
                "hbm_frac": round(gbs / hbm, 4), "hbm_peak_gbs": hbm, "algorithmic_bytes": int(nbytes),
                "timing": f"calls in a row over {rot['copies']} operand copies of {nbytes / 1e6:.0f} MB "
                          f"each (L2 {l2_bytes / 1e6:.0f} MB), no flush; median of 3 repetitions "
                          f"of >= {args.rep_ms:.0f} ms",
                "rep_ms_in_a_row": rot["rep_ms"],
                "GB/s_flushed_per_call": round(gbs_f, 1), "hbm_frac_flushed_per_call": round(gbs_f / hbm, 4)}

    def in_a_row_fields(flops_, peak_tflops, nbytes, rot):
        """The same line timed as calls in a row (the pages' benchmark method:
        back-to-back calls bracketed by CUDA events) over operand copies larger
        than L2 together (time_rotating): no flush, and the launch latency
        overlaps the previous call as for a caller issuing calls in a row."""
        tf_ = flops_ / (rot["ms"] * 1e-3) / 1e12
        return {"ms_in_a_row": round(rot["ms"], 4), "GFLOP/s_in_a_row": round(tf_ * 1e3, 1),
                "roofline_frac_in_a_row": round(tf_ / peak_tflops, 4),
                "rep_ms_in_a_row": rot["rep_ms"],
                "in_a_row": f"{rot['copies']} operand copies of {nbytes / 1e6:.1f} MB "
                            f"(L2 {l2_bytes / 1e6:.0f} MB), median of 3 repetitions of >= {args.rep_ms:.0f} ms"}

    clock_log = ClockSampler(local_rank)
    clock_log.__enter__()

    def line_clocks(t0):
        c = clock_log.summary(t0, time.time())
        return {"sm_mhz": c["sm_mhz"], "reasons": c["reasons"], "samples": c["samples"]}

    def tf32x3_line(name, case_, traffic=None):
        Ad = torch.from_numpy(case_.A).to(dev)
        Bd = torch.from_numpy(case_.B).to(dev)
        Cd = torch.from_numpy(case_.C_init).to(dev)

        def f():
            st = om.gemm_raw(case_.m, case_.n, case_.k, Ad.data_ptr(), case_.lda, Bd.data_ptr(),
                             case_.ldb, Cd.data_ptr(), case_.ldc, "tf32x3", stream)
            if st != 0:
                raise RuntimeError(f"{name}: {om.STATUS_NAMES.get(st, st)}")
        t0 = time.time()
        r = time_reps(f, flush, stream, args.rep_ms)
        t = r["ms"]
        fl = 2.0 * case_.m * case_.n * case_.k
        tf = fl / (t * 1e-3) / 1e12
        peaks = measured_peaks()
        tf32_peak = peaks["bf16_tflops"] * TF32_PER_BF16
        extras[name] = {"ms": round(t, 4), "GFLOP/s": round(tf * 1e3, 1),
                        "vs_fp32_fma_peak": round(tf / fp32_peak_tflops(sms, exact=False), 3),
                        "tensor_frac": round(3 * tf / tf32_peak, 4),
                        "tensor_peak_tflops": round(tf32_peak, 1),
                        "tensor_peak_basis": peaks["basis"] + " x nominal tf32/bf16 ratio 1.1/2.25; "
                                             "three tensor-core products per useful flop",
                        "rep_ms": r["rep_ms"], "calls_per_rep": r["calls_per_rep"],
                        "clocks": line_clocks(t0)}
        with_traffic(name, traffic)

    def conv_line(name, mode, c, use_ws=False, hbm_bound=False, traffic=None):
        OH = om.conv_out_dim(c.H, c.KH, c.stride, c.pad, c.dil)
        OW = om.conv_out_dim(c.W, c.KW, c.stride, c.pad, c.dil)
        L = om.lib()

        def make(x, w, y):
            def f():
                args_ = (c.N, c.Cin, c.H, c.W, c.Cout, c.G, c.KH, c.KW, c.stride, c.pad, c.dil,
                         x.data_ptr(), w.data_ptr(), y.data_ptr(), om.MODES[mode])
                if use_ws:
                    st = L.om_conv2d_f32_ws(*args_, wsp.data_ptr(), om.workspace_bytes(),
                                            stream.cuda_stream)
                else:
                    st = L.om_conv2d_f32(*args_, stream.cuda_stream)
                if st != 0:
                    raise RuntimeError(f"{name}: {om.STATUS_NAMES.get(st, st)}")
            return f
        ops = (torch.from_numpy(c.x).to(dev), torch.from_numpy(c.w).to(dev),
               torch.empty((c.N, c.Cout, OH, OW), dtype=torch.float32, device=dev))
        t0 = time.time()
        r = time_reps(make(*ops), flush, stream, args.rep_ms)
        t = r["ms"]
        fl = 2.0 * c.N * c.Cout * OH * OW * (c.Cin // c.G) * c.KH * c.KW
        tf = fl / (t * 1e-3) / 1e12
        pk = fp32_peak_tflops(sms, exact=(mode == "exact"))
        extras[name] = {"ms": round(t, 4), "GFLOP/s": round(tf * 1e3, 1),
                        "roofline_frac": round(tf / pk, 4), "peak_tflops": round(pk, 2),
                        "rep_ms": r["rep_ms"], "calls_per_rep": r["calls_per_rep"]}
        nbytes = 4.0 * (c.x.size + c.w.size + c.N * c.Cout * OH * OW)
        copies = [ops] + [tuple(torch.empty_like(o).copy_(o) for o in ops)
                          for _ in range(rotation_copies(nbytes, l2_bytes) - 1)]
        rr = time_rotating([make(*o) for o in copies], stream, args.rep_ms)
        del copies
        if hbm_bound:
            extras[name].update(hbm_fields(nbytes, t, rr))
        else:
            extras[name].update(in_a_row_fields(fl, pk, nbytes, rr))
        with_traffic(name, traffic)
        extras[name]["clocks"] = line_clocks(t0)

    def chain_line(name, mode):
        """ResNet-50's 53 convolutions at 224 x 224, batch 1, each with its
        bias / shortcut / ReLU epilogue: one CUDA-graph replay per step, and
        the same chain called layer by layer from the host."""
        from implicit_gemm_convolution_gb300 import chain
        ch = chain.ConvChain(chain.resnet50_convs(), 1, 224, mode, device=dev)
        graph = ch.capture()
        t0 = time.time()
        t_graph = time_reps(graph.replay, flush, stream, args.rep_ms)["ms"]
        t_eager = time_reps(ch.run, flush, stream, args.rep_ms)["ms"]
        tf = ch.flops / (t_graph * 1e-3) / 1e12
        pk = fp32_peak_tflops(sms, exact=(mode == "exact"))
        extras[name] = {"ms": round(t_graph, 4), "ms_eager_host_calls": round(t_eager, 4),
                        "GFLOP/s": round(tf * 1e3, 1), "roofline_frac": round(tf / pk, 4),
                        "peak_tflops": round(pk, 2), "layers": len(ch.layers),
                        "gflop": round(ch.flops / 1e9, 3),
                        "context": "the pages' ResNet-50 convolution chain, 16/32 CPU threads on a "
                                   "16-core Zen 4: 12.3/11.1 ms (other hardware)",
                        "clocks": line_clocks(t0)}

    if not args.headline_only:
        SG, CI, CR = "sgemm_tiled_kernel", "conv_implicit_kernel", "conv_rows_kernel"
        gemm_line("gemm_4096^3_fast_ws", "fast", case, use_ws=True, traffic=(SG, "gemm_4096^3_fast"))
        gemm_line("gemm_4096^3_exact_no_workspace", "exact", case)
        gemm_line("gemm_4096^3_fast_no_workspace", "fast", case)
        tf32x3_line("gemm_4096^3_tf32x3", case, traffic=("gemm_tf32x3_kernel", "gemm_4096^3_tf32x3"))
        gemm_line("gemm_prefill_512x11008x4096_exact_ws", "exact",
                  synth.workload_gemm_prefill(False), use_ws=True)
        gemm_line("gemm_prefill_509x11005x4096_exact_ws", "exact",
                  synth.workload_gemm_prefill(True), use_ws=True)
        gemm_line("gemm_prefill_512x11008x4096_fast_ws", "fast",
                  synth.workload_gemm_prefill(False), use_ws=True)
        gemm_line("gemm_prefill_509x11005x4096_fast_ws", "fast",
                  synth.workload_gemm_prefill(True), use_ws=True, traffic=(SG, "gemm_prefill_ragged_fast"))
        for md in ("exact", "fast"):
            conv_line(f"conv3x3_n32_c64_56_{md}_ws", md, synth.workload_conv3x3(), use_ws=True,
                      traffic=(CR, f"conv3x3_{md}"))
            conv_line(f"conv1x1_n32_c256to64_56_{md}_ws", md, synth.workload_conv1x1(), use_ws=True,
                      traffic=(CI, f"conv1x1_{md}"))
        conv_line("conv_g32_s2_d2_n16_c256_28_exact_ws", "exact", synth.workload_conv_grouped(),
                  use_ws=True)
        gemm_line("gemm_prefill_512x11008x4096_exact", "exact", synth.workload_gemm_prefill(False))
        gemm_line("gemm_prefill_509x11005x4096_exact", "exact", synth.workload_gemm_prefill(True))
        gemm_line("gemm_prefill_512x11008x4096_fast", "fast", synth.workload_gemm_prefill(False))
        gemm_line("gemm_prefill_509x11005x4096_fast", "fast", synth.workload_gemm_prefill(True))
        for md in ("exact", "fast"):
            conv_line(f"conv3x3_n32_c64_56_{md}", md, synth.workload_conv3x3())
            conv_line(f"conv1x1_n32_c256to64_56_{md}", md, synth.workload_conv1x1())
        conv_line("conv_g32_s2_d2_n16_c256_28_exact", "exact", synth.workload_conv_grouped(),
                  traffic=("conv_group_kernel", "conv_grouped_exact"))
        conv_line("conv_g32_s2_d2_n16_c256_28_fast", "fast", synth.workload_conv_grouped())
        for md in ("exact", "fast"):
            conv_line(f"conv_dw3x3_n32_c256_56_{md}", md, synth.workload_conv_depthwise(),
                      hbm_bound=True, traffic=("conv_dw_tma_kernel", f"conv_depthwise_{md}"))
            gemm_line(f"gemm_decode_1x11008x4096_{md}", md, synth.workload_gemm_decode(),
                      hbm_bound=True, traffic=("gemv_kernel", f"gemm_decode_{md}"))
        for md in ("exact", "fast"):
            conv_line(f"conv_late3x3_n1_c512_7_{md}", md, synth.workload_conv_late3x3())
        for md in ("exact", "fast"):
            chain_line(f"resnet50_conv_chain_b1_224_{md}", md)

    clock_log.__exit__(None, None, None)
    cpu = cpu_baseline(args.cpu_seconds)
    line = {
        "metric": "GFLOP/s and % of FP32 CUDA-core roofline per mode (GEMM 4096^3; conv3x3)",
        "value": round(value, 1),
        "unit": "GFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded SplitMix64, N(0,1) operands)",
        "config": {"workload": "gemm_4096^3", "m": m, "n": n, "k": k, "mode": "exact",
                   "entry_point": "om_gemm_f32_ws",
                   "layout": "row-major contiguous", "l2": "flushed before every timed call",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": {"bound": "alu", "achieved": round(achieved_tflops, 3),
                     "peak": round(peak_exact, 3), "unit": "TFLOP/s",
                     "frac": round(achieved_tflops / peak_exact, 4),
                     "traffic": recorded_traffic("sgemm_tiled_kernel", "gemm_4096^3_exact"),
                     "peak_basis": f"derived: {sms} SMs x 128 FP32 lanes x 2 flops x {SM_MAX_MHZ:.0f} MHz / 2 "
                                   "(exact mode issues a multiply and an add per term)"},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": args.steps,
        "clocks": clock_summary,
        "wall_s_timed_region": round(t_wall, 3),
        "repetitions": {"ms_median": round(reps["ms"], 4),
                        "GFLOP/s": round(flops / (reps["ms"] * 1e-3) / 1e9, 1),
                        "rep_ms": reps["rep_ms"], "calls_per_rep": reps["calls_per_rep"],
                        "method": f"after the timed steps: 3 repetitions of calls totalling >= "
                                  f"{args.rep_ms:.0f} ms of device time each (L2 flushed before "
                                  "every call), median of the repetitions' mean call times"},
        "modes": extras,
    }
    return line


def _cpu_rate(run, flops: float, min_s: float, reps: int = 3, warmup: int = 2) -> dict:
    """The pages' benchmark method on the host: warm-up calls, then
    repetitions of back-to-back calls lasting at least min_s each; the
    figure is the median of the repetitions' rates."""
    for _ in range(warmup):
        run()
    rates = []
    for _ in range(reps):
        calls, t0 = 0, time.perf_counter()
        while True:
            run()
            calls += 1
            el = time.perf_counter() - t0
            if el >= min_s:
                break
        rates.append(flops * calls / el / 1e9)
    return {"gflops": float(np.median(rates)), "rates": [round(r, 4) for r in rates]}


def cpu_baseline_cases():
    """(name, full-workload flops, {threads-kind: (sample runner factory, sample flops, text)})
    for every benchmark configuration. Samples are whole output rows of a
    product, or whole images / output channels of a convolution: every
    output is independent, so a sample's rate stands for the workload's."""
    from implicit_gemm_convolution_gb300 import synth
    import oracle

    def gemm_rows(case, rows):
        A = np.ascontiguousarray(case.A[:rows])
        C = np.ascontiguousarray(case.C_init[:rows]).copy()

        def mk(mode, threads):
            return lambda: oracle.gemm_raw(rows, case.n, case.k, A, case.lda, case.B, case.ldb, C,
                                           case.ldc, mode, threads)
        return mk, 2.0 * rows * case.n * case.k

    def conv_part(c, images, out_channels):
        x = np.ascontiguousarray(c.x[:images])
        w = np.ascontiguousarray(c.w[:out_channels])
        OH = (c.H + 2 * c.pad - c.dil * (c.KH - 1) - 1) // c.stride + 1
        OW = (c.W + 2 * c.pad - c.dil * (c.KW - 1) - 1) // c.stride + 1

        def mk(mode, threads):
            return lambda: oracle.conv2d(x, w, c.stride, c.pad, c.dil, c.G, mode, threads)
        return mk, 2.0 * images * out_channels * OH * OW * (c.Cin // c.G) * c.KH * c.KW

    def conv_full_flops(c):
        OH = (c.H + 2 * c.pad - c.dil * (c.KH - 1) - 1) // c.stride + 1
        OW = (c.W + 2 * c.pad - c.dil * (c.KW - 1) - 1) // c.stride + 1
        return 2.0 * c.N * c.Cout * OH * OW * (c.Cin // c.G) * c.KH * c.KW

    T = oracle.default_threads()
    out = []
    small = synth.workload_gemm_small_strided()
    mk, fl = gemm_rows(small, small.m)
    out.append(("gemm_67x53x300_strided", fl, {"1": (mk, fl, "whole product"),
                                               "all": (mk, fl, "whole product")}))
    for name, case in (("gemm_4096^3", synth.workload_gemm_4096()),
                       ("gemm_prefill_512x11008x4096", synth.workload_gemm_prefill(False)),
                       ("gemm_prefill_509x11005x4096", synth.workload_gemm_prefill(True))):
        full = 2.0 * case.m * case.n * case.k
        m1, f1 = gemm_rows(case, 1)
        mT, fT = gemm_rows(case, T)
        out.append((name, full, {"1": (m1, f1, f"1 of {case.m} rows"),
                                 "all": (mT, fT, f"{T} of {case.m} rows")}))
    c3 = synth.workload_conv3x3()
    m1, f1 = conv_part(c3, 1, 8)
    mT, fT = conv_part(c3, 1, c3.Cout)
    out.append(("conv3x3_n32_c64_56", conv_full_flops(c3),
                {"1": (m1, f1, "image 0, output channels 0-7"),
                 "all": (mT, fT, "image 0, all 64 output channels")}))
    c1 = synth.workload_conv1x1()
    m1, f1 = conv_part(c1, 1, 16)
    mT, fT = conv_part(c1, 1, c1.Cout)
    out.append(("conv1x1_n32_c256to64_56", conv_full_flops(c1),
                {"1": (m1, f1, "image 0, output channels 0-15"),
                 "all": (mT, fT, "image 0, all 64 output channels")}))
    cg = synth.workload_conv_grouped()
    m1, f1 = conv_part(cg, 1, cg.Cout)
    mT, fT = conv_part(cg, cg.N, cg.Cout)
    out.append(("conv_g32_s2_d2_n16_c256_28", conv_full_flops(cg),
                {"1": (m1, f1, "image 0 of 16"), "all": (mT, fT, "all 16 images")}))
    return out


def cpu_baseline(seconds: float) -> dict:
    """The oracle as it stands on the host cores, for every benchmark
    configuration in both bit-exact modes, on one thread and on all cores
    (OpenMP over output rows / (image, channel) pairs). Each figure is the
    median of three repetitions of at least max(80 ms, ``seconds``/150 s) of back-to-back
    calls on a sample of the workload; samples smaller than the whole
    workload are labelled extrapolated (the full workload's time is its flops
    over the sample's rate). The headline figure (``value``) is the 4096-cube
    product in exact mode on all cores."""
    import oracle
    oracle.build()
    threads = oracle.default_threads()
    min_s = max(0.08, seconds / 150.0)
    rows = []
    t_start = time.perf_counter()
    for name, full, kinds in cpu_baseline_cases():
        for mode_name, mode in (("exact", oracle.EXACT), ("fast", oracle.FAST)):
            for kind, nthreads in (("1", 1), ("all", threads)):
                mk, fl, text = kinds[kind]
                r = _cpu_rate(mk(mode, nthreads), fl, min_s)
                rows.append({"workload": name, "mode": mode_name, "threads": nthreads,
                             "GFLOP/s": round(r["gflops"], 4),
                             "full_ms": round(full / (r["gflops"] * 1e9) * 1e3, 2),
                             "extrapolated": fl < full, "sample": text,
                             "rep_GFLOP/s": r["rates"]})
    head = next(r for r in rows if r["workload"] == "gemm_4096^3" and r["mode"] == "exact"
                and r["threads"] == threads)
    return {"value": head["GFLOP/s"], "unit": "GFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"exact mode, {head['sample']} of the 4096^3 product, all {threads} cores; "
                      "median of 3 repetitions of back-to-back calls "
                      f"(>= {min_s * 1e3:.0f} ms each) after 2 warm-up calls",
            "per_workload": rows,
            "wall_s": round(time.perf_counter() - t_start, 2)}


def run_reference(args, rank: int):
    if rank != 0:
        return None
    import oracle
    oracle.build()
    case = gemm_workload()
    threads = oracle.default_threads()
    rows = max(threads, 16)
    A = case.A[:rows].copy()
    Cs = np.zeros((rows, case.n), np.float32)

    def step():
        oracle.gemm_raw(rows, case.n, case.k, A, case.k, case.B, case.n, Cs, case.n, oracle.EXACT,
                        threads)
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    val = 2.0 * rows * case.n * case.k / dt / 1e9
    sample = f"exact mode, {rows} of 4096 rows of the 4096^3 product per step"
    return {"impl": "reference", "metric": "GFLOP/s and % of FP32 CUDA-core roofline per mode (GEMM 4096^3; conv3x3)",
            "value": round(val, 3), "unit": "GFLOP/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded SplitMix64, N(0,1) operands)",
            "config": {"workload": "gemm_4096^3", "m": 4096, "n": 4096, "k": 4096, "mode": "exact"},
            "cpu_baseline": {"value": round(val, 3), "unit": "GFLOP/s", "cores": threads,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(val, 3), "unit": "GFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def run_profile(args):
    """Only the named workload's kernel launches (warm-up, then --steps), for
    ncu captures: no L2 flush kernels, no extra workloads, no host baseline."""
    import torch
    import implicit_gemm_convolution_gb300 as om
    from implicit_gemm_convolution_gb300 import synth
    om.build()
    L = om.lib()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    name, mode = args.profile.split(":")[:2]
    gemms = {"gemm_4096^3": synth.workload_gemm_4096,
             "gemm_prefill": lambda: synth.workload_gemm_prefill(False),
             "gemm_prefill_ragged": lambda: synth.workload_gemm_prefill(True),
             "gemm_decode": synth.workload_gemm_decode}
    convs = {"conv3x3": synth.workload_conv3x3, "conv1x1": synth.workload_conv1x1,
             "conv_grouped": synth.workload_conv_grouped,
             "conv_depthwise": synth.workload_conv_depthwise,
             "conv_late3x3": synth.workload_conv_late3x3}
    if name in gemms:
        case = gemms[name]()
        A = torch.from_numpy(case.A).to(dev)
        B = torch.from_numpy(case.B).to(dev)
        C = torch.from_numpy(case.C_init).to(dev)

        ws = om.new_workspace(dev)

        def f():
            st = om.gemm_raw(case.m, case.n, case.k, A.data_ptr(), case.lda, B.data_ptr(),
                             case.ldb, C.data_ptr(), case.ldc, mode, stream, workspace=ws)
            assert st == 0, st
    else:
        c = convs[name]()
        x = torch.from_numpy(c.x).to(dev)
        w = torch.from_numpy(c.w).to(dev)
        OH = om.conv_out_dim(c.H, c.KH, c.stride, c.pad, c.dil)
        OW = om.conv_out_dim(c.W, c.KW, c.stride, c.pad, c.dil)
        y = torch.empty((c.N, c.Cout, OH, OW), dtype=torch.float32, device=dev)

        ws = om.new_workspace(dev)

        def f():
            st = L.om_conv2d_f32_ws(c.N, c.Cin, c.H, c.W, c.Cout, c.G, c.KH, c.KW, c.stride,
                                    c.pad, c.dil, x.data_ptr(), w.data_ptr(), y.data_ptr(),
                                    om.MODES[mode], ws.data_ptr(), om.workspace_bytes(),
                                    stream.cuda_stream)
            assert st == 0, st
    for _ in range(args.warmup + args.steps):
        f()
    torch.cuda.synchronize()
    print(json.dumps({"profile": args.profile, "launches": args.warmup + args.steps}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--rep-ms", type=float, default=80.0,
                    help="device time per repetition of the per-workload lines (median of 3)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="scales the host baseline repetition length (max(80 ms, seconds/150) per repetition)")
    ap.add_argument("--headline-only", action="store_true")
    ap.add_argument("--profile", default=None,
                    help="workload:mode (gemm_4096^3, gemm_prefill, gemm_prefill_ragged, gemm_decode,"
                         " conv3x3, conv1x1, conv_grouped, conv_depthwise, conv_late3x3) -- launch"
                         " only that kernel, for ncu")
    args = ap.parse_args()
    if args.profile:
        run_profile(args)
        return
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        line = run_reference(args, rank)
    else:
        if world > 1:
            import torch
            import torch.distributed as dist
            torch.cuda.set_device(local_rank)
            dist.init_process_group("nccl")
        line = run_ours(args, rank, world, local_rank)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
