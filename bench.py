#!/usr/bin/env python3
"""Throughput of the GB300 fp16 NT GEMM, C[M,N] = A[M,K] · B[N,K]ᵀ.

One step = one call of the C-ABI entry point `gemm_f16_nt` on the whole
workload (default: M = N = K = 8192, the shape the Tilus matmul-hopper tutorial
measures in every version; inputs uniform in [-1, 1], rounded to fp16, seeded).
The timed region holds only that kernel, back to back on one stream, with the
operands resident in HBM; A, B and C together (384 MiB at 8192³) are larger
than the 129 MB L2, so no step finds its operands in L2 from the step before.
Each launch may start its set-up while the one before drains (programmatic
dependent launch), as in any chain of GEMMs on one stream; it reads no operand
before the previous launch has finished.

Printed: one JSON line with the throughput (TFLOP/s = 2·M·N·K / time), the
roofline fraction of the GEMM kernel against the measured dense 16-bit tensor
peak, an end-to-end figure through the same C ABI from pinned host memory, the
clocks seen during the timed region, and the CPU oracle timed on a bounded
sample of the same workload.  Beside the headline, on rank 0: every other
workload (256³, 4096³, the ragged shape with float and integer inputs, the MLP
shape) timed the same way through the C ABI, each with cuBLAS beside it and its
own clock record ("workloads"); three small, latency-bound shapes (1024³,
512×4096×4096, 256×256×4096) the same way ("small_shapes"); and a sustained
window of back-to-back 8192³ launches lasting seconds, long enough for the
board's power cap to set the clock ("sustained").  Workloads whose operands
fit in L2 are timed with a flush before each launch; they also report the GPU
time a launch adds after a flush (a difference of long event-timed regions,
free of the per-launch events' resolution).  Last, the timing protocol of
the Tilus pages: the headline again in three fresh processes, each after 3 s
of idle, and their median ("fresh_processes").

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

For N > 1 (under torchrun, one process per GPU) every rank runs an independent
replica of the workload: the product is a single-GPU library and the multiply
needs no exchange between GPUs.  The slowest rank's time sets the figure.
`--impl reference` times the CPU oracle instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from dense_fp16_gemm_gb300 import inputs  # noqa: E402

METRIC = "fp16 NT GEMM TFLOP/s and % of GB300 dense fp16 tensor peak"
UNIT = "TFLOP/s"
# The persistent kernel's device sources (the traffic records are of that
# kernel; gemm_f16_nt.cu is host code, small_tile.cuh the small-problem kernel)
KERNEL_SOURCES = ["dense_fp16_gemm_gb300/csrc/persistent.cuh", "dense_fp16_gemm_gb300/csrc/ptx.cuh",
                  "dense_fp16_gemm_gb300/csrc/sched.cuh"]
# DRAM bytes per launch from an Nsight Compute capture, written by
# `bench.py --record-traffic`; used only while the kernel sources hash the same
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.json")
SIDE_WORKLOADS = ["gemm_256", "gemm_4096", "ragged_4000x3000x5000", "ragged_int_4000x3000x5000",
                  "mlp_up_16384x14336x4096"]
# small, latency-bound shapes beside the configs (the small-problem kernel's range)
SMALL_SHAPES = ["gemm_1024", "gemm_512x4096x4096", "gemm_256x256x4096"]
FALLBACK_PEAK_TFLOPS = 1900.0   # one earlier GB300 bf16 burst measurement
L2_BYTES = 129 * 10**6
SMI_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


# ---------------------------------------------------------------------------
# distributed plumbing (replicas only)
# ---------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world: int, backend: str):
    if world <= 1:
        return None
    import torch.distributed as dist
    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    if not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist


def barrier(dist, device=None):
    if dist is None:
        return
    if device is not None and dist.get_backend() == "nccl":
        dist.barrier(device_ids=[device.index])
    else:
        dist.barrier()


def reduce_time_and_work(dist, seconds: float, work: float, device=None):
    """(max seconds over ranks, sum of work over ranks)."""
    if dist is None:
        return seconds, work
    import torch
    dev = device if (device is not None and dist.get_backend() == "nccl") else "cpu"
    t = torch.tensor([seconds], dtype=torch.float64, device=dev)
    w = torch.tensor([work], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(w, op=dist.ReduceOp.SUM)
    return float(t.item()), float(w.item())


# ---------------------------------------------------------------------------
# peaks, traffic record, clocks
# ---------------------------------------------------------------------------

def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(path))
        return float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", 0) or 0), "measured"
    except Exception:
        return FALLBACK_PEAK_TFLOPS, 0.0, "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """(DRAM bytes per launch, record) from the machine-readable record of an
    Nsight Compute capture of this workload, if that capture was taken on the
    current kernel sources; else (None, None).  The figure is recorded, not
    measured by this run, and the JSON line says so."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f).get(workload)
    except (OSError, ValueError):
        return None, None
    if not rec or rec.get("kernel_source_sha256_16") != kernel_source_hash():
        return None, None
    try:
        return int(rec["dram_bytes_per_launch"]), rec
    except (KeyError, ValueError, TypeError):
        return None, None


def record_traffic(rep_path: str, workload: str, command: str):
    """Read dram__bytes_{read,write}.sum of the GEMM launches in an Nsight
    Compute report (ncu -i … --page raw --csv) and store their mean per launch
    for `workload` in the traffic record, keyed by the kernel-source hash."""
    import csv
    import io
    out = subprocess.run(["ncu", "-i", rep_path, "--page", "raw", "--csv"], capture_output=True, text=True,
                         check=True).stdout
    rows = list(csv.reader(io.StringIO(out)))
    head = rows[0]
    col = {n: i for i, n in enumerate(head)}
    units = rows[1]
    scale = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9}
    per = []
    for r in rows[2:]:
        if "gemm_f16_nt_kernel" not in r[col["Kernel Name"]]:
            continue
        b = 0.0
        for m in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
            b += float(r[col[m]].replace(",", "")) * scale[units[col[m]]]
        per.append(b)
    if not per:
        raise SystemExit(f"no gemm_f16_nt_kernel launch in {rep_path}")
    try:
        with open(TRAFFIC_FILE) as f:
            data = json.load(f)
    except (OSError, ValueError):
        data = {}
    data[workload] = {"dram_bytes_per_launch": int(round(sum(per) / len(per))), "launches": len(per),
                      "kernel_source_sha256_16": kernel_source_hash(), "command": command,
                      "metrics": "dram__bytes_read.sum + dram__bytes_write.sum"}
    with open(TRAFFIC_FILE, "w") as f:
        json.dump(data, f, indent=1, sort_keys=True)
        f.write("\n")
    print(json.dumps(data[workload]))


class ClockSampler:
    """Samples the SM clock, its maximum, board power (NVML's one-second
    average) and the clock-event (throttle) reasons while the timed region runs.  Reads only: it queries
    NVML through ctypes (libnvidia-ml ships with the driver) every few ms from a
    background thread, and falls back to `nvidia-smi -lms` if NVML cannot be
    loaded.  Each sample carries a host timestamp so that only samples taken
    inside a timed window are summarised."""

    # clock-event reason bits of the NVML API
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, gpu_index: int, period_s: float = 0.005):
        import threading
        self.samples = []          # (t, sm_mhz, max_mhz, power_w, reason_bits)
        self.windows = []
        self._stop = threading.Event()
        self._smi = None
        self._nvml = self._open_nvml(gpu_index)
        if self._nvml is not None:
            self._thread = threading.Thread(target=self._poll, args=(period_s,), daemon=True)
            self._thread.start()
        else:
            self._thread = None
            self._start_smi(gpu_index)

    def _open_nvml(self, idx):
        import ctypes
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return None
            h = ctypes.c_void_p()
            if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(idx), ctypes.byref(h)) != 0:
                return None
            return lib, h
        except OSError:
            return None

    def _take(self):
        """One NVML sample (clock, max clock, power, reason bits), timestamped."""
        import ctypes
        lib, h = self._nvml
        mhz, mx, mw = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_uint()
        bits = ctypes.c_ulonglong()
        get_reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
        t = time.time()
        if lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(mhz)) == 0 and \
                lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
            pw = mw.value / 1e3 if lib.nvmlDeviceGetPowerUsage(h, ctypes.byref(mw)) == 0 else 0.0
            rb = bits.value if get_reasons(h, ctypes.byref(bits)) == 0 else 0
            self.samples.append((t, float(mhz.value), float(mx.value), pw, int(rb)))

    def sample_now(self):
        """Take a sample from the calling thread: called while launches the host
        has already enqueued keep the GPU busy, so that even a timed region of a
        few milliseconds holds at least one sample."""
        if self._nvml is not None:
            self._take()

    def _poll(self, period):
        while not self._stop.is_set():
            self._take()
            time.sleep(period)

    def _start_smi(self, idx):
        self._f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self._smi = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu=timestamp,{SMI_FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(idx), "-lms", "50"], stdout=self._f, stderr=subprocess.DEVNULL)
        except OSError:
            self._smi = None

    def window(self, t0: float, t1: float):
        self.windows.append((t0, t1))

    def summary_for(self, t0: float, t1: float):
        """Clock summary of the samples inside one wall window (after stop())."""
        return self.summary([(t0, t1)])

    def stop(self):
        self._stop.set()
        if self._thread is not None:
            self._thread.join(timeout=5)
        if self._smi is not None:
            import datetime
            self._smi.terminate()
            try:
                self._smi.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self._smi.kill()
            self._f.flush()
            self._f.seek(0)
            names = {5: 0x8, 6: 0x40, 7: 0x20, 8: 0x4}
            for line in self._f.read().splitlines():
                r = [x.strip() for x in line.split(",")]
                if len(r) < 10:
                    continue
                try:
                    t = datetime.datetime.strptime(r[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    rb = sum(bit for col, bit in names.items() if r[col + 1].lower() == "active")
                    self.samples.append((t, float(r[2]), float(r[3]), float(r[4]), rb))
                except ValueError:
                    continue
            self._f.close()
            os.unlink(self._f.name)
        return self.summary()

    def summary(self, windows=None):
        windows = self.windows if windows is None else windows
        inside = [s for s in self.samples if any(a <= s[0] <= b for a, b in windows)]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "source": "nvml" if self._nvml else "nvidia-smi"}
        reasons = set()
        for s in inside:
            reasons |= {name for bit, name in self.REASONS.items() if s[4] & bit}
        return {"sm_mhz": statistics.median(s[1] for s in inside),
                "sm_mhz_min": min(s[1] for s in inside),
                "sm_max_mhz": max(s[2] for s in inside), "reasons": sorted(reasons),
                "samples": len(inside),
                # NVML reports board power averaged over the last second, so a
                # region shorter than that also counts the idle time before it
                "power_w_1s_average_median": statistics.median(s[3] for s in inside),
                "source": "nvml" if self._nvml else "nvidia-smi"}


# ---------------------------------------------------------------------------
# CPU oracle leg (the reported baseline)
# ---------------------------------------------------------------------------

def cpu_model() -> str:
    """The host CPU's model name, as the kernel reports it."""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key, _, val = line.partition(":")
                if key.strip().lower() in ("model name", "cpu model", "hardware") and val.strip():
                    return val.strip()
    except OSError:
        pass
    try:   # Arm hosts list no model name in /proc/cpuinfo; lscpu decodes the part number
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            key, _, val = line.partition(":")
            if key.strip() == "Model name" and val.strip():
                return val.strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return platform.processor() or platform.machine()


def l2_to_sm_bytes(pl) -> int:
    """Operand bytes the plan delivers into shared memory: every cluster tile
    receives, over the whole k range, its B rows and, in each of its CTA
    pairs, the tile's A rows (with two pairs A is read from L2 once and
    multicast, but received twice)."""
    tiles, kb = pl["num_tiles"], pl["k_blocks"]
    return int(tiles * kb * 64 * 2 * (pl["tile_m"] * pl["cluster_pairs"] + pl["tile_n"]))


def oracle_fn(acc16: bool, bf16: bool = False):
    """The oracle function matching the arm's arithmetic."""
    import oracle
    if bf16:
        return oracle.gemm_bf16_nt
    return oracle.gemm_f16_nt_acc16 if acc16 else oracle.gemm_f16_nt


def cpu_oracle_sample(w, A, B, target_s: float = 15.0, acc16: bool = False, bf16: bool = False):
    """Time the oracle on the first R rows of C, R sized for about target_s."""
    import oracle
    fn = oracle_fn(acc16, bf16)
    threads = oracle.default_threads()
    r0 = max(threads, 1)
    t0 = time.perf_counter()
    fn(A[:r0], B, threads=threads)
    dt = time.perf_counter() - t0
    rows = int(min(w.M, max(r0, r0 * target_s / max(dt, 1e-3))))
    rows = max(threads, rows - rows % threads)
    t0 = time.perf_counter()
    fn(A[:rows], B, threads=threads)
    dt = time.perf_counter() - t0
    flops = 2.0 * rows * w.N * w.K
    return {"value": flops / dt / 1e12, "unit": UNIT, "cores": threads, "kind": "oracle",
            "cpu": cpu_model(),
            "sample": f"rows 0..{rows - 1} of C ({rows}x{w.N}x{w.K}, {flops:.3e} flop) "
                      f"in {dt:.1f} s"}


# ---------------------------------------------------------------------------
# arms
# ---------------------------------------------------------------------------

def workload_config(w, flushed: bool = False, accumulate: str = "f32"):
    l2 = (f"L2 flushed between steps (256 MiB write); value from per-launch events "
          f"(A+B+C = {w.compulsory_bytes / 2**20:.0f} MiB)" if flushed else
          f"operands larger than L2: A+B+C = {w.compulsory_bytes / 2**20:.0f} MiB > 129 MB")
    return {"workload": w.name, "M": w.M, "N": w.N, "K": w.K,
            "layout": "A[M,K] B[N,K] C[M,N] row-major, C = A·Bᵀ",
            "accumulate": accumulate, "inputs": f"A {w.dist_a}, B {w.dist_b}, seeds {w.seed_a},{w.seed_b}",
            "l2": l2, "parallelism": "replicas"}


def cublas_context(A_d, B_d, steps: int, stream, flush=None):
    """torch.matmul on the same operands and stream, fp32 accumulation kept
    (reduced-precision reductions off), timed the same way as the GEMM (the same
    L2 flush between steps when one is used): context only."""
    import torch
    m = torch.backends.cuda.matmul
    prev = (m.allow_fp16_reduced_precision_reduction, m.allow_bf16_reduced_precision_reduction)
    m.allow_fp16_reduced_precision_reduction = False
    m.allow_bf16_reduced_precision_reduction = False
    try:
        out = torch.empty((A_d.shape[0], B_d.shape[0]), dtype=A_d.dtype, device=A_d.device)
        for _ in range(3):
            torch.matmul(A_d, B_d.t(), out=out)
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for a, b in evs:
            if flush is not None:
                flush.zero_()
                a.record(stream)
                torch.matmul(A_d, B_d.t(), out=out)
                b.record(stream)
            else:
                torch.matmul(A_d, B_d.t(), out=out)
        t1.record(stream)
        torch.cuda.synchronize()
        if flush is not None:
            return sum(a.elapsed_time(b) for a, b in evs) / 1e3 / steps
        return t0.elapsed_time(t1) / 1e3 / steps
    finally:
        m.allow_fp16_reduced_precision_reduction, m.allow_bf16_reduced_precision_reduction = prev


def time_steps(step, steps: int, stream, flush=None, sampler=None):
    """Run `steps` calls of `step` on `stream`, timed with CUDA events on it.
    Back to back (flush None): returns (mean ms per launch from the events
    around the whole region, wall window).  With an L2 flush buffer: each
    launch is preceded by the flush and bracketed by its own events; returns
    the median of those per-launch times (robust to the odd delayed launch at
    the few-microsecond scale of small problems)."""
    import torch
    torch.cuda.synchronize()
    w0 = time.time()
    if flush is None:
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps):
            step()
        b.record(stream)
        if sampler is not None:
            sampler.sample_now()
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / steps
    else:
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        for a, b in evs:
            flush.zero_()
            a.record(stream)
            step()
            b.record(stream)
        if sampler is not None:
            sampler.sample_now()
        torch.cuda.synchronize()
        ms = statistics.median(a.elapsed_time(b) for a, b in evs)
    return ms, (w0, time.time())


def time_added_after_flush(step, stream, flush, n: int = 200, reps: int = 3) -> float:
    """The GPU time one launch adds after an L2 flush, in ms: n x (flush, launch)
    timed with CUDA events around the whole loop, less n flushes alone; the
    median of `reps` repeats.  At a few microseconds a launch the per-launch
    events of time_steps move in steps of the event timer's resolution
    (about 2 us on GB300); this difference of long regions does not."""
    import torch

    def region(with_step: bool) -> float:
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record(stream)
        for i in range(n):
            flush.fill_(i & 255)
            if with_step:
                step()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / n

    region(False)
    vals = sorted(region(True) - region(False) for _ in range(reps))
    return vals[len(vals) // 2]


def cublas_step(A_d, B_d, out):
    import torch

    def step():
        torch.matmul(A_d, B_d.t(), out=out)
    return step


def fp32_accumulate_only():
    """Context manager: cuBLAS through torch.matmul keeps fp32 accumulation."""
    import contextlib

    import torch

    @contextlib.contextmanager
    def cm():
        m = torch.backends.cuda.matmul
        prev = (m.allow_fp16_reduced_precision_reduction, m.allow_bf16_reduced_precision_reduction)
        m.allow_fp16_reduced_precision_reduction = False
        m.allow_bf16_reduced_precision_reduction = False
        try:
            yield
        finally:
            m.allow_fp16_reduced_precision_reduction, m.allow_bf16_reduced_precision_reduction = prev
    return cm()


def measure_workload(lib, name: str, device, stream, steps: int, warmup: int, cooldown: float, peaks,
                     sampler=None):
    """One workload through the C ABI entry point gemm_f16_nt, timed like the
    headline (L2 flushed between launches when its operands fit in L2), with
    torch.matmul (cuBLAS) timed the same way on the same operands beside it.
    Returns the record and the wall windows of the two timed regions."""
    import torch

    import dense_fp16_gemm_gb300 as g
    w = inputs.WORKLOADS[name]
    A, B = inputs.operands(w)
    Ad, Bd = torch.from_numpy(A).to(device), torch.from_numpy(B).to(device)
    Cd = torch.full((w.M, w.N), float("nan"), dtype=torch.float16, device=device)
    handle = stream.cuda_stream

    def step():
        st = lib.gemm_f16_nt(w.M, w.N, w.K, Ad.data_ptr(), w.K, Bd.data_ptr(), w.K, Cd.data_ptr(), w.N, handle)
        if st != 0:
            raise g.GemmError(st, "gemm_f16_nt")
    flushed = w.compulsory_bytes < 2 * L2_BYTES
    flush = torch.empty(256 * 2**20, dtype=torch.uint8, device=device) if flushed else None
    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    if g.device_status(stream) != 0 or torch.isnan(Cd).any().item():
        raise SystemExit(f"bench.py: {name}: watchdog word set or C unwritten after warm-up")
    if flushed and w.flops < 1e9:   # a few microseconds a launch: more samples for the median
        steps = max(steps, 200)
    out = torch.empty_like(Cd)
    cb = cublas_step(Ad, Bd, out)
    with fp32_accumulate_only():
        for _ in range(warmup):
            cb()
    # Flushed launches are each timed (median of the launches).  A region of
    # back-to-back launches lasts tens of milliseconds, where the board's power
    # management moves the clock from one region to the next: three regions
    # each, ours and cuBLAS alternating, and the median region of each.
    regions = 1 if flushed else 3
    runs, runs_cb = [], []
    for _ in range(regions):
        time.sleep(cooldown)
        runs.append(time_steps(step, steps, stream, flush, sampler))
        with fp32_accumulate_only():
            time.sleep(cooldown)
            runs_cb.append(time_steps(cb, steps, stream, flush, sampler))
    ms, win = sorted(runs, key=lambda r: r[0])[len(runs) // 2]
    ms_cb, win_cb = sorted(runs_cb, key=lambda r: r[0])[len(runs_cb) // 2]
    add = time_added_after_flush(step, stream, flush) if flushed and w.flops < 1e11 else None
    if g.device_status(stream) != 0:
        raise SystemExit(f"bench.py: {name}: watchdog word set during the timed region")
    with fp32_accumulate_only():
        add_cb = time_added_after_flush(cb, stream, flush) if add is not None else None
    pl = g.launch_plan(w.M, w.N, w.K, stream=stream, lib=lib)
    peak, peak_sus = peaks
    tf = w.flops / (ms * 1e-3) / 1e12
    tf_cb = w.flops / (ms_cb * 1e-3) / 1e12
    rec = {"M": w.M, "N": w.N, "K": w.K, "inputs": f"A {w.dist_a}, B {w.dist_b}, seeds {w.seed_a},{w.seed_b}",
           "steps": steps, "regions": regions, "us_per_launch": round(ms * 1e3, 2), "tflops": round(tf, 2),
           "frac_of_burst_peak": round(tf / peak, 4),
           "frac_of_sustained_peak": round(tf / peak_sus, 4) if peak_sus else None,
           "l2": "flushed between launches (per-launch events)" if flushed
                 else "operands larger than L2, launches back to back",
           "plan": {k: pl[k] for k in ("kernel", "cta_group", "tile_n", "cluster_pairs", "clusters", "num_tiles",
                                       "sk_tiles", "tail_split", "split_pieces", "claimed_tiles", "k_order")},
           "cublas_tflops": round(tf_cb, 2), "ours_over_cublas": round(tf / tf_cb, 4)}
    if add is not None:
        # what a launch adds to the GPU's time after a flush (launch latency overlapped)
        rec["us_added_after_flush"] = round(add * 1e3, 2)
        rec["cublas_us_added_after_flush"] = round(add_cb * 1e3, 2)
        rec["ours_over_cublas_added_after_flush"] = round(add_cb / add, 4)
    del Ad, Bd, Cd, out, flush
    torch.cuda.empty_cache()
    return rec, win, win_cb


def measure_sustained(step, cb_step, flops: float, ms_hint: float, seconds: float, stream, cooldown: float):
    """Back-to-back launches for `seconds` (ours, then cuBLAS after a
    cooldown): long enough for the board's power limit to set the clock."""
    n = max(10, int(seconds / (ms_hint * 1e-3)))
    time.sleep(cooldown)
    ms, win = time_steps(step, n, stream)
    with fp32_accumulate_only():
        time.sleep(cooldown)
        ms_cb, win_cb = time_steps(cb_step, n, stream)
    tf, tf_cb = flops / (ms * 1e-3) / 1e12, flops / (ms_cb * 1e-3) / 1e12
    return {"launches": n, "seconds": round(ms * n / 1e3, 3), "us_per_launch": round(ms * 1e3, 2),
            "tflops": round(tf, 2), "cublas_tflops": round(tf_cb, 2),
            "ours_over_cublas": round(tf / tf_cb, 4)}, win, win_cb


def fresh_process_headlines(args):
    """Run the headline alone in `args.fresh_processes` new processes (one after
    another, each idling `args.fresh_cooldown` s before its timed region) and return
    their values and median: the timing protocol the Tilus pages describe
    (median of three fresh processes, a cooldown before each measurement)."""
    cmd = [sys.executable, os.path.abspath(__file__), "--steps", str(args.steps), "--warmup", str(args.warmup),
           "--no-workloads", "--sustained-seconds", "0", "--no-cpu-baseline", "--no-cublas",
           "--cooldown", str(args.fresh_cooldown), "--cooldown-first", "--fresh-processes", "0",
           "--workload", args.workload, "--dtype", args.dtype, "--accumulate", args.accumulate,
           "--kernel", args.kernel]
    if args.shape:
        cmd += ["--shape", args.shape]
    if args.ld:
        cmd += ["--ld", str(args.ld)]
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    values = []
    for _ in range(args.fresh_processes):
        out = subprocess.run(cmd, capture_output=True, text=True, env=env, timeout=900)
        if out.returncode != 0:
            raise SystemExit("bench.py: a fresh-process headline failed:\n" + out.stderr[-2000:])
        values.append(json.loads(out.stdout.strip().splitlines()[-1])["value"])
    return {"values": values, "median": statistics.median(values), "unit": UNIT,
            "protocol": f"{len(values)} fresh processes, {args.fresh_cooldown} s idle before each timed region "
                        f"of {args.steps} launches"}


def run_e2e(args, w, A, B, Ad, Bd, Cd, tdt, entry, device, dist, bf16):
    """Pipelined end-to-end steps; returns (max time over ranks, total flops, steps)."""
    import torch
    steps = max(1, min(args.steps, 20))
    npA = A.view(np.int16) if bf16 else A
    npB = B.view(np.int16) if bf16 else B
    hA = torch.empty(Ad.shape, dtype=tdt, pin_memory=True)
    hB = torch.empty(Bd.shape, dtype=tdt, pin_memory=True)
    (hA.view(torch.int16) if bf16 else hA).copy_(torch.from_numpy(np.ascontiguousarray(npA)))
    (hB.view(torch.int16) if bf16 else hB).copy_(torch.from_numpy(np.ascontiguousarray(npB)))
    hC = [torch.empty(Cd.shape, dtype=tdt, pin_memory=True) for _ in range(2)]
    dA = [Ad, torch.empty_like(Ad)]
    dB = [Bd, torch.empty_like(Bd)]
    dC = [Cd, torch.empty_like(Cd)]
    s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
    s_mm = torch.cuda.current_stream(device)
    handle = s_mm.cuda_stream

    def gemm(j):
        st = entry(w.M, w.N, w.K, dA[j].data_ptr(), dA[j].stride(0), dB[j].data_ptr(), dB[j].stride(0),
                   dC[j].data_ptr(), w.N, handle)
        if st != 0:
            raise RuntimeError(f"GEMM call failed with status {st}")

    def run(n):
        ev_in = [torch.cuda.Event() for _ in range(n)]
        ev_mm = [torch.cuda.Event() for _ in range(n)]
        ev_out = [torch.cuda.Event() for _ in range(n)]
        for i in range(n):
            j = i % 2
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_mm[i - 2])      # buffers j free once GEMM i-2 has read them
                dA[j].copy_(hA, non_blocking=True)
                dB[j].copy_(hB, non_blocking=True)
                ev_in[i].record(s_in)
            s_mm.wait_event(ev_in[i])
            if i >= 2:
                s_mm.wait_event(ev_out[i - 2])         # C buffer j read back
            gemm(j)
            ev_mm[i].record(s_mm)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_mm[i])
                hC[j].copy_(dC[j], non_blocking=True)
                ev_out[i].record(s_out)
        s_mm.wait_stream(s_out)

    run(2)
    torch.cuda.synchronize(device)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    barrier(dist, device)
    torch.cuda.synchronize(device)
    e0.record(s_mm)
    run(steps)
    e1.record(s_mm)
    torch.cuda.synchronize(device)
    t, work = reduce_time_and_work(dist, e0.elapsed_time(e1) / 1e3, float(w.flops * steps), device)
    for h in hC:
        if torch.isnan(h.float() if bf16 else h).any().item():
            raise SystemExit("bench.py: end-to-end result has unwritten elements")
    return t, work, steps


def run_ours(args, w):
    import torch

    import dense_fp16_gemm_gb300 as g

    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    dist = init_dist(world, "nccl")

    bf16 = args.dtype == "bf16"
    tdt = torch.bfloat16 if bf16 else torch.float16
    if bf16:   # bf16 bit patterns, same distributions and seeds
        A = inputs.draw_bf16((w.M, w.K), w.dist_a, w.seed_a)
        B = inputs.draw_bf16((w.N, w.K), w.dist_b, w.seed_b)
        Ad = torch.from_numpy(A.view(np.int16)).to(device).view(tdt)
        Bd = torch.from_numpy(B.view(np.int16)).to(device).view(tdt)
    else:
        A, B = inputs.operands(w)
        Ad = torch.from_numpy(A).to(device)
        Bd = torch.from_numpy(B).to(device)
    if args.ld:   # operands placed with a row pitch of args.ld elements
        if args.ld < w.K or args.ld % 8:
            raise SystemExit("bench.py: --ld must be at least K and a multiple of 8")
        Ap = torch.zeros((w.M, args.ld), dtype=tdt, device=device)
        Bp = torch.zeros((w.N, args.ld), dtype=tdt, device=device)
        Ap[:, :w.K] = Ad
        Bp[:, :w.K] = Bd
        Ad, Bd = Ap[:, :w.K], Bp[:, :w.K]
    Cd = torch.full((w.M, w.N), float("nan"), dtype=tdt, device=device)
    stream = torch.cuda.current_stream(device)
    handle = stream.cuda_stream
    if args.library == "mcast":
        if world > 1:
            raise SystemExit("bench.py: the multicast build is for single-GPU runs only (--gpus 1)")
        lib = g.library_mcast()
    else:
        lib = g.library()
    acc16 = args.accumulate == "f16"
    # options: the fp16-accumulation variant, or a kernel asked for by name
    kopts = {}
    if acc16:
        kopts["accumulate"] = 1
    if args.kernel == "persistent":
        kopts["cta_group"] = 2
    elif args.kernel == "small":
        kopts["schedule"] = 5
    popts = g.Options(**kopts)
    if kopts:
        entry_ex = lib.gemm_bf16_nt_ex if bf16 else lib.gemm_f16_nt_ex

        def entry(*a):
            return entry_ex(*a, ctypes.byref(popts))
    else:
        entry = lib.gemm_bf16_nt if bf16 else lib.gemm_f16_nt

    def step():
        st = entry(w.M, w.N, w.K, Ad.data_ptr(), Ad.stride(0), Bd.data_ptr(), Bd.stride(0), Cd.data_ptr(), w.N, handle)
        if st != 0:
            raise g.GemmError(st, "gemm_bf16_nt" if bf16 else "gemm_f16_nt")

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(device)
    if g.device_status(stream) != 0:
        raise SystemExit("bench.py: watchdog word set during warm-up")
    if torch.isnan(Cd).any().item():
        raise SystemExit("bench.py: C has unwritten elements after warm-up")

    # Operands that fit in L2 would be served from it by the previous step: for
    # such workloads a 256 MiB buffer is overwritten between steps and the value
    # is taken from the per-launch events around the GEMM alone.
    flush = None
    if w.compulsory_bytes < 2 * L2_BYTES or args.flush_l2:
        flush = torch.empty(256 * 2**20, dtype=torch.uint8, device=device)
    sampler = ClockSampler(local) if rank == 0 else None
    times, launch_ms, head_windows = [], [], []
    for rep in range(args.repeat):
        if (rep or args.cooldown_first) and args.cooldown > 0:
            time.sleep(args.cooldown)
        # per-launch events only around flushed launches: between back-to-back
        # launches they would stop the next GEMM's set-up overlapping this one's tail
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps if flush is not None else 0)]
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        barrier(dist, device)
        torch.cuda.synchronize(device)
        w0 = time.time()
        t_start.record(stream)
        for i in range(args.steps):
            if flush is not None:
                flush.zero_()          # evict the operands from L2 (outside the launch events)
                evs[i][0].record(stream)
                step()
                evs[i][1].record(stream)
            else:
                step()
        t_end.record(stream)
        if sampler:
            sampler.sample_now()       # the enqueued launches are still running
        torch.cuda.synchronize(device)
        w1 = time.time()
        barrier(dist, device)
        if sampler:
            sampler.window(w0, w1)
        head_windows.append((w0, w1))
        times.append(t_start.elapsed_time(t_end) / 1e3)
        if flush is not None:
            launch_ms.extend(a.elapsed_time(b) for a, b in evs)
        else:   # back to back: the region is the launches
            launch_ms.extend([times[-1] * 1e3 / args.steps] * args.steps)
    if g.device_status(stream) != 0:
        raise SystemExit("bench.py: watchdog word set during the timed region")

    if flush is not None:   # whole-region time includes the flushes: use the GEMM launches
        per = len(launch_ms) // args.repeat
        times = [sum(launch_ms[r * per:(r + 1) * per]) / 1e3 for r in range(args.repeat)]
    t_med = statistics.median(times)
    t_max, total_flops = reduce_time_and_work(dist, t_med, float(w.flops * args.steps), device)
    value = total_flops / t_max / 1e12

    # roofline of the GEMM kernel: algorithmic flops per launch / mean launch time
    mean_launch_s = statistics.mean(launch_ms) / 1e3
    achieved = w.flops / mean_launch_s / 1e12
    peak, peak_sustained, peak_src = measured_peak()

    # End to end through the same C ABI from pinned host memory, pipelined the
    # way a serving loop would run it: two device buffer sets, the host->device
    # copy of step i+1 and the device->host copy of step i-1 on their own
    # streams while the GEMM of step i runs.  Every step's inputs are copied in
    # and its whole result copied out inside the timed region.
    e2e_t, e2e_work, e2e_steps = run_e2e(args, w, A, B, Ad, Bd, Cd, tdt, entry, device, dist, bf16)

    context = None
    if rank == 0 and not args.no_cublas:
        time.sleep(args.cooldown)
        t_cublas = cublas_context(Ad, Bd, max(args.steps, 10), stream, flush)
        context = {"torch_matmul_cublas_tflops": round(w.flops / t_cublas / 1e12, 2),
                   "note": "same operands, same stream, fp32 accumulation; run as a library, "
                           "context only (not the target, not part of the value)"}

    peaks = (peak, peak_sustained)
    windows = {}
    extras = rank == 0 and world == 1 and w.name == "gemm_8192" and not bf16 and not acc16 \
        and args.library == "default" and args.kernel == "auto"
    # Every other workload, timed the same way through the C ABI, each with
    # cuBLAS beside it and its own clock record.
    side = {}
    if extras and not args.no_workloads:
        for name in SIDE_WORKLOADS:
            rec, win, win_cb = measure_workload(lib, name, device, stream, args.workload_steps, args.warmup,
                                                args.cooldown, peaks, sampler)
            side[name] = rec
            windows[name] = (win, win_cb)
    small = {}
    if extras and not args.no_workloads:
        for name in SMALL_SHAPES:
            rec, win, win_cb = measure_workload(lib, name, device, stream, args.workload_steps, args.warmup,
                                                args.cooldown, peaks, sampler)
            small[name] = rec
            windows[name] = (win, win_cb)
    # A sustained window: seconds of back-to-back launches at the headline
    # shape, long enough for the board's power limit to settle the clock.
    sustained = None
    if extras and args.sustained_seconds > 0:
        out = torch.empty_like(Cd)
        sustained, win, win_cb = measure_sustained(step, cublas_step(Ad, Bd, out), w.flops, mean_launch_s * 1e3,
                                                   args.sustained_seconds, stream, args.cooldown)
        if g.device_status(stream) != 0:
            raise SystemExit("bench.py: watchdog word set during the sustained window")
        sustained["frac_of_burst_peak"] = round(sustained["tflops"] / peak, 4)
        sustained["frac_of_sustained_peak"] = round(sustained["tflops"] / peak_sustained, 4) if peak_sustained else None
        sustained["gpu_launches"] = sustained["launches"]
        windows["sustained"] = (win, win_cb)
        del out

    clocks = None
    if sampler:
        sampler.stop()
        clocks = sampler.summary(head_windows)
        for name, rec in list(side.items()) + list(small.items()):
            rec["clocks"] = sampler.summary([windows[name][0]])
            rec["cublas_clocks"] = sampler.summary([windows[name][1]])
        if sustained is not None:
            sustained["clocks"] = sampler.summary([windows["sustained"][0]])
            sustained["cublas_clocks"] = sampler.summary([windows["sustained"][1]])

    # The pages' protocol (by default in the full run): the headline measured
    # again in fresh processes, each after a cooldown, and the median reported
    # beside it.
    fresh = None
    if rank == 0 and world == 1 and args.fresh_processes > 0:
        fresh = fresh_process_headlines(args)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_oracle_sample(w, A, B, args.cpu_seconds, acc16, bf16)

    if rank == 0:
        traffic, traffic_rec = recorded_traffic(w.name) if not bf16 and not acc16 else (None, None)
        pl = g.launch_plan(w.M, w.N, w.K, stream=stream, options=popts, lib=lib)
        if pl["kernel"] == 1:
            kernel_desc = (f"gemm_f16_nt_small_kernel<SCfg<{pl['cta_group']},{pl['tile_n']},{pl['stages']},"
                           f"{int(bf16)},{int(pl['split_pieces'] > 1)}>>: {pl['clusters']} clusters x "
                           f"{pl['cta_group']} CTAs, {pl['tile_m']}x{pl['tile_n']} tiles, "
                           f"{pl['split_pieces']} k-piece(s) a tile")
        else:
            kernel_desc = (f"gemm_f16_nt_kernel<KCfg<{pl['cta_group']},256,{pl['stages']},{pl['cluster_pairs']},"
                           f"{int(bf16)},{int(acc16)}>>: "
                           f"{pl['clusters']} clusters x {pl['grid_ctas'] // pl['clusters']} CTAs, "
                           f"{pl['tile_m']}x{pl['tile_n']} cluster tiles, {pl['sk_tiles']} of {pl['num_tiles']} "
                           f"split in k, {pl['claimed_tiles']} claimed at run time, k order "
                           f"{'alternating by wave' if pl['k_order'] else 'up'}")
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(t_max / args.steps * 1e3, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if bf16 else "f16",
            "data": "synthetic", "config": {**workload_config(w, flush is not None, args.accumulate),
                                            **({"lda_ldb": args.ld} if args.ld else {})},
            "pct_of_peak": round(100.0 * achieved / peak, 2),
            "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak,
                         "unit": UNIT, "frac": round(achieved / peak, 4), "traffic": traffic,
                         "traffic_source": (f"recorded by an Nsight Compute capture of this kernel source "
                                            f"({traffic_rec['command']}), not measured by this run"
                                            if traffic_rec else None),
                         "peak_source": f"{peak_src} bf16 dense burst (fp16 runs at the bf16 rate)",
                         "frac_of_sustained": round(achieved / peak_sustained, 4) if peak_sustained else None,
                         "kernel": kernel_desc,
                         "compulsory_bytes_per_flop": round(w.compulsory_bytes / w.flops, 7),
                         "dram_bytes_per_flop": round(traffic / w.flops, 7) if traffic else None,
                         "l2_to_sm_bytes_per_flop": round(l2_to_sm_bytes(pl) / w.flops, 7)},
            "e2e": {"value": round(e2e_work / e2e_t / 1e12, 2), "unit": UNIT,
                    "h2d_bytes_per_step": int(Ad.numel() * Ad.element_size() + Bd.numel() * Bd.element_size()),
                    "d2h_bytes_per_step": int(Cd.numel() * Cd.element_size()), "steps": e2e_steps,
                    "pipeline": "pinned host buffers, two device buffer sets: the host-to-device copy of "
                                "step i+1 and the device-to-host copy of step i-1 overlap the GEMM of step i"},
            "gpu_launches": args.steps * args.repeat,
            "clocks": clocks,
            "timing": {"repeats": args.repeat, "cooldown_s": args.cooldown,
                       "per_repeat_ms_per_step": [round(t / args.steps * 1e3, 4) for t in times]},
            "sustained": sustained,
            "fresh_processes": fresh,
            "workloads": side or None,
            "small_shapes": small or None,
            "cpu_baseline": cpu,
            "context": context,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def run_reference(args, w):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    bf16 = args.dtype == "bf16"
    fn = oracle_fn(args.accumulate == "f16", bf16)
    if bf16:   # bf16 bit patterns, same distributions and seeds
        A = inputs.draw_bf16((w.M, w.K), w.dist_a, w.seed_a)
        B = inputs.draw_bf16((w.N, w.K), w.dist_b, w.seed_b)
    else:
        A, B = inputs.operands(w)
    threads = oracle.default_threads()
    # each step: a bounded sample of the workload, the first R rows of C
    probe = max(threads, 1)
    t0 = time.perf_counter()
    fn(A[:probe], B, threads=threads)
    dt = time.perf_counter() - t0
    per_step_target = max(0.5, args.cpu_seconds / max(args.steps + args.warmup, 1))
    rows = int(min(w.M, max(probe, probe * per_step_target / max(dt, 1e-3))))
    rows = max(threads, rows - rows % threads)
    for _ in range(args.warmup):
        fn(A[:rows], B, threads=threads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        fn(A[:rows], B, threads=threads)
    dt = time.perf_counter() - t0
    flops = 2.0 * rows * w.N * w.K * args.steps
    value = flops / dt / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {**workload_config(w, accumulate=args.accumulate),
                                        "l2": "host cores (no GPU cache involved)"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "cpu": cpu_model(),
                         "sample": f"each step: rows 0..{rows - 1} of C ({rows}x{w.N}x{w.K})"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--dtype", choices=["f16", "bf16"], default="f16",
                    help="operand/result type: f16 (the method's) or the bf16 variant")
    ap.add_argument("--workload", default="gemm_8192", choices=sorted(inputs.WORKLOADS))
    ap.add_argument("--ld", type=int, default=0,
                    help="row pitch of A and B in elements (default K); e.g. a 128-byte-aligned pitch "
                         "for a K whose rows are not")
    ap.add_argument("--shape", metavar="MxNxK",
                    help="time this shape instead of a named workload (inputs uniform in [-1, 1], "
                         "seeds 101 and 102); for profiling other shapes")
    ap.add_argument("--accumulate", choices=["f32", "f16"], default="f32",
                    help="accumulator type: f32 (the method) or the fp16-accumulation variant")
    ap.add_argument("--repeat", type=int, default=1,
                    help="timed regions of K steps per process (the median is reported)")
    ap.add_argument("--cooldown", type=float, default=1.0, help="seconds of idle before each repeat")
    ap.add_argument("--fresh-processes", type=int, default=None,
                    help="also time the headline in this many fresh processes (with --fresh-cooldown before "
                         "each) and report their median, the pages' protocol (default 3, or 0 with "
                         "--no-workloads; 0: off)")
    ap.add_argument("--fresh-cooldown", type=float, default=3.0,
                    help="seconds of idle before each fresh process's timed region")
    ap.add_argument("--cooldown-first", action="store_true",
                    help="also idle --cooldown seconds between the warm-up and the first timed region")
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="CPU oracle sample budget")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--flush-l2", action="store_true",
                    help="flush L2 between steps even for operands larger than 2x L2")
    ap.add_argument("--no-cublas", action="store_true",
                    help="skip the torch.matmul (cuBLAS) context measurement")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the other workloads' records (headline run only)")
    ap.add_argument("--workload-steps", type=int, default=30,
                    help="timed launches per other workload (the pages time 30 iterations)")
    ap.add_argument("--sustained-seconds", type=float, default=2.5,
                    help="length of the sustained back-to-back window at 8192^3 (0: skip)")
    ap.add_argument("--kernel", choices=["auto", "persistent", "small"], default="auto",
                    help="auto: the library's own choice; persistent: the persistent kernel (cta_group 2); "
                         "small: the small-problem kernel (schedule 5)")
    ap.add_argument("--library", choices=["default", "mcast"], default="default",
                    help="mcast: the single-GPU multicast build (refused with --gpus > 1)")
    ap.add_argument("--record-command", default="",
                    help="with --record-traffic: the command line the capture ran")
    ap.add_argument("--record-traffic", metavar="NCU_REP",
                    help="store the DRAM bytes per launch of the GEMM launches in an Nsight Compute "
                         "report for --workload in the traffic record, then exit")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.accumulate == "f16" and args.dtype == "bf16":
        ap.error("--accumulate f16 needs fp16 operands")
    if args.fresh_processes is None:
        args.fresh_processes = 0 if args.no_workloads else 3
    world, _, _ = dist_env()
    if args.gpus != world and world > 1:
        ap.error(f"--gpus {args.gpus} but WORLD_SIZE={world}")
    w = inputs.WORKLOADS[args.workload]
    if args.shape:
        try:
            M, N, K = (int(x) for x in args.shape.lower().split("x"))
        except ValueError:
            ap.error("--shape wants MxNxK")
        w = inputs.Workload(f"shape_{M}x{N}x{K}", M, N, K, inputs.U, inputs.U, 101, 102)
    if args.record_traffic:
        record_traffic(args.record_traffic, w.name, args.record_command or "")
        return
    if args.library == "mcast" and (world > 1 or args.gpus > 1):
        ap.error("--library mcast is for single-GPU runs only")
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
