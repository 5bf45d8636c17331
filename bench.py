#!/usr/bin/env python3
"""Benchmark of the bounds-checked tile-movement path on GB300.

One step = one sbt_gather_rows launch over the row-gather workload (bf16
table 1,000,000 x 512, 1,048,576 int32 indices of which 1 % are -1 and 0.5 %
point past the end).  The JSON line's `value` is effective HBM GB/s over all
ranks: algorithmic bytes (valid rows read + output written + indices) per
step / device time per step.  `ops` adds the other operations at their own
workloads (masked scatter, ragged load, tile load/store, bounded GEMM).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl sbt|reference]

`--impl reference` times the CPU oracle (plain single-threaded C) on a
bounded sample of the same workload; it is a slow baseline, not a target.
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

METRIC = "effective HBM GB/s and % of GB300 peak per op; bounded-GEMM TFLOP/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
GATHER_WORKLOAD = ("row gather: bf16 table 1,000,000x512 N(0,1), 1,048,576 int32 indices uniform in [0,1e6) "
                   "with 1% -1 and 0.5% >= 1e6 (read as 0.0), output 1,048,576x512 bf16")
L2_NOTE = "inputs larger than L2 (1.02 GB table + 1.07 GB output per step > 129 MB L2); no flush needed"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="sbt", choices=["sbt", "reference"])
    ap.add_argument("--no-ops", action="store_true", help="skip the per-operation extras")
    ap.add_argument("--e2e-steps", type=int, default=8)
    ap.add_argument("--cpu-seconds", type=float, default=8.0, help="CPU-baseline sample budget")
    ap.add_argument("--profile", default=None,
                    choices=["gather", "scatter", "scatter_add", "ragged", "ragged_store", "tile_load_tma", "tile_load", "tile_store", "tile_load_unaligned",
                             "tile_store_unaligned", "gemm", "gemm_scaled", "gemm_mxf4", "gemm_nvf4", "gather_cols"],
                    help="only launch one operation's workload (warmup + steps launches) for ncu")
    ap.add_argument("--scale", type=float, default=1.0, help="--profile: fraction of the workload's rows")
    return ap.parse_args()


FP8_NOMINAL_TFLOPS = 4500.0  # dense fp8 tensor rate, nominal (no measured fp8 peak is available)
FP4_NOMINAL_TFLOPS = 13500.0  # dense fp4 tensor rate, nominal (no measured fp4 peak is available)


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


# ----------------------------------------------------------------------------- distributed plumbing

class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
            import torch
            backend = "nccl" if torch.cuda.is_available() else "gloo"
            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, x: float) -> float:
        if not self.pg:
            return x
        import torch
        dev = "cuda" if self.pg.get_backend() == "nccl" else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def sum(self, x: float) -> float:
        if not self.pg:
            return x
        import torch
        dev = "cuda" if self.pg.get_backend() == "nccl" else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.SUM)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


def aggregate(dist, bytes_per_step: float, ms_total: float, steps: int):
    """Whole-job GB/s over all ranks: every rank's bytes / the slowest rank's time.
    Returns (GB/s, max ms over ranks)."""
    ms_max = dist.max(ms_total)
    total_bytes = dist.sum(float(bytes_per_step)) * steps
    return total_bytes / (ms_max / 1e3) / 1e9, ms_max


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples (every 100 ms) taken while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.rows = []
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(self.dev)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._reader = threading.Thread(target=self._read, daemon=True)
            self._reader.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), line.strip()))

    def mark(self, which: str):
        setattr(self, which, time.time())

    def stop(self):
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        parsed = []
        for ts, line in self.rows:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                parsed.append((ts, float(f[1]), float(f[2]), f[5:9]))
            except ValueError:
                continue
        if not parsed:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"], "samples": 0}
        inside = [p for p in parsed if self.t0 and self.t1 and self.t0 <= p[0] <= self.t1 + 0.1]
        use = inside or sorted(parsed, key=lambda p: abs(p[0] - (self.t0 or p[0])))[:3]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in use for i, v in enumerate(p[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(p[1] for p in use), "sm_max_mhz": max(p[2] for p in use),
                "reasons": reasons, "samples": len(use), "samples_in_timed_region": len(inside)}


class NvmlClockSampler:
    """SM clock and clock-event reasons read through NVML (ctypes, no Python package) every
    `period_s` from a host thread, so that a timed region of a few milliseconds still gets
    samples; `summary()` is None when NVML cannot be opened."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}

    def __init__(self, device_index: int, period_s: float = 0.0005):
        import ctypes
        self.period = period_s
        self.rows = []
        self.t0 = self.t1 = None
        self._stop = threading.Event()
        self.ok = False
        try:
            self.lib = ctypes.CDLL("libnvidia-ml.so.1")
            if self.lib.nvmlInit_v2() != 0:
                return
            self.h = ctypes.c_void_p()
            bus = None
            try:
                import torch
                pr = torch.cuda.get_device_properties(device_index)
                bus = "%08X:%02X:%02X.0" % (pr.pci_domain_id, pr.pci_bus_id, pr.pci_device_id)
            except Exception:
                bus = None
            if not (bus and self.lib.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(self.h)) == 0):
                if self.lib.nvmlDeviceGetHandleByIndex_v2(device_index, ctypes.byref(self.h)) != 0:
                    return
            self._mhz = ctypes.c_uint()
            self._reasons = ctypes.c_ulonglong()
            self._reason_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
            mx = ctypes.c_uint()
            self.max_mhz = float(mx.value) if self.lib.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx)) == 0 \
                else None
            self.ok = True
        except Exception:
            self.ok = False

    def _run(self):
        import ctypes
        while not self._stop.is_set():
            if self.lib.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(self._mhz)) == 0 and \
                    self._reason_fn(self.h, ctypes.byref(self._reasons)) == 0:
                self.rows.append((time.perf_counter(), float(self._mhz.value), int(self._reasons.value)))
            time.sleep(self.period)

    def start(self):
        if self.ok:
            self._thread = threading.Thread(target=self._run, daemon=True)
            self._thread.start()

    def mark(self, which: str):
        setattr(self, which, time.perf_counter())

    def stop(self):
        if self.ok:
            self._stop.set()
            self._thread.join(timeout=2)

    def summary(self):
        if not self.ok or not self.rows:
            return None
        inside = [r for r in self.rows if self.t0 is not None and self.t1 is not None and self.t0 <= r[0] <= self.t1]
        if not inside:
            return None
        reasons = sorted({name for r in inside for bit, name in self.REASONS.items() if r[2] & bit})
        return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": self.max_mhz, "reasons": reasons,
                "samples_in_timed_region": len(inside), "source": f"NVML every {self.period * 1e3:.1f} ms"}


# ----------------------------------------------------------------------------- helpers

def dev_bytes(a: np.ndarray):
    import torch
    flat = np.ascontiguousarray(a).reshape(-1).view(np.uint8)
    return torch.from_numpy(flat).to("cuda")


GATE_CYCLES = 400_000  # ~0.2 ms of device-side spin at 2 GHz


def time_launches(fn, reps: int, warmup: int = 3, flush=None):
    """Median, mean and best device time (ms) of one fn() call over reps, CUDA events on
    the current stream.  Each timed call is queued behind a short device-side spin
    (torch.cuda._sleep), so the host's own work for the call (binding, argument checks,
    launches) overlaps the spin and the events see the call's device work alone."""
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    times = []
    for _ in range(reps):
        if flush is not None:
            flush()
        torch.cuda._sleep(GATE_CYCLES)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        b.synchronize()
        times.append(a.elapsed_time(b))
    return statistics.median(times), statistics.fmean(times), min(times)


def time_back_to_back(fn, reps: int = 200):
    """Mean device time (ms) per call of fn() over reps calls queued back to back behind one
    spin (steady-state launch throughput: no call waits for a fresh launch after a gate)."""
    import torch
    for _ in range(5):
        fn()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    # a spin long enough (~50 us of device time per call) for the host to queue every call before
    # the first one runs, so that the events time the device alone
    torch.cuda._sleep(100_000 * reps)
    a.record()
    for _ in range(reps):
        fn()
    b.record()
    b.synchronize()
    return a.elapsed_time(b) / reps


def kernel_split(fn, reps: int):
    """Mean device time (ms) per launch of each kernel fn() launches, from CUPTI kernel
    records (torch.profiler); {} if the profiler is unavailable."""
    try:
        import torch
        from torch.profiler import ProfilerActivity, profile
        fn()
        torch.cuda.synchronize()
        with profile(activities=[ProfilerActivity.CUDA]) as prof:
            for _ in range(reps):
                fn()
            torch.cuda.synchronize()
        out = {}
        for ev in prof.events():
            if getattr(ev, "device_type", None) is not None and "CUDA" in str(ev.device_type):
                name = ev.name.replace("(anonymous namespace)::", "").replace("void ", "")
                name = name.split("(")[0].split("<")[0].strip()
                out[name] = out.get(name, 0.0) + ev.device_time / 1e3 / reps
        return out
    except Exception as e:  # report why, keep the bench line
        sys.stderr.write(f"kernel_split: {type(e).__name__}: {e}\n")
        return {}


def gather_bytes(idx: np.ndarray, n_rows: int, cols: int, es: int) -> int:
    valid = int(np.count_nonzero((idx >= 0) & (idx < n_rows)))
    return valid * cols * es + idx.size * cols * es + idx.size * 4


def read_profile_traffic(name: str, source: str):
    """dram read+write bytes per launch from a committed ncu summary, or None when the
    kernel source changed since the counters were taken."""
    import hashlib
    path = os.path.join(ROOT, "profiles", name)
    try:
        kv = {}
        for line in open(path):
            if ":" in line:
                k, v = line.split(":", 1)
                kv[k.strip()] = v.strip()
        src = open(os.path.join(ROOT, "scatter_boundary_tile_gb300", "csrc", source), "rb").read()
        if kv.get("kernel_source_sha256", "")[:16] != hashlib.sha256(src).hexdigest()[:16]:
            return None
        return int(kv["traffic_bytes_per_launch"])
    except Exception:
        return None


# ----------------------------------------------------------------------------- oracle (CPU) baseline

def host_info():
    """The host's usable cores (affinity mask) and CPU model."""
    import platform
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                model = line.split(":", 1)[1].strip()
                break
    except Exception:
        model = None
    if not model:
        try:
            for line in open("/proc/cpuinfo"):
                if line.lower().startswith("model name"):
                    model = line.split(":", 1)[1].strip()
                    break
        except Exception:
            model = None
    return {"host_cores_available": len(os.sched_getaffinity(0)), "cpu_model": model or "unknown",
            "arch": platform.machine()}


def oracle_gather(d, idx):
    import oracle
    return oracle.gather_rows(d["table"], d["n_rows"], d["cols"], d["cols"], idx, d["cols"])


def oracle_gather_all_cores(d, idx, threads: int):
    """The unchanged single-threaded oracle on `threads` disjoint slices of the index tile at
    once (its C call releases the GIL under ctypes, so the slices run on separate cores);
    returns the joined output."""
    import concurrent.futures as cf
    bounds = np.linspace(0, idx.size, threads + 1).astype(np.int64)
    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        parts = list(ex.map(lambda i: oracle_gather(d, idx[bounds[i]:bounds[i + 1]]), range(threads)))
    return np.concatenate(parts, axis=0)


def cpu_gather_sample(d, budget_s: float):
    """Time the oracle's gather on a prefix of the index tile, single-threaded and on every
    host core; the all-core output is checked bit for bit against the single-core one.
    Returns the cpu_baseline record."""
    idx = d["idx"]
    info = host_info()
    cores = info["host_cores_available"]

    def sample(run, n0):
        n = n0
        while True:
            t0 = time.perf_counter()
            run(idx[:n])
            dt = time.perf_counter() - t0
            if dt > budget_s / 8 or n >= idx.size:
                break
            n = min(idx.size, int(n * max(2.0, (budget_s / 8) / max(dt, 1e-3))))
        run(idx[:n])  # warm: the sizing runs above were partly first touches
        t0 = time.perf_counter()
        run(idx[:n])
        dt = time.perf_counter() - t0
        reps = min(20, max(1, int(budget_s / 2 / max(dt, 1e-3))))
        t0 = time.perf_counter()
        for _ in range(reps):
            run(idx[:n])
        dt = (time.perf_counter() - t0) / reps
        return gather_bytes(idx[:n], d["n_rows"], d["cols"], 2) / dt / 1e9, n, dt * reps

    gbs1, n1, s1 = sample(lambda ix: oracle_gather(d, ix), 16384)
    gbsp, npar, sp = sample(lambda ix: oracle_gather_all_cores(d, ix, cores), 16384 * cores)
    check_n = min(npar, idx.size)
    same = bool(np.array_equal(oracle_gather_all_cores(d, idx[:check_n], cores), oracle_gather(d, idx[:check_n])))
    return {"value": gbsp, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"oracle gather of the first {npar} of {idx.size} indices, split into {cores} disjoint slices "
                      f"run at once (one thread each), {sp:.1f} s",
            "all_core_output_equals_single_core": same,
            "single_core": {"value": gbs1, "unit": "GB/s", "cores": 1,
                            "sample": f"oracle gather of the first {n1} indices, {s1:.1f} s"},
            **info}


# ----------------------------------------------------------------------------- extra operations

def run_ops(ctx, pk):
    import torch
    import scatter_boundary_tile_gb300 as sbt
    import synth.workloads as wl
    ops = {}
    hbm = pk["hbm_gbs"]

    # masked scatter
    d = wl.scatter_rows_f32()
    rows, cols, n = d["dst_rows"], d["cols"], d["idx"].size
    dst = torch.zeros(rows * cols * 4, dtype=torch.uint8, device="cuda")
    s, i, m = dev_bytes(d["src"]), dev_bytes(d["idx"]), dev_bytes(d["mask"])
    fn = lambda: sbt.scatter_rows_masked(ctx, dst, rows, cols, cols, i, n, s, cols, cols, mask=m, ld_mask=cols,
                                         dtype="f32")
    med, mean, best = time_launches(fn, 20)
    nbytes = n * cols * 4 + n * cols + n * 4 + int(d["mask"].sum(dtype=np.int64)) * 4
    entry = {"workload": "fp32 dst 4,194,304x256, 1,048,576 unique rows, Bernoulli(0.9) mask",
             "ms": med, "GB/s": nbytes / med / 1e6, "frac_hbm": nbytes / med / 1e6 / hbm, "algorithmic_bytes": nbytes}
    # DRAM traffic per launch: the ncu capture at a quarter of the workload (every unit a quarter
    # as many), scaled by 4; null once the kernel source has changed since the capture
    q = read_profile_traffic("scatter_rows_f32_quarter.txt", "k_bulk.cu")
    if q:
        entry["traffic"] = 4 * q
        entry["frac_traffic"] = 4 * q / med / 1e6 / hbm
        entry["note"] = ("DRAM bytes exceed the algorithmic ones by the L2's fills of partially written 32-byte "
                         "destination sectors: with a Bernoulli(0.9) fp32 mask 57% of sectors are partial and "
                         "their untouched bytes must be read to merge; frac_traffic is the DRAM rate against the "
                         "copy peak")
    ops["scatter_rows_masked"] = entry
    del dst, s, i, m, d

    # row scatter-add: the backward of the headline gather (bf16 gradients into a zero table)
    import synth
    g = wl.gather_rows_bf16()
    n = g["idx"].size
    grad = synth.normal_bf16(0x5B7102, (n, 512))
    table = torch.zeros(1_000_000 * 512 * 2, dtype=torch.uint8, device="cuda")
    gi, gg = dev_bytes(g["idx"]), dev_bytes(grad)
    fn = lambda: sbt.scatter_add_rows(ctx, table, 1_000_000, 512, 512, gi, n, gg, 512, 512, dtype="bf16")
    med, mean, best = time_launches(fn, 20)
    valid = (g["idx"] >= 0) & (g["idx"] < 1_000_000)
    uniq = int(np.unique(g["idx"][valid]).size)
    nbytes = n * 1024 + n * 4 + 2 * uniq * 1024
    ops["scatter_add_rows"] = {"workload": "bf16 gradients 1,048,576x512 added into a 1,000,000x512 table through "
                                           "the gather's indices (repeats accumulate)",
                               "ms": med, "GB/s": nbytes / med / 1e6, "frac_hbm": nbytes / med / 1e6 / hbm,
                               "algorithmic_bytes": nbytes,
                               "note": "bytes = gradients + indices + each distinct target row read and written once"}
    del table, gi, gg, grad, g

    # column gather (axis 1): 4,096 random columns of every row of a 2,048 x 100,003 bf16 matrix
    a = synth.normal_bf16(0x5B7103, (2048, 100_003))
    ci = synth.int_below(0x5B7104, 4096, 100_003).astype(np.int32)
    ad, cid = dev_bytes(a), dev_bytes(ci)
    outc = torch.empty(2048 * 4096 * 2, dtype=torch.uint8, device="cuda")
    fn = lambda: sbt.gather_cols(ctx, ad, 2048, 100_003, 100_003, cid, 4096, outc, 4096, 2048, dtype="bf16")
    med, _, _ = time_launches(fn, 20)
    nbytes = 2 * 2048 * 4096 * 2 + 4096 * 4
    sector_bytes = 2048 * 4096 * 32 + 2048 * 4096 * 2 + 4096 * 4  # one 32-byte sector per element read
    # DRAM serves misses in 128-byte pieces: count the distinct pieces the reads touch
    offs = (np.arange(2048, dtype=np.int64)[:, None] * 100_003 + ci.astype(np.int64)[None, :]) * 2 // 128
    line_bytes = int(np.unique(offs).size) * 128 + 2048 * 4096 * 2 + 4096 * 4
    ops["gather_cols"] = {"workload": "bf16 2,048 x 100,003, 4,096 random columns gathered from every row",
                          "ms": med, "GB/s": nbytes / med / 1e6, "frac_hbm": nbytes / med / 1e6 / hbm,
                          "algorithmic_bytes": nbytes, "sector_bytes": sector_bytes,
                          "frac_hbm_sectors": sector_bytes / med / 1e6 / hbm, "line_bytes": line_bytes,
                          "frac_hbm_lines": line_bytes / med / 1e6 / hbm,
                          "note": "each 2-byte element read costs a 32-byte sector and DRAM serves misses in 128-byte "
                                  "pieces: with 4,096 random columns of 100,003 the kernel reads ~94% of the table"}
    del a, ad, cid, outc

    # ragged 3D tile load
    d = wl.ragged_bf16()
    out = torch.empty(64 * 8 * 4096 * 128 * 2, dtype=torch.uint8, device="cuda")
    x, cu = dev_bytes(d["x"]), dev_bytes(d["cu_seqlens"])
    fn = lambda: sbt.ragged_tile_load(ctx, x, d["total_rows"], 8, 128, 1024, 128, cu, 64, 4096, out, dtype="bf16")
    med, mean, best = time_launches(fn, 20)
    nbytes = d["total_rows"] * 8 * 128 * 2 + out.numel() + 65 * 4
    ops["ragged_tile_load"] = {"workload": "bf16 batch 64, len U[1,4096], 8 heads, depth 128 -> [64][8][4096][128]",
                               "ms": med, "GB/s": nbytes / med / 1e6, "frac_hbm": nbytes / med / 1e6 / hbm,
                               "algorithmic_bytes": nbytes}
    # ragged 3D tile store: the padded tiles back into the packed array (valid rows only)
    xs = torch.empty(d["total_rows"] * 8 * 128 * 2, dtype=torch.uint8, device="cuda")
    fn = lambda: sbt.ragged_tile_store(ctx, out, 64, 8, 128, 4096, cu, xs, d["total_rows"], 1024, 128, dtype="bf16")
    med, mean, best = time_launches(fn, 20)
    nbytes = 2 * d["total_rows"] * 8 * 128 * 2 + 65 * 4
    ops["ragged_tile_store"] = {"workload": "bf16 [64][8][4096][128] tiles -> packed [sum(len)][8][128], len U[1,4096]",
                                "ms": med, "GB/s": nbytes / med / 1e6, "frac_hbm": nbytes / med / 1e6 / hbm,
                                "algorithmic_bytes": nbytes}
    del out, x, cu, d, xs

    # tile load / store over a 16381 x 16411 fp32 array, 64 x 32 tiles (aligned and unaligned rows)
    import synth
    # 16,384 x 16,416 with ld 16,416 (16-byte rows) and 16,381 x 16,411 with ld 16,411 (unaligned rows)
    for r_, c_, ld, tag in ((16384, 16416, 16416, "aligned_ld"), (16381, 16411, 16411, "unaligned_ld")):
        a = synth.uniform_f32(0x5B7101, (r_, ld), -1.0, 1.0)
        gr, gc = -(-r_ // 64), -(-c_ // 32)
        ad = dev_bytes(a)
        tiles = torch.empty(gr * gc * 64 * 32 * 4, dtype=torch.uint8, device="cuda")
        fn = lambda: sbt.tile_load_padded(ctx, ad, r_, c_, ld, 1, 0, 0, 64, 32, gr, gc, 64, 32, tiles, dtype="f32")
        med, _, _ = time_launches(fn, 20)
        nbytes = r_ * c_ * 4 + tiles.numel()
        ops[f"tile_load_padded_{tag}"] = {"workload": f"fp32 {r_}x{c_} ld {ld}, 64x32 tile grid {gr}x{gc}",
                                          "ms": med, "GB/s": nbytes / med / 1e6, "frac_hbm": nbytes / med / 1e6 / hbm,
                                          "algorithmic_bytes": nbytes}
        fn = lambda: sbt.tile_store_clipped(ctx, tiles, gr, gc, 64, 32, ad, r_, c_, ld, 1, 0, 0, 64, 32, dtype="f32")
        med, _, _ = time_launches(fn, 20)
        nbytes = 2 * r_ * c_ * 4
        ops[f"tile_store_clipped_{tag}"] = {"workload": f"fp32 {r_}x{c_} ld {ld}, 64x32 tile grid {gr}x{gc}",
                                            "ms": med, "GB/s": nbytes / med / 1e6,
                                            "frac_hbm": nbytes / med / 1e6 / hbm, "algorithmic_bytes": nbytes}
        if tag == "aligned_ld":  # 128 x 64 tiles (32 KiB): the TMA tensor-copy path
            gr2, gc2 = -(-r_ // 128), -(-c_ // 64)
            t2 = torch.empty(gr2 * gc2 * 128 * 64 * 4, dtype=torch.uint8, device="cuda")
            fn = lambda: sbt.tile_load_padded(ctx, ad, r_, c_, ld, 1, 0, 0, 128, 64, gr2, gc2, 128, 64, t2,
                                              dtype="f32")
            med, _, _ = time_launches(fn, 20)
            nbytes = r_ * c_ * 4 + t2.numel()
            ops["tile_load_padded_tma_128x64"] = {"workload": f"fp32 {r_}x{c_} ld {ld}, 128x64 tile grid {gr2}x{gc2}",
                                                  "ms": med, "GB/s": nbytes / med / 1e6,
                                                  "frac_hbm": nbytes / med / 1e6 / hbm, "algorithmic_bytes": nbytes}
            fn = lambda: sbt.tile_store_clipped(ctx, t2, gr2, gc2, 128, 64, ad, r_, c_, ld, 1, 0, 0, 128, 64,
                                                dtype="f32")
            med, _, _ = time_launches(fn, 20)
            nbytes = 2 * r_ * c_ * 4
            ops["tile_store_clipped_tma_128x64"] = {"workload": f"fp32 {r_}x{c_} ld {ld}, 128x64 tile grid {gr2}x{gc2}",
                                                    "ms": med, "GB/s": nbytes / med / 1e6,
                                                    "frac_hbm": nbytes / med / 1e6 / hbm, "algorithmic_bytes": nbytes}
            del t2
        del ad, tiles, a

    # bounded GEMM
    try:
        for (M, N, K) in wl.GEMM_SHAPES:
            g = wl.gemm_bf16(M=M, N=N, K=K)
            A, B = dev_bytes(g["A"]), dev_bytes(g["B"])
            C = torch.empty(M * g["ldc"] * 2, dtype=torch.uint8, device="cuda")
            ws_n = sbt.gemm_bounded_workspace_size(ctx, M, N, K, g["lda"], g["ldb"])
            ws = torch.empty(max(ws_n, 1), dtype=torch.uint8, device="cuda")
            fn = lambda: sbt.gemm_bounded(ctx, A, g["lda"], B, g["ldb"], C, g["ldc"], M, N, K, ws, ws_n)
            med, _, _ = time_launches(fn, 10 if M > 4000 else 30)
            flops = 2.0 * M * N * K
            tf = flops / med / 1e9
            entry = {"ms": med, "TFLOP/s": tf, "frac_bf16": tf / pk["bf16_tflops"],
                     "frac_bf16_sustained": tf / pk["bf16_tflops_sustained"], "flops": flops,
                     "lda": g["lda"], "ldb": g["ldb"], "ldc": g["ldc"],
                     "note": "whole call: one realigning staging launch (odd leading dimensions) + tensor-core kernel"}
            if flops < 1e10:  # small shapes: per-call time with the launches of consecutive calls overlapped
                entry["ms_back_to_back"] = time_back_to_back(fn)
            split = kernel_split(fn, 5)
            if split:
                entry["kernels_ms"] = split
                main = sum(v for k, v in split.items() if "k_gemm" in k)
                if main > 0:
                    entry["tensor_kernel_TFLOP/s"] = flops / main / 1e9
                    entry["tensor_kernel_frac_bf16"] = flops / main / 1e9 / pk["bf16_tflops"]
            ops[f"gemm_bounded_{M}x{N}x{K}"] = entry
            del A, B, C, ws
        # 16-byte-aligned rows: TMA reads A and B where they lie, one launch, no staging
        M, N, K = 8192, 8192, 4096
        g = wl.gemm_bf16(M=M, N=N, K=K)
        A = np.ascontiguousarray(g["A"][:, :K])
        B = np.ascontiguousarray(g["B"][:, :N])
        Ad, Bd = dev_bytes(A), dev_bytes(B)
        C = torch.empty(M * N * 2, dtype=torch.uint8, device="cuda")
        ws_n = sbt.gemm_bounded_workspace_size(ctx, M, N, K, K, N)
        ws = torch.empty(max(ws_n, 1), dtype=torch.uint8, device="cuda")
        fn = lambda: sbt.gemm_bounded(ctx, Ad, K, Bd, N, C, N, M, N, K, ws, ws_n)
        med, _, _ = time_launches(fn, 10)
        # (1000, 1000, 1000) with rows 16-byte aligned: one launch per call
        m1, n1, k1 = 1000, 1000, 1000
        g1 = wl.gemm_bf16(M=m1, N=n1, K=k1)
        A1 = np.zeros((m1, 1000), np.uint16)
        A1[:, :k1] = g1["A"][:, :k1]
        B1 = np.zeros((k1, 1000), np.uint16)
        B1[:, :n1] = g1["B"][:, :n1]
        A1d, B1d = dev_bytes(A1), dev_bytes(B1)
        C1 = torch.empty(m1 * 1000 * 2, dtype=torch.uint8, device="cuda")
        ws1_n = sbt.gemm_bounded_workspace_size(ctx, m1, n1, k1, 1000, 1000)
        ws1 = torch.empty(max(ws1_n, 1), dtype=torch.uint8, device="cuda")
        f1 = lambda: sbt.gemm_bounded(ctx, A1d, 1000, B1d, 1000, C1, 1000, m1, n1, k1, ws1, ws1_n)
        n0 = ctx.launch_count
        f1()
        launches1 = ctx.launch_count - n0
        ms1, _, _ = time_launches(f1, 30)
        ops["gemm_bounded_1000x1000x1000_aligned"] = {
            "ms": ms1, "ms_back_to_back": time_back_to_back(f1), "launches_per_call": launches1,
            "lda": 1000, "ldb": 1000, "ldc": 1000,
            "note": "rows 16-byte aligned: TMA reads A and B where they lie; ms is one call behind a device "
                    "spin, ms_back_to_back the steady-state time per call"}
        del A1d, B1d, C1, ws1
        flops = 2.0 * M * N * K
        tf = flops / med / 1e9
        entry = {"ms": med, "TFLOP/s": tf, "frac_bf16": tf / pk["bf16_tflops"],
                 "frac_bf16_sustained": tf / pk["bf16_tflops_sustained"], "flops": flops, "lda": K, "ldb": N, "ldc": N,
                 "note": "aligned leading dimensions: the tensor-core kernel alone (TMA reads A and B where they lie)"}
        split = kernel_split(fn, 5)
        if split:
            entry["kernels_ms"] = split
        ops[f"gemm_bounded_{M}x{N}x{K}_aligned"] = entry
        del Ad, Bd, C, ws
    except Exception as e:  # a library built without the GEMM
        ops["gemm_bounded"] = {"unavailable": str(e).splitlines()[0][:200]}

    # block-scaled GEMM: E4M3 operands, E8M0 scales over blocks of 32 along K, fp32 out;
    # "auto" runs the tcgen05 block-scaled kernel, "scalar" the bf16-staging path
    for (M, N, K) in [(8191, 8193, 4096)]:
        g = wl.gemm_block_scaled(M=M, N=N, K=K, block=32)
        A, B, SA, SB = (dev_bytes(g[k]) for k in ("A", "B", "SA", "SB"))
        D = torch.empty(M * g["ldd"] * 4, dtype=torch.uint8, device="cuda")
        ws_n = sbt.gemm_block_scaled_workspace_size(ctx, M, N, K)
        ws = torch.empty(max(ws_n, 256), dtype=torch.uint8, device="cuda")
        fn = lambda: sbt.gemm_block_scaled(ctx, A, g["lda"], B, g["ldb"], SA, g["ld_sa"], SB, g["ld_sb"], g["Ks"],
                                           D, g["ldd"], M, N, K, workspace=ws, workspace_bytes=ws_n)
        flops = 2.0 * M * N * K
        for path, note in [("auto", "whole call: 8-bit staging + tcgen05 kind::mxf8f6f4 block-scaled kernel"),
                           ("scalar", "whole call: scaled operands staged as bf16 + the bf16 tcgen05 kernel")]:
            ctx.set_path(path)
            med, _, _ = time_launches(fn, 10)
            tf = flops / med / 1e9
            entry = {"ms": med, "TFLOP/s": tf, "frac_fp8_nominal": tf / FP8_NOMINAL_TFLOPS,
                     "workload": "E4M3 x E4M3, E8M0 scales per 32 along K, fp32 D, no acc", "note": note}
            split = kernel_split(fn, 5)
            if split:
                entry["kernels_ms"] = split
            ops[f"gemm_block_scaled_{M}x{N}x{K}" + ("" if path == "auto" else "_bf16_staging")] = entry
        ctx.set_path("auto")
        del A, B, SA, SB, D, ws
        # 4-bit operands (E2M1, two per byte) on the packed forms of the tensor path:
        # E8M0 scales per 32 (kind::mxf4) and E4M3 scales per 16 (kind::mxf4nvf4)
        for sfmt, block, tag, note in [
                ("e8m0", 32, "e2m1", "whole call: packed 4-bit staging + tcgen05 kind::mxf4 block-scaled kernel"),
                ("e4m3", 16, "e2m1_e4m3_per16",
                 "whole call: packed 4-bit staging (E4M3 scale signs onto the codes) + tcgen05 kind::mxf4nvf4 kernel")]:
            g = wl.gemm_block_scaled(M=M, N=N, K=K, block=block, afmt="e2m1", bfmt="e2m1", sfmt=sfmt)
            A, B, SA, SB = (dev_bytes(g[k]) for k in ("A", "B", "SA", "SB"))
            D = torch.empty(M * g["ldd"] * 4, dtype=torch.uint8, device="cuda")
            ws = torch.empty(max(ws_n, 256), dtype=torch.uint8, device="cuda")
            fn = lambda: sbt.gemm_block_scaled(ctx, A, g["lda"], B, g["ldb"], SA, g["ld_sa"], SB, g["ld_sb"], g["Ks"],
                                               D, g["ldd"], M, N, K, workspace=ws, workspace_bytes=ws_n,
                                               a_fmt="e2m1", b_fmt="e2m1", s_fmt=sfmt)
            med, _, _ = time_launches(fn, 10)
            tf = flops / med / 1e9
            entry = {"ms": med, "TFLOP/s": tf, "frac_fp4_nominal": tf / FP4_NOMINAL_TFLOPS,
                     "workload": f"E2M1 x E2M1 (packed), {sfmt.upper()} scales per {block} along K, fp32 D, no acc",
                     "note": note}
            split = kernel_split(fn, 5)
            if split:
                entry["kernels_ms"] = split
            ops[f"gemm_block_scaled_{M}x{N}x{K}_{tag}"] = entry
            del A, B, SA, SB, D, ws
    return ops


def box_record(device_index: int):
    """Which machine and GPU produced this line (host-link and clock behaviour differ by box)."""
    import socket
    import torch
    rec = {"host": socket.gethostname()}
    try:
        pr = torch.cuda.get_device_properties(device_index)
        rec.update(gpu=pr.name, gpu_uuid=str(pr.uuid), pci_bus_id=int(pr.pci_bus_id), sm_count=pr.multi_processor_count)
    except Exception:
        pass
    return rec


def clocks_record(smi: ClockSampler, nvml: NvmlClockSampler):
    """nvidia-smi samples (100 ms) of the timed region, refined by NVML samples taken every
    0.5 ms when the region is too short for nvidia-smi: the SM clock median and the
    reasons come from whichever source saw more samples inside the region; both are kept."""
    a = smi.summary()
    b = nvml.summary()
    if b and b["samples_in_timed_region"] > a.get("samples_in_timed_region", 0):
        out = dict(b)
        out["sm_max_mhz"] = b["sm_max_mhz"] or a.get("sm_max_mhz")
        out["reasons"] = sorted(set(b["reasons"]) | set(r for r in a.get("reasons", []) if r != "no nvidia-smi samples"))
        out["nvidia_smi"] = a
        return out
    if b:
        a = dict(a)
        a["nvml"] = b
    return a


# ----------------------------------------------------------------------------- arms

def run_e2e(ctx, table, idx, n_rows, cols, t_dev, i_dev, out, steps, dist):
    """Pipelined end-to-end gather through host buffers; returns (ms per step, H2D bytes, D2H bytes)."""
    import torch
    import scatter_boundary_tile_gb300 as sbt
    h_table = torch.from_numpy(np.ascontiguousarray(table).reshape(-1).view(np.uint8)).pin_memory()
    h_idx = torch.from_numpy(np.ascontiguousarray(idx).reshape(-1).view(np.uint8)).pin_memory()
    n = idx.size
    dev_t = [t_dev, torch.empty_like(t_dev)]
    dev_i = [i_dev, torch.empty_like(i_dev)]
    dev_o = [out, torch.empty_like(out)]
    h_out = [torch.empty(out.numel(), dtype=torch.uint8).pin_memory() for _ in range(2)]
    s_in, s_run, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_run = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    used = [False, False]

    def step(i):
        b = i % 2
        if used[b]:
            s_in.wait_event(ev_run[b])    # the previous gather on this buffer has read its inputs
            s_run.wait_event(ev_out[b])   # the previous download of this buffer has read it
        with torch.cuda.stream(s_in):
            dev_t[b].copy_(h_table, non_blocking=True)
            dev_i[b].copy_(h_idx, non_blocking=True)
            ev_in[b].record(s_in)
        s_run.wait_event(ev_in[b])
        sbt.gather_rows(ctx, dev_t[b], n_rows, cols, cols, dev_i[b], n, dev_o[b], cols, cols, dtype="bf16",
                        stream=s_run)
        ev_run[b].record(s_run)
        s_out.wait_event(ev_run[b])
        with torch.cuda.stream(s_out):
            h_out[b].copy_(dev_o[b], non_blocking=True)
            ev_out[b].record(s_out)
        used[b] = True

    for i in range(2):
        step(i)
    torch.cuda.synchronize()
    dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    s_run.wait_event(e0)
    s_out.wait_event(e0)
    for i in range(steps):
        step(i)
    e1.record(s_out)
    e1.synchronize()
    ms = dist.max(e0.elapsed_time(e1)) / steps
    last = (steps - 1) % 2
    assert np.array_equal(h_out[last].numpy()[:cols * 2 * 64], dev_o[last][:cols * 2 * 64].cpu().numpy())
    h2d, d2h = h_table.numel() + h_idx.numel(), h_out[0].numel()
    del dev_t[1], dev_i[1], dev_o[1]
    return ms, h2d, d2h


def run_reference(args, dist):
    if dist.rank != 0:
        return 0
    import synth.workloads as wl
    d = wl.gather_rows_bf16()
    info = host_info()
    cores = info["host_cores_available"]
    n = 65536 * cores  # each step: the oracle on a prefix of the workload, one slice per host core
    idx = d["idx"][:n]
    for _ in range(min(args.warmup, 3)):
        oracle_gather_all_cores(d, idx, cores)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle_gather_all_cores(d, idx, cores)
        times.append(time.perf_counter() - t0)
        if sum(times) > 120:
            break
    dt = statistics.fmean(times)
    gbs = gather_bytes(idx, d["n_rows"], d["cols"], 2) / dt / 1e9
    sample = (f"oracle gather of the first {idx.size} of 1,048,576 indices per step, {cores} disjoint slices "
              f"run at once (one thread each; the oracle itself is single-threaded C) ({len(times)} steps)")
    line = {"impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": len(times), "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": GATHER_WORKLOAD, "l2": "CPU run"},
            "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample,
                             **info},
            "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_sbt(args, dist):
    import torch
    import scatter_boundary_tile_gb300 as sbt
    import synth.workloads as wl

    torch.cuda.set_device(dist.local_rank)
    pk, pk_src = peaks()
    ctx = sbt.Context(dist.local_rank)

    d = wl.gather_rows_bf16(seed=wl.SEED_GATHER + 1000 * dist.rank)  # each rank: its own batch (weak scaling)
    table, idx = d["table"], d["idx"]
    n, cols, n_rows = idx.size, d["cols"], d["n_rows"]
    bytes_step = gather_bytes(idx, n_rows, cols, 2)
    t_dev, i_dev = dev_bytes(table), dev_bytes(idx)
    out = torch.empty(n * cols * 2, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        sbt.gather_rows(ctx, t_dev, n_rows, cols, cols, i_dev, n, out, cols, cols, dtype="bf16")

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    ctx.check_status()

    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    fine = NvmlClockSampler(torch.cuda.current_device())
    fine.start()
    time.sleep(0.3)
    dist.barrier()
    torch.cuda.synchronize()
    launches0 = ctx.launch_count
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler.mark("t0")
    fine.mark("t0")
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    ev1.synchronize()
    fine.mark("t1")
    sampler.mark("t1")
    torch.cuda.synchronize()
    dist.barrier()
    launches = ctx.launch_count - launches0
    sampler.stop()
    fine.stop()
    ms_total = ev0.elapsed_time(ev1)
    value, ms_max = aggregate(dist, bytes_step, ms_total, args.steps)
    ms_step = ms_max / args.steps
    achieved = bytes_step / (ms_total / args.steps / 1e3) / 1e9  # this rank's kernel, per launch
    ctx.check_status()

    # End to end through host buffers: every step copies its inputs (pinned table + indices)
    # in and its gathered rows out.  Steps are pipelined over two buffer sets and three
    # streams, so step i+1's upload overlaps step i's download (the copy engines are full
    # duplex); each buffer is reused only after its previous gather and download finished.
    e2e_ms, h2d_bytes, d2h_bytes = run_e2e(ctx, table, idx, n_rows, cols, t_dev, i_dev, out, args.e2e_steps, dist)
    e2e_value = dist.sum(float(bytes_step)) / (e2e_ms / 1e3) / 1e9

    traffic = read_profile_traffic("gather_rows_bf16_1Mx512.txt", "k_rows.cu")
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": dist.world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": GATHER_WORKLOAD, "l2": L2_NOTE, "parallelism": f"replicas x{dist.world}",
                   "algorithmic_bytes_per_step": bytes_step,
                   "note": "bf16 rows moved as raw 16-bit words; index arithmetic in int64"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / pk["hbm_gbs"], "traffic": traffic, "peak_source": pk_src,
                     "kernel": "k_gather_rows<2,vector,no-mask>"},
        "gpu_launches": launches,
        "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d_bytes,
                "d2h_bytes_per_step": d2h_bytes, "ms_per_step": e2e_ms,
                "note": "inputs copied host->device and the output device->host every step; steps pipelined "
                        "over two buffer sets (upload of step i+1 overlaps download of step i)"},
        "clocks": clocks_record(sampler, fine),
        "box": box_record(torch.cuda.current_device()),
    }
    if not args.no_ops:
        del out, t_dev
        torch.cuda.empty_cache()
        line["ops"] = run_ops(ctx, pk)
    if dist.rank == 0:
        line["cpu_baseline"] = cpu_gather_sample(d, args.cpu_seconds)
        print(json.dumps(line), flush=True)
    ctx.close()
    return 0


def run_profile(args):
    """Launch one operation `warmup + steps` times on its workload (scaled by --scale) and
    print the mean device time; used as the command under ncu."""
    import torch
    import scatter_boundary_tile_gb300 as sbt
    import synth
    import synth.workloads as wl
    ctx = sbt.Context(0)
    op, f = args.profile, args.scale
    if op == "gather":
        d = wl.gather_rows_bf16(n_rows=max(1, int(1_000_000 * f)), n_idx=max(1, int(1_048_576 * f)))
        t, i = dev_bytes(d["table"]), dev_bytes(d["idx"])
        n, rows = d["idx"].size, d["n_rows"]
        out = torch.empty(n * 512 * 2, dtype=torch.uint8, device="cuda")
        fn = lambda: sbt.gather_rows(ctx, t, rows, 512, 512, i, n, out, 512, 512, dtype="bf16")
    elif op == "scatter":
        d = wl.scatter_rows_f32(dst_rows=max(1, int(4_194_304 * f)), n_idx=max(1, int(1_048_576 * f)))
        rows, n = d["dst_rows"], d["idx"].size
        dst = torch.zeros(rows * 256 * 4, dtype=torch.uint8, device="cuda")
        s_, i, m = dev_bytes(d["src"]), dev_bytes(d["idx"]), dev_bytes(d["mask"])
        fn = lambda: sbt.scatter_rows_masked(ctx, dst, rows, 256, 256, i, n, s_, 256, 256, mask=m, ld_mask=256,
                                             dtype="f32")
    elif op == "ragged":
        d = wl.ragged_bf16(batch=max(1, int(64 * f)))
        b = d["cu_seqlens"].size - 1
        out = torch.empty(b * 8 * 4096 * 128 * 2, dtype=torch.uint8, device="cuda")
        x, cu = dev_bytes(d["x"]), dev_bytes(d["cu_seqlens"])
        fn = lambda: sbt.ragged_tile_load(ctx, x, d["total_rows"], 8, 128, 1024, 128, cu, b, 4096, out,
                                          dtype="bf16")
    elif op == "scatter_add":
        d = wl.gather_rows_bf16(n_rows=max(1, int(1_000_000 * f)), n_idx=max(1, int(1_048_576 * f)))
        n, rows = d["idx"].size, d["n_rows"]
        grad = synth.normal_bf16(0x5B7102, (n, 512))
        table = torch.zeros(rows * 512 * 2, dtype=torch.uint8, device="cuda")
        gi, gg = dev_bytes(d["idx"]), dev_bytes(grad)
        fn = lambda: sbt.scatter_add_rows(ctx, table, rows, 512, 512, gi, n, gg, 512, 512, dtype="bf16")
    elif op == "ragged_store":
        d = wl.ragged_bf16(batch=max(1, int(64 * f)))
        b = d["cu_seqlens"].size - 1
        tiles = torch.empty(b * 8 * 4096 * 128 * 2, dtype=torch.uint8, device="cuda")
        xs = torch.empty(d["total_rows"] * 8 * 128 * 2, dtype=torch.uint8, device="cuda")
        cu = dev_bytes(d["cu_seqlens"])
        fn = lambda: sbt.ragged_tile_store(ctx, tiles, b, 8, 128, 4096, cu, xs, d["total_rows"], 1024, 128,
                                           dtype="bf16")
    elif op == "tile_load_tma":
        r_, c_ = max(128, int(16384 * f)), 16416
        a = synth.uniform_f32(0x5B7101, (r_, c_), -1.0, 1.0)
        gr, gc = -(-r_ // 128), -(-c_ // 64)
        ad = dev_bytes(a)
        tiles = torch.empty(gr * gc * 128 * 64 * 4, dtype=torch.uint8, device="cuda")
        fn = lambda: sbt.tile_load_padded(ctx, ad, r_, c_, c_, 1, 0, 0, 128, 64, gr, gc, 128, 64, tiles, dtype="f32")
    elif op.startswith("tile"):
        unal = op.endswith("unaligned")
        r_, c_ = max(64, int((16381 if unal else 16384) * f)), (16411 if unal else 16416)
        ld = c_
        a = synth.uniform_f32(0x5B7101, (r_, ld), -1.0, 1.0)
        gr, gc = -(-r_ // 64), -(-c_ // 32)
        ad = dev_bytes(a)
        tiles = torch.empty(gr * gc * 64 * 32 * 4, dtype=torch.uint8, device="cuda")
        if op.startswith("tile_load"):
            fn = lambda: sbt.tile_load_padded(ctx, ad, r_, c_, ld, 1, 0, 0, 64, 32, gr, gc, 64, 32, tiles,
                                              dtype="f32")
        else:
            fn = lambda: sbt.tile_store_clipped(ctx, tiles, gr, gc, 64, 32, ad, r_, c_, ld, 1, 0, 0, 64, 32,
                                                dtype="f32")
    elif op == "gather_cols":  # bf16 2,048 x 100,003, 4,096 random columns (rows scaled)
        rows_ = max(1, int(2048 * f))
        a = synth.normal_bf16(0x5B7103, (rows_, 100_003))
        ci = synth.int_below(0x5B7104, 4096, 100_003).astype(np.int32)
        ad, cid = dev_bytes(a), dev_bytes(ci)
        outc = torch.empty(rows_ * 4096 * 2, dtype=torch.uint8, device="cuda")
        fn = lambda: sbt.gather_cols(ctx, ad, rows_, 100_003, 100_003, cid, 4096, outc, 4096, rows_, dtype="bf16")
    elif op in ("gemm_scaled", "gemm_mxf4", "gemm_nvf4"):
        # (8191, 8193, 4096) scaled along M: E4M3 / E8M0 per 32, E2M1 / E8M0 per 32, E2M1 / E4M3 per 16
        M, N, K = max(1, int(8191 * f)), 8193, 4096
        fmt, sfmt, block = {"gemm_scaled": ("e4m3", "e8m0", 32), "gemm_mxf4": ("e2m1", "e8m0", 32),
                            "gemm_nvf4": ("e2m1", "e4m3", 16)}[op]
        g = wl.gemm_block_scaled(M=M, N=N, K=K, block=block, afmt=fmt, bfmt=fmt, sfmt=sfmt)
        A, B, SA, SB = (dev_bytes(g[k]) for k in ("A", "B", "SA", "SB"))
        D = torch.empty(M * g["ldd"] * 4, dtype=torch.uint8, device="cuda")
        ws_n = sbt.gemm_block_scaled_workspace_size(ctx, M, N, K)
        ws = torch.empty(max(ws_n, 256), dtype=torch.uint8, device="cuda")
        fn = lambda: sbt.gemm_block_scaled(ctx, A, g["lda"], B, g["ldb"], SA, g["ld_sa"], SB, g["ld_sb"], g["Ks"],
                                           D, g["ldd"], M, N, K, workspace=ws, workspace_bytes=ws_n, a_fmt=fmt,
                                           b_fmt=fmt, s_fmt=sfmt)
    else:  # gemm: (8191, 8193, 4097) scaled along M
        M, N, K = max(1, int(8191 * f)), 8193, 4097
        g = wl.gemm_bf16(M=M, N=N, K=K)
        A, B = dev_bytes(g["A"]), dev_bytes(g["B"])
        C = torch.empty(M * g["ldc"] * 2, dtype=torch.uint8, device="cuda")
        ws_n = sbt.gemm_bounded_workspace_size(ctx, M, N, K, g["lda"], g["ldb"])
        ws = torch.empty(max(ws_n, 256), dtype=torch.uint8, device="cuda")
        fn = lambda: sbt.gemm_bounded(ctx, A, g["lda"], B, g["ldb"], C, g["ldc"], M, N, K, ws, ws_n)
    med, mean, best = time_launches(fn, args.steps, warmup=args.warmup)
    ctx.check_status()
    print(json.dumps({"profile": op, "scale": f, "ms_median": med, "ms_mean": mean, "ms_best": best,
                      "launches": ctx.launch_count}), flush=True)
    return 0


def main():
    args = parse()
    if args.profile:
        return run_profile(args)
    if args.warmup < 3:
        args.warmup = 3
    dist = Dist()
    try:
        rc = run_reference(args, dist) if args.impl == "reference" else run_sbt(args, dist)
    finally:
        dist.close()
    return rc


if __name__ == "__main__":
    sys.exit(main())
