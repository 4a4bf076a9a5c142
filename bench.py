"""RMSNorm forward benchmark on GB300 (one JSON line on rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--e2e-steps E] [--cpu-seconds S]
                    [--op rmsnorm|qk_norm|bias|mxfp8|mxfp4|nvfp4|latency]
                    [--weight-bias B]

A step is one RMSNorm forward over one batch: the headline workload is the
prefill-shaped batch, 16384 rows x 4096 hidden, bf16 in/out, fp32
accumulation, eps 1e-6 (x ~ N(0,1), weight ~ N(1,0.1), seeded).  Inputs are
resident in HBM before the timed region; consecutive steps rotate over
several input/output sets whose total is larger than the 129 MB L2, so every
step reads x from HBM.

Timing: W untimed warm-up steps, then R timed regions (--regions, default 5)
of exactly K steps each, every region bracketed by a barrier and
torch.cuda.synchronize() on both sides, with one pair of CUDA events on the
launching stream around it (it holds only the kernel's K back-to-back
launches, so region time / K is the kernel's average launch duration, launch
gaps included); max over ranks per region; the median region is reported,
the others beside it.  SM clocks and throttle reasons are sampled with
nvidia-smi over all the regions.

value = algorithmic bytes (read x + read weight + write y) of every step of
every rank / the slowest rank's time, in GB/s.  e2e = the same metric through
the public API with the step's input copied host->device from pinned memory
and the result copied back, every step.  cpu_baseline = the fp64 CPU oracle
timed on this host on a bounded sample of the same workload (one thread; its
row_parallel entry: the same oracle on every host core).

--impl reference times the oracle itself (there is no other implementation
of this path to compare with): rank 0 only, each step a bounded sample of the
workload, same metric and unit.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from rmsnorm_fwd_gb300 import inputs  # noqa: E402

L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0
METRIC = "RMSNorm achieved HBM GB/s (% of GB300 peak) and rows/s at 16384x4096 bf16"
UNIT = "GB/s"


# ----------------------------------------------------------------- distributed

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
    dist.init_process_group(backend=backend)
    return dist


def reduce_max(value: float, dist, device=None) -> float:
    """Max over ranks (identity on one process)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist, device=None):
    if dist is None:
        return
    if device is not None:
        dist.barrier(device_ids=[device.index])
    else:
        dist.barrier()


# ----------------------------------------------------------------- clocks

CLOCK_FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    """nvidia-smi sampling of one GPU while the timed region runs."""

    def __init__(self, gpu_index: int, period_ms: int = 50):
        self.gpu = gpu_index
        self.period = period_ms
        self.proc = None
        self.lines: list[str] = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={CLOCK_FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.period)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)  # let the first samples land before the region starts

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self):
        return time.time()

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)

    def summary(self, t0: float, t1: float) -> dict:
        rows = []
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm, smax = float(parts[0]), float(parts[1])
            except ValueError:
                continue
            rows.append((ts, sm, smax, parts[3:]))
        inside = [r for r in rows if t0 <= r[0] <= t1]
        if not inside and rows:  # a very short region: take the nearest sample
            inside = [min(rows, key=lambda r: abs(r[0] - 0.5 * (t0 + t1)))]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        reasons = set()
        for r in inside:
            for name, val in zip(names[1:], r[3][1:]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r[1] for r in inside),
                "sm_max_mhz": max(r[2] for r in inside),
                "reasons": sorted(reasons), "samples": len(inside)}


class NvmlPoller:
    """Read-only NVML queries (the driver's libnvidia-ml) of one GPU's SM
    clock and clock-event reasons, every `period_s` on a background thread
    while the timed regions run: nvidia-smi's own sampling gives one or two
    samples over regions of a few milliseconds.  Silent when NVML cannot be
    loaded (the nvidia-smi record stands alone then)."""

    # NVML clock-event reason bits (nvml.h)
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, torch_device, period_s: float = 0.0005):
        self.period = period_s
        self.samples: list[tuple[float, int, int]] = []
        self.max_mhz = None
        self.lib = self.handle = None
        self.stop_flag = threading.Event()
        self.thread = None
        try:
            import ctypes
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return
            h = ctypes.c_void_p()
            pr = None
            try:
                import torch
                pr = torch.cuda.get_device_properties(torch_device)
            except Exception:
                pass
            ok = False
            if pr is not None and hasattr(pr, "pci_bus_id"):
                bus = (f"{getattr(pr, 'pci_domain_id', 0):08x}:{pr.pci_bus_id:02x}:"
                       f"{pr.pci_device_id:02x}.0").encode()
                ok = lib.nvmlDeviceGetHandleByPciBusId_v2(bus, ctypes.byref(h)) == 0
            if not ok:
                idx = torch_device.index if hasattr(torch_device, "index") else 0
                ok = lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(idx or 0),
                                                       ctypes.byref(h)) == 0
            if not ok:
                return
            self.reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                lib.nvmlDeviceGetCurrentClocksThrottleReasons
            mx = ctypes.c_uint()
            if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:  # 1 = SM clock
                self.max_mhz = mx.value
            self.lib, self.handle, self.ct = lib, h, ctypes
        except Exception:
            self.lib = None

    def _run(self):
        ct, lib, h = self.ct, self.lib, self.handle
        clk, rs = ct.c_uint(), ct.c_ulonglong()
        while not self.stop_flag.is_set():
            if lib.nvmlDeviceGetClockInfo(h, 1, ct.byref(clk)) == 0 and \
                    self.reasons_fn(h, ct.byref(rs)) == 0:
                self.samples.append((time.time(), clk.value, rs.value))
            time.sleep(self.period)

    def start(self):
        if self.lib is not None:
            self.thread = threading.Thread(target=self._run, daemon=True)
            self.thread.start()

    def stop(self):
        if self.thread is not None:
            self.stop_flag.set()
            self.thread.join(timeout=2)

    def summary(self, t0: float, t1: float):
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        if self.lib is None or not inside:
            return None
        reasons = sorted({name for _, _, r in inside for bit, name in self.REASONS.items()
                          if r & bit})
        mhz = [m for _, m, _ in inside]
        return {"samples": len(inside), "sm_mhz": statistics.median(mhz), "sm_mhz_min": min(mhz),
                "sm_max_mhz": self.max_mhz, "reasons": reasons,
                "source": "NVML, every 0.5 ms inside the timed regions"}


# ----------------------------------------------------------------- peaks, traffic

def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            v = float(json.load(fh)["hbm_gbs"])
        return v, "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# The translation unit that holds the register-resident row kernels of each
# element type, and every file it includes from the tree.
ROWREG_SOURCES = ("rowreg.cuh", "device_common.cuh", "internal.h")


_COMMENT = re.compile(rb"/\*.*?\*/|//[^\n]*", re.S)


def kernel_source_hash(dtype: str = "bf16") -> str:
    """Hash of the sources of the plain row kernels of `dtype` (the unit that
    compiles them and the headers it includes, plus the build flags), with
    comments taken out and runs of white space made one space: other kernels,
    host-only files such as the selector, comments and layout do not change
    them."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "rmsnorm_fwd_gb300", "csrc")
    paths = [os.path.join(csrc, f) for f in (f"rowreg_{dtype}.cu",) + ROWREG_SOURCES]
    paths.append(os.path.join(ROOT, "include", "rmsnorm.h"))
    for p in paths:
        with open(p, "rb") as fh:
            code = re.sub(rb"\s+", b" ", _COMMENT.sub(b" ", fh.read())).strip()
            h.update(os.path.basename(p).encode() + code)
    from rmsnorm_fwd_gb300 import _build
    h.update(repr((_build.GENCODE, _build.CFLAGS, _build.CUDA_FLAGS)).encode())
    return h.hexdigest()[:16]


def ncu_traffic(wl, variant: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources for this workload; else None."""
    workload = wl.name
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    try:
        text = open(path).read()
    except OSError:
        return None
    src = kernel_source_hash(wl.dtype)
    for m in re.finditer(r"^workload=(\S+) variant=(\S+) src=(\S+) dram_bytes_per_launch=(\d+)",
                         text, flags=re.M):
        if m.group(1) == workload and m.group(2) == variant and m.group(3) == src:
            return int(m.group(4))
    return None


def workload(args):
    """The named workload, or its inputs at another shape (--shape ROWSxHIDDEN:
    same element type, eps and distributions; for profiling other bodies)."""
    wl = inputs.WORKLOADS[args.workload]
    if args.shape:
        rows, hidden = (int(v) for v in args.shape.lower().split("x"))
        wl = wl.with_shape(rows, hidden)
    return wl


# ----------------------------------------------------------------- CPU oracle

def oracle_sample(wl, seconds: float, max_rows: int | None = None):
    """Time the CPU oracle, as it stands, on leading rows of the workload
    until `seconds` of work (one thread).  Returns (GB/s, rows/s, rows done,
    seconds)."""
    import oracle
    block = max(1, min(wl.rows, 256))
    sample = wl.with_shape(block)
    x, w = inputs.make_inputs(sample)
    oracle.rmsnorm(x[:1], w, wl.eps, wl.dtype)  # load the library outside the clock
    done = 0
    t0 = time.perf_counter()
    while True:
        n = block if max_rows is None else max(1, min(block, max_rows - done))
        oracle.rmsnorm(x[:n], w, wl.eps, wl.dtype)
        done += n
        el = time.perf_counter() - t0
        if el >= seconds or (max_rows is not None and done >= max_rows):
            break
    es = inputs.ITEMSIZE[wl.dtype]
    bytes_done = 2 * done * wl.hidden * es + wl.hidden * es
    return bytes_done / el / 1e9, done / el, done, el


def oracle_sample_parallel(wl, seconds: float, threads: int):
    """The same oracle run row-parallel: `threads` host threads each
    normalise their own block of the workload's leading rows (the C call
    releases the interpreter lock) until `seconds` have passed.  Returns
    (GB/s, rows/s, rows done, seconds)."""
    import threading as th
    from concurrent.futures import ThreadPoolExecutor

    import oracle
    block = max(1, min(wl.rows, 64))
    x, w = inputs.make_inputs(wl.with_shape(block))
    oracle.rmsnorm(x[:1], w, wl.eps, wl.dtype)
    stop = th.Event()

    def worker(_):
        done = 0
        while not stop.is_set():
            oracle.rmsnorm(x, w, wl.eps, wl.dtype)
            done += block
        return done

    t0 = time.perf_counter()
    with ThreadPoolExecutor(max_workers=threads) as ex:
        futs = [ex.submit(worker, i) for i in range(threads)]
        time.sleep(seconds)
        stop.set()
        done = sum(f.result() for f in futs)
    el = time.perf_counter() - t0
    es = inputs.ITEMSIZE[wl.dtype]
    bytes_done = 2 * done * wl.hidden * es + wl.hidden * es
    return bytes_done / el / 1e9, done / el, done, el


def run_reference(args, world, rank):
    """--impl reference: the oracle timed on the host cores (rank 0 only)."""
    if rank != 0:
        return 0
    import oracle
    wl = workload(args)
    es = inputs.ITEMSIZE[wl.dtype]
    x, w = inputs.make_inputs(wl.with_shape(min(wl.rows, 64)))
    oracle.rmsnorm(x[:1], w, wl.eps, wl.dtype)
    t0 = time.perf_counter()
    oracle.rmsnorm(x[:8], w, wl.eps, wl.dtype)
    t_row = (time.perf_counter() - t0) / 8
    budget = args.reference_budget_s / max(1, args.steps + args.warmup)
    rows_per_step = int(max(1, min(x.shape[0], budget / max(t_row, 1e-9))))
    xs = x[:rows_per_step]
    for _ in range(args.warmup):
        oracle.rmsnorm(xs, w, wl.eps, wl.dtype)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.rmsnorm(xs, w, wl.eps, wl.dtype)
    el = time.perf_counter() - t0
    step_bytes = 2 * rows_per_step * wl.hidden * es + wl.hidden * es
    value = step_bytes * args.steps / el / 1e9
    sample = (f"{rows_per_step} of {wl.rows} rows x {wl.hidden} per step "
              f"({wl.dtype}, seeded workload inputs), {args.steps} steps")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(el / args.steps * 1e3, 6), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "rows": wl.rows, "hidden": wl.hidden, "eps": wl.eps,
                   "io_dtype": wl.dtype, "rows_per_step_sampled": rows_per_step},
        "rows_per_s": round(rows_per_step * args.steps / el, 2),
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    if args.cpu_seconds > 0:   # context: the same oracle on every host core
        ncores = os.cpu_count() or 1
        pg, prps, pdone, pel = oracle_sample_parallel(wl, min(args.cpu_seconds, 5.0), ncores)
        line["cpu_baseline"]["row_parallel"] = {
            "value": round(pg, 5), "unit": UNIT, "cores": ncores,
            "sample": (f"the same oracle on {ncores} host threads, each repeating the first "
                       f"{min(wl.rows, 64)} rows: {pdone} rows x {wl.hidden} in {pel:.1f} s"),
            "rows_per_s": round(prps, 2)}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------- GPU arm

def to_torch(a, dtype: str, torch):
    if dtype == "f32":
        return torch.from_numpy(a)
    import numpy as np
    return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16 if dtype == "bf16"
                                                      else torch.float16)


def run_ours(args, world, rank, local):
    import torch

    import rmsnorm_fwd_gb300 as rn

    if not torch.cuda.is_available():
        print(json.dumps({"error": "bench.py needs a CUDA device (GB300)"}), flush=True)
        return 1
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist = init_dist(world, "nccl")
    wl = workload(args)
    es = inputs.ITEMSIZE[wl.dtype]
    step_bytes = wl.bytes_per_call

    x_np, w_np = inputs.make_inputs(wl, seed=rank)
    x_host = to_torch(x_np, wl.dtype, torch)
    w_host = to_torch(w_np, wl.dtype, torch)
    set_bytes = 2 * wl.rows * wl.hidden * es
    nsets = max(2, -(-3 * L2_BYTES // set_bytes))
    xs = [x_host.to(device) for _ in range(nsets)]
    ys = [torch.empty_like(xs[0]) for _ in range(nsets)]
    w = w_host.to(device)

    rn.ensure_context(local)
    stream = torch.cuda.current_stream(device)
    sptr = stream.cuda_stream
    plan = rn.Plan()
    dt = rn.DTYPE_CODES[wl.dtype]
    rn.rmsnorm_fwd_ex(xs[0].data_ptr(), w.data_ptr(), ys[0].data_ptr(), wl.rows, wl.hidden,
                      wl.eps, dt, sptr, rn.VARIANT_AUTO, plan)
    variant = rn.VARIANT_NAMES[plan.variant]
    fwd = rn._load().rmsnorm_fwd_ex
    xp = [t.data_ptr() for t in xs]
    yp = [t.data_ptr() for t in ys]
    wp = w.data_ptr()
    pref = rn.ctypes.byref(plan)  # launch exactly the selector's plan every step

    def step(i):
        rc = fwd(xp[i % nsets], wp, yp[i % nsets], wl.rows, wl.hidden, wl.eps, dt, sptr, 0, pref)
        if rc != rn.OK:
            raise rn.RmsnormError(rc, "rmsnorm_fwd_ex")

    if args.profile_graph <= 0 and args.profile_range <= 0:
        # The sampler's start-up pause comes before the warm-up, so the first
        # timed region follows the warm-up launches with no idle gap.
        sampler = ClockSampler(local)
        sampler.start()
    for i in range(max(3, args.warmup)):
        step(i)
    torch.cuda.synchronize()

    if args.profile_graph > 0:
        # For a profiler that takes a CUDA graph as one workload (ncu
        # --graph-profiling graph): N launches of the plan captured into one
        # graph on a side stream, then replayed once between
        # cudaProfilerStart and cudaProfilerStop.  The device runs the N
        # kernels back to back with no host launch gaps between them.
        gs = torch.cuda.Stream(device)
        g = torch.cuda.CUDAGraph()
        gptr = gs.cuda_stream

        def gstep(i):
            rc = fwd(xp[i % nsets], wp, yp[i % nsets], wl.rows, wl.hidden, wl.eps, dt, gptr, 0,
                     pref)
            if rc != rn.OK:
                raise rn.RmsnormError(rc, "rmsnorm_fwd_ex")

        with torch.cuda.stream(gs):
            with torch.cuda.graph(g, stream=gs):
                for i in range(args.profile_graph):
                    gstep(i)
        g.replay()  # untimed replay: the graph's own first launch
        torch.cuda.synchronize()
        torch.cuda.profiler.start()
        g.replay()
        torch.cuda.synchronize()
        torch.cuda.profiler.stop()
        if rank == 0:
            print(json.dumps({"profile_graph": {
                "launches": args.profile_graph, "workload": wl.name, "variant": variant,
                "plan": plan.as_dict(), "sets": nsets,
                "algorithmic_bytes_per_launch": step_bytes}}), flush=True)
        return 0

    if args.profile_range > 0:
        # For a profiler's range replay (ncu --replay-mode range
        # --profile-from-start off): exactly N back-to-back launches of the
        # plan between cudaProfilerStart and cudaProfilerStop, nothing else.
        torch.cuda.profiler.start()
        for i in range(args.profile_range):
            step(i)
        torch.cuda.synchronize()
        torch.cuda.profiler.stop()
        if rank == 0:
            print(json.dumps({"profile_range": {
                "launches": args.profile_range, "workload": wl.name, "variant": variant,
                "plan": plan.as_dict(), "sets": nsets,
                "algorithmic_bytes_per_launch": step_bytes}}), flush=True)
        return 0

    K = args.steps
    R = max(1, args.regions)
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    poller = NvmlPoller(device)
    poller.start()
    t_wall0 = time.time()
    region_ms = []
    for reg in range(R):
        barrier(dist, device)
        torch.cuda.synchronize()
        start.record(stream)
        for i in range(K):
            step(reg * K + i)
        end.record(stream)
        torch.cuda.synchronize()
        barrier(dist, device)
        region_ms.append(reduce_max(start.elapsed_time(end), dist, device))
    t_wall1 = time.time()
    sampler.stop()
    poller.stop()
    # Each timed region holds nothing but this kernel's K back-to-back
    # launches on one stream, so its average launch duration (launch gaps
    # included) is the region's time / K.  Reported: the median region (the
    # regions are short, so one alone carries the run-to-run noise of a
    # sub-millisecond event pair), with the others beside it.
    max_ms = statistics.median(region_ms)
    max_kernel_ms = max_ms / K
    clocks = sampler.summary(t_wall0, t_wall1)
    nv = poller.summary(t_wall0, t_wall1)
    if nv is not None:
        clocks["nvml"] = nv
    status = rn.rmsnorm_get_device_status()

    # ---- e2e through the public API: x from pinned host memory, y back to
    # pinned host memory, every step (rmsnorm_fwd_host: with page-locked
    # buffers the kernel reads and writes host memory directly; the weight is
    # a resident parameter)
    E = args.e2e_steps
    xh = x_host.pin_memory()
    yh = torch.empty_like(xh).pin_memory()
    ws_bytes = 64 << 20
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=device)

    def e2e_step():
        rn.rmsnorm_fwd_host(xh.data_ptr(), w.data_ptr(), yh.data_ptr(), wl.rows, wl.hidden,
                            wl.eps, dt, ws.data_ptr(), ws_bytes, 0, sptr)

    e2e_gbs = None
    if E > 0:
        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        barrier(dist, device)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(E):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(dist, device)
        e2e_ms = reduce_max(e0.elapsed_time(e1), dist, device)
        e2e_gbs = world * E * step_bytes / (e2e_ms / 1e3) / 1e9

    value = world * K * step_bytes / (max_ms / 1e3) / 1e9
    peak, peak_kind = hbm_peak()
    achieved = step_bytes / (max_kernel_ms / 1e3) / 1e9
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": max(3, args.warmup), "ms_per_step": round(max_ms / K, 6),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {
            "workload": wl.name, "rows": wl.rows, "hidden": wl.hidden, "eps": wl.eps,
            "io_dtype": wl.dtype, "accumulate": "f32", "variant": variant,
            "plan": plan.as_dict(),
            "l2": (f"inputs larger than L2: {nsets} rotating x/y sets of "
                   f"{set_bytes / 1e6:.0f} MB ({nsets * set_bytes / 1e6:.0f} MB) vs 129 MB L2"),
            "parallelism": f"replicas x{world} (rows are independent; no collective)",
        },
        "rows_per_s": round(world * K * wl.rows / (max_ms / 1e3), 1),
        "pct_of_peak": round(100 * value / peak, 2),
        "pct_of_nominal_hbm": round(100 * value / NOMINAL_HBM_GBS, 2),
        "gpu_launches": K,
        "timing": {"regions": R, "launches_per_region": K, "statistic": "median region",
                   "region_ms": [round(t, 6) for t in region_ms],
                   "per_launch_ms_min": round(min(region_ms) / K, 6),
                   "per_launch_ms_max": round(max(region_ms) / K, 6),
                   "spread_pct": round(100 * (max(region_ms) - min(region_ms)) / max_ms, 2)},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_kind == "measured" else "fallback 6.8 TB/s",
                     "nominal_peak": NOMINAL_HBM_GBS,
                     "frac_of_nominal": round(achieved / NOMINAL_HBM_GBS, 4),
                     "nominal_source": "GB300 HBM3e nominal bandwidth, 7.9 TB/s",
                     "traffic": ncu_traffic(wl, variant),
                     "algorithmic_bytes_per_launch": step_bytes,
                     "kernel_ms_avg": round(max_kernel_ms, 6),
                     "kernel_ms_basis": "median timed region / launches (gaps included)"},
        "e2e": {"value": round(e2e_gbs, 2) if e2e_gbs is not None else None, "unit": UNIT,
                "steps": E, "api": "rmsnorm_fwd_host: pinned host x/y read and written by the "
                "kernel over NVLink-C2C; weight resident on the device",
                "h2d_bytes_per_step": int(xh.numel() * xh.element_size()),
                "d2h_bytes_per_step": int(yh.numel() * yh.element_size())},
        "clocks": clocks,
        "device_status": status,
    }
    if rank == 0 and world == 1 and args.cpu_seconds > 0:
        gbs, rps, rows_done, el = oracle_sample(wl, args.cpu_seconds)
        line["cpu_baseline"] = {
            "value": round(gbs, 5), "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": (f"first {min(wl.rows, 256)} rows of the same seeded workload, repeated: "
                       f"{rows_done} rows x {wl.hidden} in {el:.1f} s, one thread"),
            "rows_per_s": round(rps, 2)}
        ncores = os.cpu_count() or 1
        pg, prps, pdone, pel = oracle_sample_parallel(wl, min(args.cpu_seconds, 5.0), ncores)
        line["cpu_baseline"]["row_parallel"] = {
            "value": round(pg, 5), "unit": UNIT, "cores": ncores,
            "sample": (f"the same oracle on {ncores} host threads, each repeating the first "
                       f"{min(wl.rows, 64)} rows: {pdone} rows x {wl.hidden} in {pel:.1f} s"),
            "rows_per_s": round(prps, 2)}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def run_qk(args, world, rank, local):
    """--op qk_norm: the per-head QK norm on a fused [q | k | v] buffer
    (rmsnorm_qk_norm, one launch for q and k, in place), and, for context,
    the same heads stored contiguously normalised by two launches of the
    general RMSNorm entry point (the page's "normal RMSNorm" path)."""
    import torch

    import rmsnorm_fwd_gb300 as rn
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    wl = inputs.QK_WORKLOADS[args.qk_workload]
    es = inputs.ITEMSIZE[wl.dtype]
    buf, qw_np, kw_np = inputs.make_qk_inputs(wl, seed=rank)
    tdt = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[wl.dtype]
    host = torch.from_numpy(buf.view(np.int16) if wl.dtype != "f32" else buf)
    host = host.view(tdt) if wl.dtype != "f32" else host
    set_bytes = buf.size * es
    nsets = max(2, -(-3 * L2_BYTES // set_bytes))
    bufs = [host.to(device) for _ in range(nsets)]
    qw = torch.from_numpy(qw_np.view(np.int16)).view(tdt).to(device)
    kw = torch.from_numpy(kw_np.view(np.int16)).view(tdt).to(device)
    rn.ensure_context(local)
    stream = torch.cuda.current_stream(device)
    sptr = stream.cuda_stream
    dt = rn.DTYPE_CODES[wl.dtype]
    d, hq, hk, T = wl.head_dim, wl.q_heads, wl.k_heads, wl.tokens
    fn = rn._load().rmsnorm_qk_norm
    qp = [b.data_ptr() for b in bufs]

    def step(i):
        rc = fn(qp[i % nsets], qp[i % nsets] + hq * d * es, qw.data_ptr(), kw.data_ptr(), T, hq,
                hk, d, wl.width, wl.width, 0.0, wl.eps, dt, sptr)
        if rc != rn.OK:
            raise rn.RmsnormError(rc, "rmsnorm_qk_norm")

    def timed(fn_step, K):
        for i in range(max(3, args.warmup)):
            fn_step(i)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(K):
            fn_step(i)
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / K

    K = args.steps
    ms = timed(step, K)
    # the general entry point on contiguous q and k: two launches per step
    qc = [torch.empty(T * hq * d, dtype=tdt, device=device) for _ in range(nsets)]
    kc = [torch.empty(T * hk * d, dtype=tdt, device=device) for _ in range(nsets)]
    gen = rn._load().rmsnorm_fwd

    def step2(i):
        j = i % nsets
        gen(qc[j].data_ptr(), qw.data_ptr(), qc[j].data_ptr(), T * hq, d, wl.eps, dt, sptr)
        gen(kc[j].data_ptr(), kw.data_ptr(), kc[j].data_ptr(), T * hk, d, wl.eps, dt, sptr)

    ms2 = timed(step2, K)
    value = wl.bytes_per_call / (ms / 1e3) / 1e9
    peak, peak_kind = hbm_peak()
    line = {
        "metric": "QK-norm achieved HBM GB/s (fused QKV layout, one launch for q and k)",
        "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": max(3, args.warmup), "ms_per_step": round(ms, 6), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": wl.name, "tokens": T, "q_heads": hq, "k_heads": hk,
                   "head_dim": d, "io_dtype": wl.dtype, "layout": "fused [q|k|v] per token",
                   "l2": f"{nsets} rotating buffers of {set_bytes / 1e6:.0f} MB"},
        "gpu_launches": K,
        "roofline": {"bound": "hbm", "achieved": round(value, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(value / peak, 4), "peak_source": peak_kind,
                     "algorithmic_bytes_per_launch": wl.bytes_per_call},
        "general_two_launches": {"ms_per_step": round(ms2, 6),
                                 "GBps": round(wl.bytes_per_call / (ms2 / 1e3) / 1e9, 2),
                                 "speedup_of_qk_norm": round(ms2 / ms, 3)},
        "device_status": rn.rmsnorm_get_device_status(),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def run_epi(args, world, rank, local):
    """--op bias | mxfp8 | mxfp4 | nvfp4: the row norm with the weight offset
    (1.0 unless --weight-bias), or with a fused block-scaled output (codes and
    one scale per 32 or 16 elements; no weight offset unless --weight-bias),
    on the chosen workload; the plain kernel on the same inputs is timed
    beside it for context."""
    import torch

    import rmsnorm_fwd_gb300 as rn
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    wl = workload(args)
    es = inputs.ITEMSIZE[wl.dtype]
    x_np, w_np = inputs.make_inputs(wl, seed=rank)
    x_host = to_torch(x_np, wl.dtype, torch)
    w = to_torch(w_np, wl.dtype, torch).to(device)
    epi = rn.EPI_CODES[args.op]
    mx = epi in rn.QUANT_FORMATS
    n = wl.rows * wl.hidden
    block, bits = rn.QUANT_FORMATS.get(epi, (1, 8 * es))
    out_bytes = (n * bits // 8 + n // block) if mx else n * es
    step_bytes = n * es + wl.hidden * es + out_bytes
    set_bytes = n * es + out_bytes
    nsets = max(2, -(-3 * L2_BYTES // set_bytes))
    xs = [x_host.to(device) for _ in range(nsets)]
    if mx:
        ys = [torch.empty(n * bits // 8, dtype=torch.uint8, device=device) for _ in range(nsets)]
        ss = [torch.empty(n // block, dtype=torch.uint8, device=device) for _ in range(nsets)]
    else:
        ys = [torch.empty_like(xs[0]) for _ in range(nsets)]
        ss = [None] * nsets
    rn.ensure_context(local)
    stream = torch.cuda.current_stream(device)
    sptr = stream.cuda_stream
    dt = rn.DTYPE_CODES[wl.dtype]
    # the weight offset: 1.0 for --op bias; none (-0.0, the identity) for the
    # block-scaled outputs unless --weight-bias says otherwise
    bias = args.weight_bias if args.weight_bias is not None else \
        (1.0 if epi == rn.EPI_BIAS else -0.0)
    gscale = 1.0 / (448 * 6) * 4.0  # a per-tensor NVFP4 scale for values of magnitude ~4
    plan = rn.Plan()
    rn.rmsnorm_fwd_epilogue_ex(xs[0].data_ptr(), w.data_ptr(), ys[0].data_ptr(),
                               ss[0].data_ptr() if mx else None, wl.rows, wl.hidden, epi, bias,
                               wl.eps, dt, sptr, rn.VARIANT_AUTO, plan, gscale)
    fn = rn._load().rmsnorm_fwd_epilogue_ex
    pref = rn.ctypes.byref(plan)
    xp = [t.data_ptr() for t in xs]
    yp = [t.data_ptr() for t in ys]
    sp = [t.data_ptr() if t is not None else None for t in ss]

    def step(i):
        j = i % nsets
        rc = fn(xp[j], w.data_ptr(), yp[j], sp[j], wl.rows, wl.hidden, epi, bias, gscale, wl.eps,
                dt, sptr, 0, pref)
        if rc != rn.OK:
            raise rn.RmsnormError(rc, "rmsnorm_fwd_epilogue_ex")

    ys_plain = [torch.empty_like(xs[0]) for _ in range(nsets)]
    gen = rn._load().rmsnorm_fwd

    def step_plain(i):
        j = i % nsets
        gen(xp[j], w.data_ptr(), ys_plain[j].data_ptr(), wl.rows, wl.hidden, wl.eps, dt, sptr)

    def timed(fn_step, K):
        for i in range(max(3, args.warmup)):
            fn_step(i)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(K):
            fn_step(i)
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / K

    K = args.steps
    sampler = ClockSampler(local)
    sampler.start()
    t0 = time.time()
    ms = timed(step, K)
    t1 = time.time()
    sampler.stop()
    ms_plain = timed(step_plain, K)
    value = step_bytes / (ms / 1e3) / 1e9
    peak, peak_kind = hbm_peak()
    plain_bytes = wl.bytes_per_call
    line = {
        "metric": (f"RMSNorm + {args.op.upper()} output achieved HBM GB/s" if mx else
                   "RMSNorm with weight offset achieved HBM GB/s"),
        "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": max(3, args.warmup), "ms_per_step": round(ms, 6), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": wl.name, "rows": wl.rows, "hidden": wl.hidden,
                   "io_dtype": wl.dtype, "epilogue": rn.EPI_NAMES[epi], "weight_bias": bias,
                   "global_scale": gscale if epi == rn.EPI_NVFP4 else None,
                   "variant": rn.VARIANT_NAMES[plan.variant], "plan": plan.as_dict(),
                   "l2": f"{nsets} rotating input/output sets of {set_bytes / 1e6:.0f} MB"},
        "rows_per_s": round(wl.rows / (ms / 1e3), 1),
        "gpu_launches": K,
        "roofline": {"bound": "hbm", "achieved": round(value, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(value / peak, 4), "peak_source": peak_kind,
                     "algorithmic_bytes_per_launch": step_bytes},
        "plain_output_same_rows": {"ms_per_step": round(ms_plain, 6),
                                   "GBps": round(plain_bytes / (ms_plain / 1e3) / 1e9, 2),
                                   "time_ratio": round(ms / ms_plain, 4)},
        "clocks": sampler.summary(t0, t1),
        "device_status": rn.rmsnorm_get_device_status(),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def run_latency(args, world, rank, local):
    """--op latency: per-call time of the automatic plan on one workload --
    back-to-back launches (one event pair over K), the same K launches
    replayed from a CUDA graph, and cold calls (L2 flushed by writing a
    buffer of twice its size before each, one event pair around each call;
    median) -- with the GB/s each implies."""
    import torch

    import rmsnorm_fwd_gb300 as rn
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    wl = workload(args)
    x_np, w_np = inputs.make_inputs(wl, seed=rank)
    x = to_torch(x_np, wl.dtype, torch).to(device)
    w = to_torch(w_np, wl.dtype, torch).to(device)
    y = torch.empty_like(x)
    rn.ensure_context(local)
    stream = torch.cuda.current_stream(device)
    sptr = stream.cuda_stream
    dt = rn.DTYPE_CODES[wl.dtype]
    plan = rn.Plan()
    rn.rmsnorm_fwd_ex(x.data_ptr(), w.data_ptr(), y.data_ptr(), wl.rows, wl.hidden, wl.eps, dt,
                      sptr, rn.VARIANT_AUTO, plan)
    fwd = rn._load().rmsnorm_fwd_ex
    pref = rn.ctypes.byref(plan)
    args_ = (x.data_ptr(), w.data_ptr(), y.data_ptr(), wl.rows, wl.hidden, wl.eps, dt)

    def call(s):
        rc = fwd(*args_, s, 0, pref)
        if rc != rn.OK:
            raise rn.RmsnormError(rc, "rmsnorm_fwd_ex")

    K = args.steps
    for _ in range(max(3, args.warmup)):
        call(sptr)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(K):
        call(sptr)
    e1.record(stream)
    torch.cuda.synchronize()
    warm_us = e0.elapsed_time(e1) / K * 1e3

    cs = torch.cuda.Stream(device)

    def graph_time(fn):
        """Per-call us of K calls of fn(stream) captured in a CUDA graph, replayed."""
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cs):
            for _ in range(K):
                fn(cs.cuda_stream)
        g.replay()
        torch.cuda.synchronize()
        e0.record(stream)
        g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / K * 1e3

    graph_us = graph_time(call)
    # The same calls without programmatic dependent launch, and the floor: a
    # kernel that does nothing but write one float, replayed the same way.
    pdl_was = rn.rmsnorm_get_pdl()
    rn.rmsnorm_set_pdl(False)
    graph_nopdl_us = graph_time(call)
    rn.rmsnorm_set_pdl(pdl_was)
    one = torch.zeros(1, dtype=torch.float32, device=device)
    floor_us = graph_time(lambda _s: one.fill_(1.0))

    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=device)
    cold = []
    for i in range(min(K, 200)):
        flush.fill_(float(i))
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        call(sptr)
        b.record(stream)
        b.synchronize()
        cold.append(a.elapsed_time(b) * 1e3)
    cold_us = statistics.median(cold)
    nbytes = wl.bytes_per_call

    def gbs(us):
        return round(nbytes / (us * 1e-6) / 1e9, 2)

    line = {
        "metric": "RMSNorm per-call time (us) and GB/s", "value": round(graph_us, 3),
        "unit": "us per call (graph-replayed)", "n_gpus": world, "steps": K,
        "warmup": max(3, args.warmup), "higher_is_better": False, "data": "synthetic",
        "dtype": "f32", "config": {"workload": wl.name, "rows": wl.rows, "hidden": wl.hidden,
                                   "io_dtype": wl.dtype,
                                   "variant": rn.VARIANT_NAMES[plan.variant],
                                   "plan": plan.as_dict()},
        "back_to_back_us": round(warm_us, 3), "back_to_back_GBps": gbs(warm_us),
        "graph_us": round(graph_us, 3), "graph_GBps": gbs(graph_us),
        "graph_us_without_pdl": round(graph_nopdl_us, 3),
        "graph_floor_us": round(floor_us, 3),
        "graph_floor_basis": "a one-element fill kernel, K launches replayed from a graph",
        "cold_median_us": round(cold_us, 3), "cold_GBps": gbs(cold_us),
        "cold_basis": "L2 flushed (2 x L2 written) before each call; one event pair per call",
        "gpu_launches": K, "device_status": rn.rmsnorm_get_device_status(),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--shape", default=None,
                    help="ROWSxHIDDEN: the workload's inputs at another shape (profiling)")
    ap.add_argument("--profile-range", type=int, default=0,
                    help="N > 0: only N launches between cudaProfilerStart/Stop (for ncu's "
                         "range replay), then exit")
    ap.add_argument("--profile-graph", type=int, default=0,
                    help="N > 0: only N launches captured in one CUDA graph, replayed once "
                         "between cudaProfilerStart/Stop (for ncu --graph-profiling graph), "
                         "then exit")
    ap.add_argument("--regions", type=int, default=5,
                    help="timed regions of K launches each; the median region is reported")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=inputs.HEADLINE, choices=sorted(inputs.WORKLOADS))
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--reference-budget-s", type=float, default=60.0)
    ap.add_argument("--op", choices=["rmsnorm", "qk_norm", "bias", "mxfp8", "mxfp4", "nvfp4",
                                     "latency"], default="rmsnorm")
    ap.add_argument("--qk-workload", default="qk_bf16_16384tok_32q8k_128",
                    choices=sorted(inputs.QK_WORKLOADS))
    ap.add_argument("--weight-bias", type=float, default=None,
                    help="weight offset for --op bias|mxfp8|mxfp4|nvfp4 (default 1.0 for bias, "
                         "-0.0 = no offset for the block-scaled outputs)")
    args = ap.parse_args(argv)
    world, rank, local = dist_env()
    if args.op == "qk_norm":
        return run_qk(args, world, rank, local)
    if args.op in ("bias", "mxfp8", "mxfp4", "nvfp4"):
        return run_epi(args, world, rank, local)
    if args.op == "latency":
        return run_latency(args, world, rank, local)
    if args.impl == "reference":
        return run_reference(args, world, rank)
    return run_ours(args, world, rank, local)


if __name__ == "__main__":
    sys.exit(main())
