"""Benchmark: fused GEMM + elementwise epilogue on GB300, one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference|vendor]
                    [--workload NAME]

(--impl vendor times torch.matmul, i.e. cuBLAS, on the workload's A and B
alone, for context: it is not one of the two arms.)

A step is one pass of the whole hot path over one batch of synthetic input:
one fused GEMM + epilogue launch (plan creation is outside the timed region).
By default 20 warm-up steps, then 100 timed steps, each bracketed by CUDA
events on the launch stream; longer runs (--steps 500) settle lower, under
the board's power cap.
The default workload is the 8192^3 fp16 GEMM with the Alpha-Beta-Scaling
epilogue (Y = accum; D = 2*accum + C + 3*X), whose inputs (512 MiB) are larger
than twice the 129 MB L2, so no L2 flush is needed between steps; workloads
with smaller inputs flush the L2 before every timed step.

Reported next to the device-timed value:
  roofline      the fused kernel's achieved TFLOP/s (CUDA events on its
                launch stream) against the measured dense bf16 peak
                (MEASURED_PEAKS.json; fp16 has the same nominal rate)
  e2e           the same metric with pinned-host inputs copied in and the
                outputs copied back inside every timed step
  unfused       the same GEMM storing fp32 accum + a separate elementwise
                kernel (the bytes fusion saves)
  cpu_baseline  the fp64 CPU oracle on a bounded sample of rows
  clocks        clock, power and throttle-reason samples taken during the
                timed region (NVML every 2 ms, else nvidia-smi every 50 ms)

Under torchrun (N > 1) every rank runs an independent replica on its own GPU
(the problem has no exchange step); value = all ranks' FLOPs / max time.
"""
import argparse
import atexit
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fused GEMM+epilogue TFLOP/s and % of GB300 dense FP16 peak (1 GPU)"
DEFAULT_WORKLOAD = "alpha_beta_x_8192"
L2_BYTES = 129 * 1000 * 1000  # GB300 L2
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference", "vendor"],
                    help="vendor: torch.matmul (cuBLAS) on A and B alone, for context")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--mnk", default=None,
                    help="M,N,K override of the workload's sizes (profiling on a smaller case)")
    ap.add_argument("--opt", default="",
                    help="plan options, e.g. cta_group=2,tile_n=256,stages=5,raster_group=8")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-unfused", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other workloads' figures (the configs object)")
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def roofline(flops, alg_bytes, ms, traffic):
    """The launch against the bound its arithmetic intensity sets: tensor
    (flops / measured dense peak) or HBM (algorithmic bytes / measured copy
    bandwidth), whichever takes longer; the other fraction rides along."""
    pk, pk_src = peaks()
    tflops = float(pk.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    tflops_sus = float(pk.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    gbs = float(pk.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    sec = ms * 1e-3
    t_frac = flops / sec / 1e12 / tflops
    h_frac = alg_bytes / sec / 1e9 / gbs
    extra = {"alg_bytes_per_launch": alg_bytes, "flops_per_launch": flops,
             "frac_of_sustained": flops / sec / 1e12 / tflops_sus,
             "frac_of_nominal_2250": flops / sec / 1e12 / 2250.0,
             "tensor_frac": t_frac, "hbm_frac": h_frac}
    if alg_bytes / (gbs * 1e9) > flops / (tflops * 1e12):
        return dict({"bound": "hbm", "achieved": alg_bytes / sec / 1e9, "peak": gbs,
                     "unit": "GB/s", "frac": h_frac, "traffic": traffic,
                     "peak_source": "%s copy bandwidth" % pk_src}, **extra)
    return dict({"bound": "tensor", "achieved": flops / sec / 1e12, "peak": tflops,
                 "unit": "TFLOP/s", "frac": t_frac, "traffic": traffic,
                 "peak_source": "%s bf16 dense burst (fp16 has the same nominal rate)" % pk_src},
                **extra)


# host-only sources: they choose a launch's configuration, which a traffic
# record matches separately (its "plan"), but hold no device code
HOST_ONLY_SOURCES = ("plan.cu", "jit.cu")


def kernel_source_hash():
    """Hash of the device code: every source under csrc/ but the host-only
    ones."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "dense_gemm_elementwise_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name in HOST_ONLY_SOURCES:
            continue
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload, plan=None):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current device code and, where the record names the launch
    configuration it was taken with, on the same configuration as `plan`."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    ent = d.get(workload)
    if not ent or ent.get("kernel_hash") != kernel_source_hash():
        return None
    want = ent.get("plan")
    if want is not None and (plan is None or any(plan.get(k) != v for k, v in want.items())):
        return None
    return ent.get("dram_bytes_per_launch")


# ------------------------------------------------------------ clocks ---

# NVML clock-event reason bits (nvml.h, nvmlClocksEventReason*)
NVML_REASON_BITS = (("sw_power_cap", 0x4), ("hw_slowdown", 0x8),
                    ("sw_thermal_slowdown", 0x20), ("hw_thermal_slowdown", 0x40))


def nvml_sampler_main(bus, period_ms):
    """Body of ClockSampler's child process: read-only NVML queries of the GPU
    at PCI address `bus` every `period_ms`, one line per sample (wall time,
    SM clock and its maximum in MHz, power in W, clock-event reason bits),
    until it is stopped, its output closes or its parent exits.  Exits 3
    when NVML or the device cannot be opened."""
    import ctypes
    try:
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            sys.exit(3)
        try:
            reasons_fn = lib.nvmlDeviceGetCurrentClocksEventReasons
        except AttributeError:
            reasons_fn = lib.nvmlDeviceGetCurrentClocksThrottleReasons
    except OSError:
        sys.exit(3)
    h = ctypes.c_void_p()
    if lib.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(h)) != 0:
        sys.exit(3)
    clk, smax, mw, bits = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
    sm_clock = 1  # NVML_CLOCK_SM
    lib.nvmlDeviceGetMaxClockInfo(h, sm_clock, ctypes.byref(smax))
    period = max(period_ms, 1) / 1000.0
    out = sys.stdout
    parent = os.getppid()
    while os.getppid() == parent:  # a parent that died without stopping us: exit
        ok = lib.nvmlDeviceGetClockInfo(h, sm_clock, ctypes.byref(clk)) == 0
        if lib.nvmlDeviceGetPowerUsage(h, ctypes.byref(mw)) != 0:
            mw.value = 0
        if reasons_fn(h, ctypes.byref(bits)) != 0:
            bits.value = 0
        if ok:
            try:
                out.write("%.6f,%d,%d,%.3f,%d\n" % (time.time(), clk.value, smax.value,
                                                     mw.value / 1000.0, bits.value))
                out.flush()
            except (BrokenPipeError, OSError):
                return
        time.sleep(period)


class ClockSampler:
    """Clock, power and throttle-reason samples of the GPU, each stamped with
    the wall time it was taken at; window(t0, t1) keeps the samples between
    two time.time() marks.  Preferred source: a child process that polls
    NVML (read-only queries) every 2 ms, so even a timed region of ~10 ms
    holds samples; else nvidia-smi every 50 ms.  The sampler starts before
    the inputs are made, so its start-up is over well before the timed
    region.  Lines are read by a thread as they come, so none are lost when
    the child is stopped."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    NVML_PERIOD_MS = 2

    def __init__(self, gpu_index, bus=None):
        self.proc = None
        self.gpu = gpu_index
        self.bus = bus
        self.source = None
        self.lines = []
        self.thread = None

    def _spawn(self, cmd):
        import threading
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
            return False
        self.lines = []
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        return True

    def start(self):
        import shutil
        atexit.register(self.stop)  # never leave the child running
        if self.bus and self._spawn([sys.executable, os.path.abspath(__file__), "--nvml-sampler",
                                     self.bus, str(self.NVML_PERIOD_MS)]):
            t_end = time.time() + 5.0
            while not self.lines and self.proc.poll() is None and time.time() < t_end:
                time.sleep(0.01)
            if self.lines:
                self.source = "nvml every %d ms" % self.NVML_PERIOD_MS
                return self
            self.stop()
            self.proc = None
        cmd = ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
               "--format=csv,noheader,nounits", "-lms", "50"]
        if shutil.which("stdbuf"):
            cmd = ["stdbuf", "-oL"] + cmd
        if self._spawn(cmd):
            self.source = "nvidia-smi every 50 ms"
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line))

    def stop(self):
        if self.proc is None or self.proc.poll() is not None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            self.proc.wait()
        self.thread.join(timeout=5)

    def _samples(self):
        import datetime
        out = []
        for received, line in list(self.lines):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == 5:  # NVML child: time, sm, max, power, reason bits
                try:
                    t, sm, smax, pw, bits = (float(parts[0]), float(parts[1]), float(parts[2]),
                                             float(parts[3]), int(parts[4]))
                except ValueError:
                    continue
                out.append((t, sm, smax, pw, [n for n, b in NVML_REASON_BITS if bits & b]))
                continue
            if len(parts) < 9:
                continue
            try:
                t = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                t = received  # unknown timestamp format: the time the line arrived
            try:
                sm, smax, pw = float(parts[1]), float(parts[2]), float(parts[3])
            except ValueError:
                continue
            active = [n for n, v in zip(self.REASONS, parts[5:9]) if v.lower().startswith("active")]
            out.append((t, sm, smax, pw, active))
        return out

    def window(self, t0, t1):
        """Statistics of the samples taken in [t0, t1] (wall clock).  A region
        shorter than the sampling period may hold none: then the nearest
        samples within 0.25 s of it are used, and "window" says so."""
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None,
                    "reasons": ["neither NVML nor nvidia-smi available"]}
        samples = self._samples()
        inside = [x for x in samples if t0 <= x[0] <= t1]
        n_inside = len(inside)
        where = "timed region"
        if not inside:
            inside = [x for x in samples if t0 - 0.25 <= x[0] <= t1 + 0.25]
            where = "timed region +- 0.25 s (no sample inside it)"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no clock sample"],
                    "samples": 0, "samples_total": len(samples), "source": self.source}
        return {"sm_mhz": statistics.median(x[1] for x in inside),
                "sm_max_mhz": max(x[2] for x in inside),
                "reasons": sorted({r for x in inside for r in x[4]}),
                "samples": len(inside), "samples_inside_region": n_inside, "window": where,
                "source": self.source,
                "window_s": round(t1 - t0, 3),
                "power_w_median": statistics.median(x[3] for x in inside),
                "power_w_max": max(x[3] for x in inside)}


# ------------------------------------------------------------ helpers ---

def _numa_nodes_of(addr_lo, addr_hi):
    """NUMA nodes holding the pages of [addr_lo, addr_hi) of this process
    (from /proc/self/numa_maps: per mapping, pages resident on each node)."""
    nodes = {}
    try:
        with open("/proc/self/numa_maps") as f:
            lines = f.readlines()
        with open("/proc/self/maps") as f:
            spans = {}
            for ln in f:
                lo, hi = (int(x, 16) for x in ln.split()[0].split("-"))
                spans[lo] = hi
    except OSError:
        return None
    for ln in lines:
        parts = ln.split()
        lo = int(parts[0], 16)
        hi = spans.get(lo, lo)
        if hi <= addr_lo or lo >= addr_hi:
            continue
        for p in parts[1:]:
            if p.startswith("N") and "=" in p:
                k, v = p[1:].split("=", 1)
                if k.isdigit():
                    nodes[int(k)] = nodes.get(int(k), 0) + int(v)
    return nodes


def gpu_pci_bus(local):
    """PCI address of CUDA device `local` (domain:bus:device.function), or
    None where torch does not report it."""
    import torch
    try:
        p = torch.cuda.get_device_properties(local)
        return "%04x:%02x:%02x.0" % (p.pci_domain_id, p.pci_bus_id, p.pci_device_id)
    except (AttributeError, RuntimeError):
        return None


def host_numa_note(local, tensors=()):
    """Where the end-to-end leg's pinned host buffers sit relative to the
    GPU: the GPU's NUMA node (sysfs), the nodes of this process's CPUs, and
    the nodes holding the buffers' pages."""
    out = {}
    bus = gpu_pci_bus(local)
    if bus:
        try:
            with open("/sys/bus/pci/devices/%s/numa_node" % bus.lower()) as f:
                out["gpu_numa_node"] = int(f.read().strip())
        except (OSError, ValueError):
            out["gpu_numa_node"] = None
        out["gpu_pci"] = bus.lower()
    try:
        cpus = sorted(os.sched_getaffinity(0))
        cnodes = set()
        for c in cpus:
            d = "/sys/devices/system/cpu/cpu%d" % c
            for name in os.listdir(d):
                if name.startswith("node") and name[4:].isdigit():
                    cnodes.add(int(name[4:]))
        out["cpu_numa_nodes"] = sorted(cnodes)
    except OSError:
        pass
    pages = {}
    for t in tensors:
        lo = t.data_ptr()
        got = _numa_nodes_of(lo, lo + t.numel() * t.element_size())
        for k, v in (got or {}).items():
            pages[k] = pages.get(k, 0) + v
    if tensors:
        out["buffer_pages_by_node"] = {str(k): v for k, v in sorted(pages.items())}
    return out


def dist_setup(n):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("gloo", rank=rank, world_size=world)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def oracle_sample(w, A, Bm, aux, scalars, rows, threads):
    import numpy as np

    import oracle
    from dense_gemm_elementwise_gb300 import workloads as W
    t0 = time.perf_counter()
    oracle.gemm_epilogue(w.L, w.M, w.N, w.K, w.ab, W.to_codes(A), W.to_codes(Bm),
                         [W.to_codes(a) for a in aux], [s[2] for s in w.aux], scalars, w.dag,
                         [dt for _, dt in w.outs], rows=np.asarray(rows, dtype=np.int64),
                         threads=threads)
    return time.perf_counter() - t0


def cpu_baseline(w, inputs, target_s=10.0):
    """The oracle as it stands, timed on this host's cores on a bounded
    sample of output rows (each row: N*K multiply-adds)."""
    import oracle
    threads = oracle.threads_default()
    A, Bm, aux, scalars = inputs
    n = max(threads, 1)
    t = oracle_sample(w, A, Bm, aux, scalars, list(range(n)), threads)
    rows = int(min(w.L * w.M, max(n, n * max(1.0, target_s / max(t, 1e-3)))))
    rows = max(n, (rows // n) * n)
    t = oracle_sample(w, A, Bm, aux, scalars, list(range(rows)), threads)
    tflops = 2.0 * rows * w.N * w.K / t / 1e12
    return {"value": tflops, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": "%d of %d output rows (%d x %d multiply-adds each), fp64, %.1f s wall"
                      % (rows, w.L * w.M, w.N, w.K, t)}


def workload_config(w, world):
    """The workload's identity: the same keys in both arms' lines."""
    return {"workload": w.name, "L": w.L, "M": w.M, "N": w.N, "K": w.K,
            "ab_dtype": w.ab, "acc_dtype": "f32", "epilogue_dtype": "f32",
            "outs": [n + ":" + dt for n, dt in w.outs],
            "parallelism": "replicas" if world > 1 else "single"}


def grouped_config(w, world):
    return {"workload": w.name, "problems": len(w.problems), "ab_dtype": w.ab,
            "acc_dtype": "f32", "epilogue_dtype": "f32",
            "outs": [n + ":" + dt for n, dt in w.outs],
            "flops_per_step": w.flops(), "alg_bytes_per_step": w.alg_bytes(),
            "parallelism": "replicas" if world > 1 else "single"}


# ------------------------------------------------------- reference arm ---

def run_reference(args, w):
    """The oracle, as it stands, on the same workload: every step evaluates
    a bounded sample of output rows of it on the host cores."""
    import oracle
    from dense_gemm_elementwise_gb300 import workloads as W
    rank, world, _ = dist_setup(args.gpus)
    if rank != 0:
        return
    inputs = W.make_inputs(w)
    A, Bm, aux, scalars = inputs
    threads = oracle.threads_default()
    rows_per_step = 2 * threads
    n_rows = w.L * w.M
    for i in range(args.warmup):
        oracle_sample(w, A, Bm, aux, scalars, [(i * rows_per_step + r) % n_rows
                                                for r in range(rows_per_step)], threads)
    total = 0.0
    for i in range(args.steps):
        rows = [((args.warmup + i) * rows_per_step + r) % n_rows for r in range(rows_per_step)]
        total += oracle_sample(w, A, Bm, aux, scalars, sorted(set(rows)), threads)
    ms = total / args.steps * 1e3
    value = 2.0 * rows_per_step * w.N * w.K / (ms * 1e-3) / 1e12
    sample = "%d output rows per step of %d (%d x %d multiply-adds each), fp64" % (
        rows_per_step, n_rows, w.N, w.K)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic",
            "config": workload_config(w, args.gpus),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------ vendor context ---

def run_vendor(args, w):
    """Context, not an arm of the comparison: the vendor GEMM (torch.matmul,
    i.e. cuBLAS) on the workload's A and B alone, no epilogue tensors, timed
    under the same protocol (per-launch CUDA events on one stream, the L2
    flushed before each launch when the inputs are smaller than twice it).
    Rank 0 only."""
    import torch

    from dense_gemm_elementwise_gb300 import workloads as W
    rank, world, local = dist_setup(args.gpus)
    if rank != 0:
        return
    torch.cuda.set_device(local)
    dev_ = torch.device("cuda", local)
    stream = torch.cuda.Stream(device=dev_)
    clocks = ClockSampler(local, gpu_pci_bus(local)).start()
    A, Bm, _, _ = W.make_inputs(w)
    Ad, Bd = A.to(dev_), Bm.to(dev_)
    out = torch.empty(w.L, w.M, w.N, dtype=W.TORCH_DTYPE[w.outs[0][1]], device=dev_)
    in_bytes = Ad.numel() * Ad.element_size() + Bd.numel() * Bd.element_size()
    flush = in_bytes < 2 * L2_BYTES
    if flush:
        fbuf = torch.empty(512 << 20, dtype=torch.uint8, device=dev_)
        cbuf = torch.ones(64 << 20, dtype=torch.float32, device=dev_)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            torch.matmul(Ad, Bd, out=out)
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    t0 = time.time()
    with torch.cuda.stream(stream):
        for s_, e_ in evs:
            if flush:
                fbuf.zero_()
                cbuf.sum()
            s_.record(stream)
            torch.matmul(Ad, Bd, out=out)
            e_.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    clk = clocks.window(t0, t1)
    clocks.stop()
    ms = sum(s_.elapsed_time(e_) for s_, e_ in evs) / args.steps
    gemm_flops = 2.0 * w.L * w.M * w.N * w.K
    line = {"impl": "vendor", "metric": "vendor GEMM TFLOP/s (torch.matmul: A @ B only)",
            "value": gemm_flops / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "dtype": w.ab, "data": "synthetic",
            "config": workload_config(w, 1), "l2": l2_note(flush, in_bytes), "clocks": clk}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------ our arm ---

def parse_opts(B, text):
    if not text:
        return None
    return B.ge_options(**{k: int(v) for k, v in (kv.split("=") for kv in text.split(","))})


def l2_note(flush, in_bytes):
    if flush:
        return ("flushed before every timed step: 512 MiB write, then 256 MiB read "
                "(inputs %d MiB)" % (in_bytes >> 20))
    return "no flush: inputs (%d MiB) larger than twice the L2" % (in_bytes >> 20)


class Measured:
    """One workload planned, resident in device memory and timed under the
    benchmark's protocol: W warm-up launches, then K timed ones, each between
    CUDA events on the launch stream, the L2 flushed before every timed
    launch when the inputs are smaller than twice the L2."""

    def __init__(self, w, dev_, stream, world, opts, host_inputs=None):
        import torch

        from dense_gemm_elementwise_gb300 import binding as B
        from dense_gemm_elementwise_gb300 import workloads as W
        self.w, self.dev, self.stream, self.world, self.opts = w, dev_, stream, world, opts
        self.B = B
        self.inputs = host_inputs if host_inputs is not None else W.make_inputs(w)
        A, Bm, aux, self.scalars = self.inputs
        self.Ad, self.Bd = A.to(dev_), Bm.to(dev_)
        self.auxd = [a.to(dev_) for a in aux]
        self.outs = [torch.empty(w.L, w.M, w.N, dtype=W.TORCH_DTYPE[dt], device=dev_)
                     for _, dt in w.outs]
        self.dtypes = B.make_dtypes(w.ab, [s[2] for s in w.aux], len(w.scalars),
                                    [dt for _, dt in w.outs])
        self.plan = B.gemm_epi_plan_create(w.L, w.M, w.N, w.K, self.dtypes, B.make_dag(w.dag),
                                           opts)
        self.info = B.gemm_epi_plan_info(self.plan)
        self.flops = w.flops()
        self.in_bytes = w.alg_bytes() - sum(w.L * w.M * w.N * W.ESIZE[dt] for _, dt in w.outs)
        # inputs smaller than twice the L2: flush it before every timed step by
        # writing 512 MiB and reading 256 MiB (the read pays the write-back of
        # the dirty lines before the step starts)
        self.flush_l2 = self.in_bytes < 2 * L2_BYTES
        if self.flush_l2:
            self.fbuf = torch.empty(512 << 20, dtype=torch.uint8, device=dev_)
            self.cbuf = torch.ones(64 << 20, dtype=torch.float32, device=dev_)

    def timed(self, fn, steps):
        """CUDA events around every step on the launch stream; returns ms/step."""
        import torch
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        torch.cuda.synchronize()
        barrier(self.world)
        torch.cuda.synchronize()
        with torch.cuda.stream(self.stream):
            for s, e in evs:
                if self.flush_l2:
                    self.fbuf.zero_()
                    self.cbuf.sum()
                s.record(self.stream)
                fn()
                e.record(self.stream)
        torch.cuda.synchronize()
        barrier(self.world)
        torch.cuda.synchronize()
        return sum(s.elapsed_time(e) for s, e in evs) / steps

    def fused(self):
        self.B.gemm_epi_run(self.plan, self.Ad, self.Bd, self.auxd, self.scalars, self.outs,
                            stream=self.stream)

    def run_fused(self, steps, warmup):
        import torch
        for _ in range(warmup):
            self.fused()
        torch.cuda.synchronize()
        if self.B.gemm_epi_last_error(self.plan) != self.B.GE_OK:
            raise RuntimeError("device-side timeout during warm-up (%s)" % self.w.name)
        ms = self.timed(self.fused, steps)
        if self.B.gemm_epi_last_error(self.plan) != self.B.GE_OK:
            raise RuntimeError("device-side timeout during the timed region (%s)" % self.w.name)
        return ms

    def run_unfused(self, steps, warmup, ms_fused):
        import torch
        B, w = self.B, self.w
        ws = torch.empty(B.gemm_epi_unfused_workspace_bytes(self.plan) // 4,
                         dtype=torch.float32, device=self.dev)

        def unf():
            B.gemm_epi_run_unfused(self.plan, self.Ad, self.Bd, self.auxd, self.scalars,
                                   self.outs, ws, stream=self.stream)

        for _ in range(warmup):
            unf()
        ums = self.timed(unf, steps)
        del ws
        return {"ms_per_step": ums, "value": self.flops / (ums * 1e-3) / 1e12,
                "fused_speedup": ums / ms_fused, "launches_per_step": 2,
                "extra_bytes_per_step": 8 * w.L * w.M * w.N}

    def run_stream(self, replays):
        """Back-to-back throughput of independent launches whose inputs are
        not in the L2: R replicas of the inputs and outputs (R * inputs >=
        twice the L2), one launch per replica captured in a CUDA graph (the
        tensor maps of each replica are encoded while capturing), the graph
        replayed `replays` times between two CUDA events on the launch
        stream.  Every launch reads its inputs from DRAM; no event or host
        call sits between two launches."""
        import torch
        B, w = self.B, self.w
        reps = max(2, -(-2 * L2_BYTES // max(self.in_bytes, 1)))
        if reps > 4096:
            return None
        A, Bm, aux, _ = self.inputs
        src = [self.Ad, self.Bd] + self.auxd
        copies = [[t.clone() for t in src] for _ in range(reps)]
        outs = [[torch.empty_like(o) for o in self.outs] for _ in range(reps)]
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=self.stream):
            for c, o in zip(copies, outs):
                B.gemm_epi_run(self.plan, c[0], c[1], c[2:], self.scalars, o, stream=self.stream)
        graph.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        barrier(self.world)
        with torch.cuda.stream(self.stream):
            e0.record(self.stream)
            for _ in range(replays):
                graph.replay()
            e1.record(self.stream)
        torch.cuda.synchronize()
        barrier(self.world)
        if B.gemm_epi_last_error(self.plan) != B.GE_OK:
            raise RuntimeError("device-side timeout in the back-to-back launches (%s)" % w.name)
        launches = reps * replays
        ms = e0.elapsed_time(e1) / launches
        del graph, copies, outs
        torch.cuda.empty_cache()
        roof = roofline(self.flops, w.alg_bytes(), ms, None)
        return {"us_per_launch": ms * 1e3, "value": self.flops / (ms * 1e-3) / 1e12,
                "unit": "TFLOP/s", "launches": launches, "replicas": reps,
                "roofline": {k: roof[k] for k in ("bound", "achieved", "peak", "unit", "frac")},
                "how": "%d input replicas (%d MiB in all, more than twice the L2) launched back "
                       "to back from a CUDA graph, %d replays between two CUDA events"
                       % (reps, (reps * self.in_bytes) >> 20, replays)}

    def close(self):
        if self.plan is not None:
            self.B.gemm_epi_plan_destroy(self.plan)
            self.plan = None


def config_entry(m, ms, unfused, stream=None):
    """One workload's figures for the bench line's ``configs`` object:
    per-launch CUDA-event timing (the headline protocol) and, for workloads
    whose inputs fit in the L2, the back-to-back stream figure."""
    w = m.w
    roof = roofline(m.flops, w.alg_bytes(), ms, ncu_traffic(w.name, m.info))
    return {"workload": w.name, "L": w.L, "M": w.M, "N": w.N, "K": w.K, "ab_dtype": w.ab,
            "outs": [n + ":" + dt for n, dt in w.outs],
            "ms_per_step": ms, "value": m.flops / (ms * 1e-3) / 1e12, "unit": "TFLOP/s",
            "roofline": {k: roof[k] for k in ("bound", "achieved", "peak", "unit", "frac",
                                              "traffic", "tensor_frac", "hbm_frac")},
            "unfused": unfused, "back_to_back": stream, "l2": l2_note(m.flush_l2, m.in_bytes),
            "plan": m.info}


def run_ours(args, w):
    import torch

    from dense_gemm_elementwise_gb300 import binding as B
    from dense_gemm_elementwise_gb300 import workloads as W

    rank, world, local = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    dev_ = torch.device("cuda", local)
    stream = torch.cuda.Stream(device=dev_)
    clocks = ClockSampler(local, gpu_pci_bus(local)).start()
    opts = parse_opts(B, args.opt)
    m = Measured(w, dev_, stream, world, opts)
    inputs = m.inputs
    A, Bm, aux, scalars = inputs
    info, flops, dtypes = m.info, m.flops, m.dtypes

    for _ in range(args.warmup):
        m.fused()
    torch.cuda.synchronize()
    if B.gemm_epi_last_error(m.plan) != B.GE_OK:
        raise RuntimeError("device-side timeout during warm-up")
    t_begin = time.time()
    ms = m.timed(m.fused, args.steps)
    t_end = time.time()
    # the sampler stops once the first sample after the region is in, so its
    # polling overlaps none of the other legs (the CPU oracle uses every core)
    time.sleep(0.05)
    clocks.stop()
    clk = clocks.window(t_begin, t_end)
    ms_max = max_over_ranks(ms, world)
    if B.gemm_epi_last_error(m.plan) != B.GE_OK:
        raise RuntimeError("device-side timeout during the timed region")
    value = world * flops / (ms_max * 1e-3) / 1e12

    roof = roofline(flops, w.alg_bytes(), ms, ncu_traffic(w.name, info))

    unfused = None
    if not args.no_unfused:
        unfused = m.run_unfused(max(3, args.steps // 4), max(3, args.warmup // 4), ms)
    back_to_back = m.run_stream(max(3, args.steps // 4)) if m.flush_l2 else None

    e2e = None
    if not args.no_e2e:
        # End to end through the C ABI with host buffers: every step copies its
        # inputs from pinned host memory and its outputs back.  Steps are
        # pipelined over three streams (H2D of step i+1, compute of step i,
        # D2H of step i-1) with two device buffer sets, ordered by events.
        Ad, Bd, auxd, outs = m.Ad, m.Bd, m.auxd, m.outs
        hA, hB = A.pin_memory(), Bm.pin_memory()
        haux = [a.pin_memory() for a in aux]
        houts = [[torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in outs] for _ in range(2)]
        h2d = sum(t.numel() * t.element_size() for t in [hA, hB] + haux)
        d2h = sum(t.numel() * t.element_size() for t in houts[0])
        dev = [(Ad, Bd, auxd, outs),
               (torch.empty_like(Ad), torch.empty_like(Bd), [torch.empty_like(a) for a in auxd],
                [torch.empty_like(o) for o in outs])]
        plans = [m.plan, B.gemm_epi_plan_create(w.L, w.M, w.N, w.K, dtypes, B.make_dag(w.dag),
                                                opts)]
        s_in, s_out = torch.cuda.Stream(device=dev_), torch.cuda.Stream(device=dev_)
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_done = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]

        def pipeline(n):
            for i in range(n):
                b = i % 2
                dA_, dB_, daux_, douts_ = dev[b]
                if i >= 2:
                    s_in.wait_event(ev_done[b])  # step i-2 finished reading buffer b
                with torch.cuda.stream(s_in):
                    dA_.copy_(hA, non_blocking=True)
                    dB_.copy_(hB, non_blocking=True)
                    for d, h in zip(daux_, haux):
                        d.copy_(h, non_blocking=True)
                    ev_in[b].record(s_in)
                stream.wait_event(ev_in[b])
                if i >= 2:
                    stream.wait_event(ev_out[b])  # outputs of step i-2 copied out
                B.gemm_epi_run(plans[b], dA_, dB_, daux_, scalars, douts_, stream=stream)
                ev_done[b].record(stream)
                s_out.wait_event(ev_done[b])
                with torch.cuda.stream(s_out):
                    for h, d in zip(houts[b], douts_):
                        h.copy_(d, non_blocking=True)
                    ev_out[b].record(s_out)

        pipeline(4)
        torch.cuda.synchronize()
        e_steps = max(30, args.steps // 10)
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        t0.record(s_in)
        pipeline(e_steps)
        s_in.wait_stream(s_out)
        s_in.wait_stream(stream)
        t1.record(s_in)
        torch.cuda.synchronize()
        barrier(world)
        ems = max_over_ranks(t0.elapsed_time(t1) / e_steps, world)
        B.gemm_epi_plan_destroy(plans[1])
        del dev, houts
        e2e = {"value": world * flops / (ems * 1e-3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e_steps,
               "ms_per_step": ems, "pipelined_streams": 3,
               "host_memory": host_numa_note(local, [hA, hB] + haux)}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, inputs)

    # every workload of the task's table under the same protocol (the headline
    # figures above are its entry), with the fused kernel's roofline and the
    # unfused comparison; default-sized workloads only (not under --mnk)
    configs = None
    if not args.no_configs and not args.mnk:
        configs = {}
        for cw in W.WORKLOADS:
            if cw.name == w.name:
                configs[cw.name] = config_entry(m, ms, unfused, back_to_back)
                continue
            cm = Measured(cw, dev_, stream, world, None)
            try:
                cms = cm.run_fused(args.steps, args.warmup)
                cun = None if args.no_unfused else cm.run_unfused(
                    max(3, args.steps // 4), max(3, args.warmup // 4), cms)
                cst = cm.run_stream(max(3, args.steps // 4)) if cm.flush_l2 else None
                configs[cw.name] = config_entry(cm, cms, cun, cst)
            finally:
                cm.close()
            del cm
            torch.cuda.empty_cache()

    m.close()
    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": w.ab, "data": "synthetic",
        "config": workload_config(w, world),
        "l2": l2_note(m.flush_l2, m.in_bytes), "plan": info, "options": args.opt or "auto",
        "pct_of_peak": 100.0 * roof["tensor_frac"],
        "roofline": roof, "gpu_launches": args.steps, "clocks": clk,
        "unfused": unfused, "back_to_back": back_to_back, "e2e": e2e, "cpu_baseline": cpu,
        "configs": configs,
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------- grouped GEMM ---

GROUPED_METRIC = "grouped GEMM+epilogue TFLOP/s, all problems in one launch (1 GPU)"


def grouped_oracle_time(w, inputs):
    import oracle
    from dense_gemm_elementwise_gb300 import workloads as W
    As, Bs, auxs, scalars = inputs
    t0 = time.perf_counter()
    oracle.grouped_gemm_epilogue(
        w.problems, w.ab, [W.to_codes(a) for a in As], [W.to_codes(b) for b in Bs],
        [[W.to_codes(x) for x in per] for per in auxs], [s[2] for s in w.aux], scalars, w.dag,
        [dt for _, dt in w.outs], threads=oracle.threads_default())
    return time.perf_counter() - t0


def run_grouped_reference(args, w):
    """The oracle, as it stands, on the whole grouped workload per step."""
    import oracle
    from dense_gemm_elementwise_gb300 import workloads as W
    rank, world, _ = dist_setup(args.gpus)
    if rank != 0:
        return
    inputs = W.make_grouped_inputs(w)
    for _ in range(args.warmup):
        grouped_oracle_time(w, inputs)
    total = sum(grouped_oracle_time(w, inputs) for _ in range(args.steps))
    ms = total / args.steps * 1e3
    value = w.flops() / (ms * 1e-3) / 1e12
    threads = oracle.threads_default()
    sample = "all %d problems per step, fp64" % len(w.problems)
    print(json.dumps({
        "impl": "reference", "metric": GROUPED_METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": grouped_config(w, args.gpus),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0}}), flush=True)


def run_grouped(args, w):
    """One grouped launch per step over every problem of the workload, against
    one gemm_epi_run launch per problem on the same data."""
    import torch

    from dense_gemm_elementwise_gb300 import binding as B
    from dense_gemm_elementwise_gb300 import workloads as W

    rank, world, local = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    dev_ = torch.device("cuda", local)
    stream = torch.cuda.Stream(device=dev_)
    clocks = ClockSampler(local, gpu_pci_bus(local)).start()
    inputs = W.make_grouped_inputs(w)
    As, Bs, auxs, scalars = inputs
    Ad = [a.to(dev_) for a in As]
    Bd = [b.to(dev_) for b in Bs]
    auxd = [[x.to(dev_) for x in per] for per in auxs]
    outs = [[torch.empty(m, n, dtype=W.TORCH_DTYPE[dt], device=dev_) for _, dt in w.outs]
            for m, n, k in w.problems]
    dtypes = B.make_dtypes(w.ab, [s[2] for s in w.aux], len(w.scalars), [dt for _, dt in w.outs])
    dag = B.make_dag(w.dag)
    opts = None
    if args.opt:
        opts = B.ge_options(**{k: int(v) for k, v in (kv.split("=") for kv in args.opt.split(","))})
    plan = B.gemm_epi_grouped_plan_create(w.problems, dtypes, dag, opts)
    info = B.gemm_epi_plan_info(plan)
    flops = w.flops()
    # the inputs fit in L2: flush it before every timed step by writing 512 MiB
    # and then reading 256 MiB, so that the write-back of the dirty lines the
    # write leaves behind is paid before the step, not inside it
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev_)
    clean = torch.ones(64 << 20, dtype=torch.float32, device=dev_)

    def flush_l2():
        flush.zero_()
        clean.sum()

    def timed(fn, steps):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        torch.cuda.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            for s, e in evs:
                flush_l2()
                s.record(stream)
                fn()
                e.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        return sum(s.elapsed_time(e) for s, e in evs) / steps

    # arguments marshalled once: a step's host work is one C call, far shorter
    # than the L2 flush queued before it, so the GPU never waits on the host
    grouped_call = B.prepare_grouped_run(plan, Ad, Bd, auxd, scalars, outs, stream=stream)

    def grouped():
        st = grouped_call()
        if st != B.GE_OK:
            raise B.GemmEpiError(st, "gemm_epi_grouped_run")

    for _ in range(args.warmup):
        grouped()
    torch.cuda.synchronize()
    if B.gemm_epi_last_error(plan) != B.GE_OK:
        raise RuntimeError("device-side timeout during warm-up")
    t_begin = time.time()
    ms = timed(grouped, args.steps)
    t_end = time.time()
    time.sleep(0.1)
    clocks.stop()
    clk = clocks.window(t_begin, t_end)
    ms_max = max_over_ranks(ms, world)
    if B.gemm_epi_last_error(plan) != B.GE_OK:
        raise RuntimeError("device-side timeout during the timed region")
    value = world * flops / (ms_max * 1e-3) / 1e12

    # one launch per problem (a plan each), same buffers: issued eagerly (the
    # host's launch rate included) and replayed from a CUDA graph (device time)
    plans = [B.gemm_epi_plan_create(1, m, n, k, dtypes, dag, opts) for m, n, k in w.problems]
    calls = [B.prepare_run(pl, Ad[g], Bd[g], auxd[g], scalars, outs[g], stream=stream)
             for g, pl in enumerate(plans)]

    def per_problem():
        for c in calls:
            st = c()
            if st != B.GE_OK:
                raise B.GemmEpiError(st, "gemm_epi_run")

    for _ in range(max(3, args.warmup // 4)):
        per_problem()
    pms = timed(per_problem, max(3, args.steps // 4))
    graph = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.graph(graph, stream=stream):
        per_problem()
    graph.replay()
    torch.cuda.synchronize()
    gms = timed(graph.replay, max(3, args.steps // 4))
    del graph
    torch.cuda.synchronize()
    if B.gemm_epi_last_error(None) != B.GE_OK:
        raise RuntimeError("device-side timeout in the per-problem launches")
    for pl in plans:
        B.gemm_epi_plan_destroy(pl)
    separate = {"ms_per_step": pms, "value": flops / (pms * 1e-3) / 1e12,
                "grouped_speedup": pms / ms, "launches_per_step": len(w.problems),
                "graph_ms_per_step": gms, "graph_value": flops / (gms * 1e-3) / 1e12,
                "grouped_speedup_vs_graph": gms / ms}

    b2b = grouped_back_to_back(w, plan_args=(dtypes, dag, opts), dev_tensors=(Ad, Bd, auxd, outs),
                               scalars=scalars, stream=stream, world=world,
                               replays=max(3, args.steps // 4))

    e2e = None
    if not args.no_e2e:
        hA = [a.pin_memory() for a in As]
        hB = [b.pin_memory() for b in Bs]
        haux = [[x.pin_memory() for x in per] for per in auxs]
        houts = [[torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in per] for per in outs]
        h2d = sum(t.numel() * t.element_size() for t in hA + hB + [x for p in haux for x in p])
        d2h = sum(t.numel() * t.element_size() for p in houts for t in p)

        def e2e_step():
            for d, h in zip(Ad + Bd + [x for p in auxd for x in p],
                            hA + hB + [x for p in haux for x in p]):
                d.copy_(h, non_blocking=True)
            grouped()
            for pd, ph in zip(outs, houts):
                for d, h in zip(pd, ph):
                    h.copy_(d, non_blocking=True)

        with torch.cuda.stream(stream):
            for _ in range(3):
                e2e_step()
        ems = max_over_ranks(timed(e2e_step, max(3, args.steps // 10)), world)
        e2e = {"value": world * flops / (ems * 1e-3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ems}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        t = grouped_oracle_time(w, inputs)
        cpu = {"value": flops / t / 1e12, "unit": "TFLOP/s", "cores": oracle.threads_default(),
               "kind": "oracle", "sample": "all %d problems, fp64, %.2f s wall"
                                           % (len(w.problems), t)}

    B.gemm_epi_plan_destroy(plan)
    if rank != 0:
        return
    roof = roofline(flops, w.alg_bytes(), ms, None)
    print(json.dumps({
        "metric": GROUPED_METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": w.ab, "data": "synthetic",
        "config": grouped_config(w, world),
        "l2": "flushed before every timed step: 512 MiB write, then 256 MiB read",
        "plan": info, "options": args.opt or "auto",
        "roofline": roof,
        "gpu_launches": args.steps, "clocks": clk, "one_launch_per_problem": separate,
        "back_to_back": b2b, "e2e": e2e, "cpu_baseline": cpu}), flush=True)


def grouped_back_to_back(w, plan_args, dev_tensors, scalars, stream, world, replays):
    """Back-to-back throughput of grouped launches whose inputs are not in the
    L2: R replicas of every problem's inputs and outputs (R * inputs >= twice
    the L2), a grouped plan per replica whose problem table its first run
    uploads, then `replays` rounds of one launch per replica issued between
    two CUDA events (tables reused: no copy between launches; one host call
    per launch, several times shorter than the launch itself)."""
    import torch

    from dense_gemm_elementwise_gb300 import binding as B
    dtypes, dag, opts = plan_args
    Ad, Bd, auxd, outs = dev_tensors
    in_bytes = sum(t.numel() * t.element_size() for t in Ad + Bd + [x for p in auxd for x in p])
    reps = max(2, -(-2 * L2_BYTES // max(in_bytes, 1)))
    if reps > 64:
        return None
    plans, calls, keep = [], [], []
    try:
        for _ in range(reps):
            a_ = [t.clone() for t in Ad]
            b_ = [t.clone() for t in Bd]
            x_ = [[t.clone() for t in p] for p in auxd]
            o_ = [[torch.empty_like(t) for t in p] for p in outs]
            keep.append((a_, b_, x_, o_))
            plans.append(B.gemm_epi_grouped_plan_create(w.problems, dtypes, dag, opts))
            calls.append(B.prepare_grouped_run(plans[-1], a_, b_, x_, scalars, o_, stream=stream))

        def run_all():
            for c in calls:
                st = c()
                if st != B.GE_OK:
                    raise B.GemmEpiError(st, "gemm_epi_grouped_run")

        with torch.cuda.stream(stream):
            run_all()  # uploads every replica's problem table
            run_all()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(replays):
                run_all()
            e1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        if B.gemm_epi_last_error(None) != B.GE_OK:
            raise RuntimeError("device-side timeout in the back-to-back grouped launches")
        launches = reps * replays
        ms = e0.elapsed_time(e1) / launches
    finally:
        for pl in plans:
            B.gemm_epi_plan_destroy(pl)
        del keep
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    flops = w.flops()
    roof = roofline(flops, w.alg_bytes(), ms, None)
    return {"us_per_launch": ms * 1e3, "value": flops / (ms * 1e-3) / 1e12, "unit": "TFLOP/s",
            "launches": launches, "replicas": reps,
            "roofline": {k: roof[k] for k in ("bound", "achieved", "peak", "unit", "frac")},
            "how": "%d input replicas (%d MiB in all, more than twice the L2), a grouped plan "
                   "each, launched back to back on one stream, %d rounds between two CUDA "
                   "events" % (reps, (reps * in_bytes) >> 20, replays)}


def main():
    args = parse()
    from dense_gemm_elementwise_gb300 import workloads as W
    if args.workload in W.GROUPED_BY_NAME:
        w = W.GROUPED_BY_NAME[args.workload]
        if args.impl == "reference":
            run_grouped_reference(args, w)
        elif args.impl == "vendor":
            raise SystemExit("--impl vendor times batched workloads only")
        else:
            from dense_gemm_elementwise_gb300 import build as gbuild
            gbuild.build()
            run_grouped(args, w)
        return
    table = dict(W.BY_NAME)
    table.update({x.name: x for x in W.page_examples()})
    w = table[args.workload]
    if args.mnk:
        import dataclasses
        m, n, k = (int(x) for x in args.mnk.split(","))
        w = dataclasses.replace(w, M=m, N=n, K=k, name="%s@%dx%dx%d" % (w.name, m, n, k))
    if args.impl == "reference":
        run_reference(args, w)
    elif args.impl == "vendor":
        run_vendor(args, w)
    else:
        from dense_gemm_elementwise_gb300 import build as gbuild
        gbuild.build()
        run_ours(args, w)


if __name__ == "__main__":
    if len(sys.argv) == 4 and sys.argv[1] == "--nvml-sampler":
        nvml_sampler_main(sys.argv[2], int(sys.argv[3]))
    else:
        main()
