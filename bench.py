"""Benchmark of the GEMM library: one JSON line on rank 0.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one GEMM call D = alpha*op(A)*op(B) + beta*C on the workload's
seeded synthetic inputs (default: BF16 8192^3, A row-major, B column-major,
D FP32), inputs resident in HBM.  ``value`` is whole-job throughput in
TFLOPS (2MNK / time, "GEMM on NVIDIA GPUs", section 1); ``e2e`` is the same
metric with the host->device copy of A and B (pinned memory) and the
device->host copy of D inside every step.  Under torchrun every rank runs an
independent replica on its own GPU (the path needs no exchange): the time is
the maximum over ranks and ``value`` counts the work of all ranks.

``--impl reference`` times the CPU oracle (the slow plain reference) on a
bounded sample of the same workload on this machine's host cores.
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
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GEMM TFLOPS (2MNK/s) and % of GB300 BF16/FP32 peak at 8192^3, 1 GPU"
UNIT = "TFLOPS"
L2_BYTES = 129 * 1000 * 1000  # GB300 L2 (~129 MB)
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# torch.cuda._sleep spins for a number of SM clock cycles; this converts
# seconds at the maximum SM clock (a longer delay at a lower clock is harmless).
SLEEP_CYCLES_PER_S = 2.07e9

KERNEL_SOURCES = {
    "gemm_bf16_tc": "dense_gemm_08_gb300/csrc/gemm_tc.cu",
    "gemm_f16_tc": "dense_gemm_08_gb300/csrc/gemm_tc.cu",
    "sgemm_simt": "dense_gemm_08_gb300/csrc/sgemm_simt.cu",
    "sgemm_cluster": "dense_gemm_08_gb300/csrc/sgemm_cluster.cu",
    "skinny": "dense_gemm_08_gb300/csrc/skinny.cu",
}


# ------------------------------------------------------------- pure helpers
def algorithmic_bytes(M, N, K, in_bytes, beta):
    """Bytes the method must move: A and B once, D once, C once if beta != 0
    ("GEMM on NVIDIA GPUs", section 2, "GEMM arithmetic intensity")."""
    b = in_bytes * (M * K + K * N) + 4 * M * N
    if beta != 0:
        b += 4 * M * N
    return b


def roofline_tflops(flops, nbytes, peak_tflops, hbm_gbs):
    """min(peak, I * BW) in TFLOP/s, I = flops / bytes."""
    intensity = flops / nbytes
    return min(peak_tflops, intensity * hbm_gbs * 1e9 / 1e12)


def hbm_bound_roof(roof, alg_bytes, seconds, hbm_gbs, peak_src, roof_tflops):
    """The roofline object of a launch: when I x BW_HBM is below the compute
    peak, the shape is HBM-bound and the fraction is taken against the HBM
    bandwidth (algorithmic bytes / time); otherwise `roof` (compute) as is."""
    if roof_tflops >= roof["peak"]:
        return roof
    achieved = alg_bytes / seconds / 1e9
    return {"bound": "hbm", "achieved": achieved, "peak": hbm_gbs, "unit": "GB/s",
            "frac": achieved / hbm_gbs, "peak_source": f"{peak_src} HBM copy bandwidth",
            "compute": {k: roof[k] for k in ("bound", "achieved", "peak", "unit", "frac")}}


def fp32_core_peak_tflops(sms, mhz):
    """FP32 CUDA-core peak: SMs x 128 FP32 lanes x 2 FLOP (FMA) x clock."""
    return sms * 128 * 2 * mhz * 1e6 / 1e12


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def source_digest(rel_path):
    with open(os.path.join(ROOT, rel_path), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def rotation_copies(working_set, l2_bytes):
    """How many copies of a step's working set the timed steps rotate over so
    that each step reads operands not in L2: 1 if the set alone is at least
    twice L2, else enough copies to exceed twice L2."""
    if working_set >= 2 * l2_bytes:
        return 1
    return -(-2 * l2_bytes // max(working_set, 1))


def committed_traffic(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary of this kernel and
    workload, or None if there is none or the kernel source changed since."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}_traffic.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    m_bytes = re.search(r"^traffic_bytes_per_launch:\s*([0-9.eE+]+)", text, re.M)
    m_src = re.search(r"^source_sha256_16:\s*([0-9a-f]+)", text, re.M)
    if not m_bytes or not m_src:
        return None
    if m_src.group(1) != source_digest(KERNEL_SOURCES[kernel]):
        return None
    return float(m_bytes.group(1))


def clock_summary(rows):
    """rows: parsed nvidia-smi CSV samples -> clocks object of the JSON line."""
    if not rows:
        return None
    sm = [r["sm"] for r in rows if r["sm"] is not None]
    max_mhz = max((r["max"] for r in rows if r["max"] is not None), default=None)
    loaded = [r["sm"] for r in rows if r["sm"] is not None and r["power"] is not None
              and r["power"] > 0.3 * max(x["power"] for x in rows if x["power"] is not None)]
    reasons = set()
    for r in rows:
        reasons.update(r["reasons"])
    return {"sm_mhz": statistics.median(loaded or sm) if sm else None, "sm_max_mhz": max_mhz,
            "reasons": sorted(reasons), "samples": len(rows)}


def window(rows, t0, t1):
    """The samples taken between wall-clock times t0 and t1 (seconds)."""
    return [r for r in rows if r.get("t") is not None and t0 <= r["t"] <= t1]


def nvml_bus_id(device_index):
    """PCI bus id "dddddddd:bb:dd.0" of CUDA device `device_index`, the key
    NVML and nvidia-smi share whatever CUDA_VISIBLE_DEVICES says; None if
    torch does not expose it."""
    import torch
    prop = torch.cuda.get_device_properties(device_index)
    bus = getattr(prop, "pci_bus_id", None)
    dev = getattr(prop, "pci_device_id", None)
    dom = getattr(prop, "pci_domain_id", None)
    if bus is None or dev is None or dom is None:
        return None
    return f"{dom:08x}:{bus:02x}:{dev:02x}.0"


class NvmlSampler:
    """SM clock and clock-event reasons (and, every 8th sample, power) read
    from the driver's NVML library (by ctypes) in a thread, as fast as NVML
    answers (at most every 0.1 ms), so that a timed region of a few
    milliseconds still has samples; rows as ClockSampler's.
    Reads only: NVML query calls, no setting is changed."""
    REASON_BITS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                   0x40: "hw_thermal_slowdown"}
    NVML_CLOCK_SM = 1

    def __init__(self, bus_id, index, period_s=0.0001):
        self.bus_id, self.index, self.period = bus_id, index, period_s
        self.rows, self.ok, self._stop = [], False, None

    def _open(self):
        import ctypes
        nv = ctypes.CDLL("libnvidia-ml.so.1")
        if nv.nvmlInit_v2() != 0:
            return None
        h = ctypes.c_void_p()
        r = 1
        if self.bus_id:
            r = nv.nvmlDeviceGetHandleByPciBusId_v2(self.bus_id.encode(), ctypes.byref(h))
        if r != 0:
            r = nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.index), ctypes.byref(h))
        if r != 0:
            return None
        reasons = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(nv, "nvmlDeviceGetCurrentClocksThrottleReasons")
        return nv, h, reasons

    def _run(self, nv, h, reasons_fn):
        import ctypes
        clk, mx, pw, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        nv.nvmlDeviceGetMaxClockInfo(h, self.NVML_CLOCK_SM, ctypes.byref(mx))
        n = 0
        while not self._stop.is_set():
            t = time.time()
            row = {"t": t, "sm": None, "max": float(mx.value) or None, "power": None,
                   "reasons": []}
            if nv.nvmlDeviceGetClockInfo(h, self.NVML_CLOCK_SM, ctypes.byref(clk)) == 0:
                row["sm"] = float(clk.value)
            if reasons_fn(h, ctypes.byref(rs)) == 0:
                row["reasons"] = [n for b, n in self.REASON_BITS.items() if rs.value & b]
            # the power reading is a running average: every 8th sample is enough
            if n % 8 == 0 and nv.nvmlDeviceGetPowerUsage(h, ctypes.byref(pw)) == 0:
                row["power"] = pw.value / 1000.0
            n += 1
            self.rows.append(row)
            self._stop.wait(self.period)

    def __enter__(self):
        import threading
        try:
            opened = self._open()
        except (OSError, AttributeError):
            opened = None
        if opened is None:
            return self
        self.ok = True
        # switch between Python threads every 0.1 ms while sampling
        self._switch = sys.getswitchinterval()
        sys.setswitchinterval(1e-4)
        self._stop = threading.Event()
        self._thread = threading.Thread(target=self._run, args=opened, daemon=True)
        self._thread.start()
        time.sleep(0.05)
        return self

    def __exit__(self, *exc):
        if self.ok:
            time.sleep(0.02)
            self._stop.set()
            self._thread.join(timeout=5)
            sys.setswitchinterval(self._switch)
        return False


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 50 ms while running."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, index):
        self.index = index  # nvidia-smi --id: an index or a PCI bus id
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.rows = []
        if self.proc is None:
            return False
        time.sleep(0.3)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue

            def num(x):
                try:
                    return float(x)
                except ValueError:
                    return None
            reasons = [n for n, v in zip(self.NAMES, parts[5:9]) if v.lower() == "active"]
            try:
                import datetime
                t = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                t = None
            self.rows.append({"t": t, "sm": num(parts[1]), "max": num(parts[2]),
                              "power": num(parts[3]), "reasons": reasons})
        return False


# ----------------------------------------------------------------- our arm
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(value, ws, device):
    if ws == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws, device=None):
    if ws > 1:
        import torch.distributed as dist
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def run_cpu_baseline(w, inp, target_s=12.0, max_rows=None, threads=0):
    """Time the oracle on whole rows of D (bounded sample) with `threads`
    host threads (0: one per core).  Returns the JSON object."""
    import numpy as np
    import oracle

    def bits(t):
        if t is None:
            return None
        t = t.contiguous()
        if t.dtype.is_floating_point and t.element_size() == 2:
            import torch
            view = np.float16 if t.dtype == torch.float16 else np.uint16
            return t.view(torch.int16).numpy().view(view).reshape(-1)
        return t.numpy().reshape(-1)

    A, B, C = bits(inp["A"]), bits(inp["B"]), bits(inp["C"])
    threads = threads if threads > 0 else oracle.default_threads()

    def rows_run(r0, nrows):
        I = np.repeat(np.arange(r0, r0 + nrows, dtype=np.int64), w.N)
        J = np.tile(np.arange(w.N, dtype=np.int64), nrows)
        t0 = time.perf_counter()
        D, S = oracle.gemm_points(w.M, w.N, w.K, w.alpha, A, inp["lda"], w.order_a, B,
                                  inp["ldb"], w.order_b, w.beta, C, inp["ldc"], w.order_cd, I, J,
                                  nthreads=threads)
        return time.perf_counter() - t0, D, S

    # calibrate on one row per thread, then size the sample to ~target_s
    cal_rows = min(w.M, max(1, threads))
    dt, _, _ = rows_run(0, cal_rows)
    per_row = dt / cal_rows
    rows = int(max(1, min(w.M, target_s / max(per_row, 1e-9))))
    if max_rows is not None:
        rows = min(rows, max_rows)
    dt, D, S = rows_run(0, rows)
    flops = 2.0 * rows * w.N * w.K
    return {"value": flops / dt / 1e12, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"rows 0..{rows - 1} of D ({rows} x {w.N} entries, K = {w.K}), "
                      f"{dt:.2f} s", "seconds": dt, "_rows": rows, "_D": D, "_S": S}


def resolve_workload(args):
    from dense_gemm_08_gb300.inputs import WORKLOADS
    w = WORKLOADS[args.workload]
    if args.shape:
        M, N, K = (int(x) for x in args.shape.split(","))
        w = w.with_(name=f"{w.name}@{M}x{N}x{K}", M=M, N=N, K=K)
    return w


def region_clocks(nvml_rows, smi_rows, t0, t1):
    """The clocks object of one timed region [t0, t1] (wall-clock seconds):
    the NVML samples taken inside it (about one per millisecond), the
    nvidia-smi samples inside it (50 ms apart: often none for a short region)
    and the nvidia-smi summary of the whole run around it."""
    inside = window(nvml_rows, t0, t1)
    smi_inside = window(smi_rows, t0, t1)
    src = inside or smi_inside
    out = {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": len(src),
           "source": ("NVML, inside the timed region" if inside else
                      "nvidia-smi, 50 ms apart, inside the timed region" if smi_inside else
                      "no sample inside the timed region"),
           "region_s": t1 - t0}
    if src:
        sm = [r["sm"] for r in src if r["sm"] is not None]
        out["sm_mhz"] = statistics.median(sm) if sm else None
        out["sm_mhz_min"] = min(sm) if sm else None
        out["sm_max_mhz"] = max((r["max"] for r in src if r["max"] is not None), default=None)
        out["power_w_max"] = max((r["power"] for r in src if r["power"] is not None), default=None)
    reasons = set()
    for r in inside + smi_inside:
        reasons.update(r["reasons"])
    out["reasons"] = sorted(reasons)
    whole = clock_summary(smi_rows)
    if whole:
        out["nvidia_smi_run"] = whole
        if out["sm_max_mhz"] is None:
            out["sm_max_mhz"] = whole["sm_max_mhz"]
        if out["sm_mhz"] is None:
            out["sm_mhz"] = whole["sm_mhz"]
            out["reasons"] = whole["reasons"]
    return out


def workload_config(w, **extra):
    """The `config` object of a JSON line: the workload, named by what it is."""
    cfg = {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "alpha": w.alpha, "beta": w.beta,
           "in_dtype": w.dtype, "acc_dtype": "f32", "out_dtype": "f32",
           "order_a": "row" if w.order_a == 0 else "col",
           "order_b": "row" if w.order_b == 0 else "col",
           "order_cd": "row" if w.order_cd == 0 else "col",
           "inputs": f"seed 0, {w.dist}" + (f" sigma {w.sigma}" if w.dist == "normal" else "")}
    cfg.update(extra)
    return cfg


class Workbench:
    """Device copies of one workload's inputs (rotated over enough copies that
    every step reads operands not in L2) and the call that runs one step."""

    def __init__(self, lib, w, device, stream):
        import torch
        from dense_gemm_08_gb300.inputs import make_inputs
        self.lib, self.w, self.device, self.stream = lib, w, device, stream
        self.inp = inp = make_inputs(w, seed=0)
        self.fn = {"f32": lib.gemm_f32, "bf16": lib.gemm_bf16_f32acc,
                   "f16": lib.gemm_f16_f32acc}[w.dtype]
        self.in_bytes = 4 if w.dtype == "f32" else 2
        A = inp["A"].to(device)
        B = inp["B"].to(device)
        C = inp["C"].to(device) if inp["C"] is not None else None
        D = torch.empty((w.M, w.N), dtype=torch.float32, device=device)
        ws = A.numel() * A.element_size() + B.numel() * B.element_size() + D.numel() * 4
        if C is not None:
            ws += C.numel() * 4
        self.working_set = ws
        # Inputs larger than L2 between timed steps: a working set under twice
        # L2 is copied until the copies exceed it, and step i uses copy i mod
        # n, so every step reads operands that at least 2 x L2 of other data
        # has passed through L2 since their last use.  All copies hold the
        # same values.
        self.n_rot = rotation_copies(ws, L2_BYTES)
        self.rot = [(A, B, C, D)]
        for _ in range(self.n_rot - 1):
            self.rot.append((A.clone(), B.clone(), C.clone() if C is not None else None,
                             torch.empty_like(D)))
        self.n_step = 0

    def step(self):
        w, inp = self.w, self.inp
        a, b, c, d = self.rot[self.n_step % self.n_rot]
        self.n_step += 1
        self.fn(w.M, w.N, w.K, w.alpha, a, inp["lda"], w.order_a, b, inp["ldb"], w.order_b,
                w.beta, c, inp["ldc"], d, w.N, w.order_cd, self.stream)
        return self.lib.gemm_last_kernel()

    def l2_note(self):
        mib = self.working_set / 2**20
        if self.n_rot == 1:
            return f"inputs larger than L2 (working set {mib:.0f} MiB)"
        return (f"inputs larger than L2: steps rotate over {self.n_rot} copies of the "
                f"{mib:.1f} MiB working set ({self.n_rot * mib:.0f} MiB)")

    def warm(self, n):
        """n untimed steps; returns (last kernel name, host seconds per call)."""
        import torch
        t = time.perf_counter()
        kernel = ""
        for _ in range(n):
            kernel = self.step()
        t_host = (time.perf_counter() - t) / max(n, 1)
        torch.cuda.synchronize(self.device)
        assert self.lib.gemm_last_device_status(self.stream) == self.lib.GEMM_OK
        return kernel, t_host

    def timed(self, steps, t_host, ws=1):
        """Time exactly `steps` back-to-back steps between CUDA events on the
        launching stream, with a barrier and a device synchronize on both
        sides.  Returns (elapsed ms, kernel names, launches, wall t0, wall t1)
        -- t0 and t1 bracket the GPU's execution of the steps (polled event
        completion), for the clock samples."""
        import torch
        barrier(ws, self.device)
        torch.cuda.synchronize(self.device)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        # Keep the GPU busy, before the start event, for twice as long as the
        # host takes to enqueue the timed steps: the steps then run back to
        # back and the events time the GPU, not the host's call overhead
        # (about 15 us per call through the Python binding).
        if hasattr(torch.cuda, "_sleep"):
            torch.cuda._sleep(int(min(2.0, 2.0 * steps * t_host) * SLEEP_CYCLES_PER_S))
        e0.record(self.stream)
        names, launches = set(), 0
        for _ in range(steps):
            names.add(self.step())
            launches += 1
        e1.record(self.stream)
        # Poll the events' completion for the clock samples' window.  The
        # sleeps hand the interpreter to the sampler thread, which would
        # otherwise get it only every switch interval.
        while not e0.query():
            time.sleep(2e-5)
        t0 = time.time()
        while not e1.query():
            time.sleep(2e-5)
        t1 = time.time()
        torch.cuda.synchronize(self.device)
        elapsed_ms = e0.elapsed_time(e1)
        barrier(ws, self.device)
        assert self.lib.gemm_last_device_status(self.stream) == self.lib.GEMM_OK
        return elapsed_ms, names, launches, t0, t1

    def roofline(self, kernel, ms_per_step, timed_s, clocks, sms):
        """Roofline object of the dominant (only) kernel of the timed region."""
        w = self.w
        peaks, peak_src = load_peaks()
        kname = kernel.split("<")[0]
        achieved = w.flops / (ms_per_step * 1e-3) / 1e12
        if kname in ("gemm_bf16_tc", "gemm_f16_tc"):
            key = "bf16_tflops_sustained" if timed_s > 1.0 else "bf16_tflops"
            peak = float(peaks.get(key, FALLBACK_PEAKS[key]))
            kind = "sustained" if key.endswith("sustained") else "burst"
            roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                    "frac": achieved / peak, "peak_source": f"{peak_src} cuBLAS bf16 {kind}"}
            other = "bf16_tflops" if kind == "sustained" else "bf16_tflops_sustained"
            if other in peaks:
                roof["frac_vs_" + ("burst" if kind == "sustained" else "sustained")] = \
                    achieved / float(peaks[other])
        else:
            max_mhz = float(peaks.get("sm_max_mhz", 2070.0))
            peak = fp32_core_peak_tflops(sms, max_mhz)
            roof = {"bound": "alu", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                    "frac": achieved / peak,
                    "peak_source": f"FP32 FMA peak {sms} SMs x 128 lanes x 2 x {max_mhz:.0f} MHz"}
            if clocks and clocks.get("sm_mhz"):
                roof["peak_at_run_clock"] = fp32_core_peak_tflops(sms, clocks["sm_mhz"])
                roof["frac_at_run_clock"] = achieved / roof["peak_at_run_clock"]
        hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
        alg = algorithmic_bytes(w.M, w.N, w.K, self.in_bytes, w.beta)
        roof_tflops = roofline_tflops(w.flops, alg, peak, hbm)
        roof = hbm_bound_roof(roof, alg, ms_per_step * 1e-3, hbm, peak_src, roof_tflops)
        roof["algorithmic_bytes"] = alg
        roof["roof_min_peak_ibw"] = roof_tflops
        roof["traffic"] = committed_traffic(kname, w.name)
        roof["kernel"] = kname
        return roof

    def spot_check(self, target_s, threads=0):
        """The oracle on whole rows of the first copy's D (bounded sample):
        returns (cpu_baseline object, largest |D - D_ref| / bound)."""
        import numpy as np
        w, inp = self.w, self.inp
        cpu = run_cpu_baseline(w, inp, target_s=target_s, threads=threads)
        rows = cpu.pop("_rows")
        Dref, S = cpu.pop("_D"), cpu.pop("_S")
        D = self.rot[0][3]
        got = D[:rows].cpu().numpy().reshape(-1).astype(np.float64)
        ref = Dref.astype(np.float32).astype(np.float64)
        if w.dtype == "f32":
            tol = 1e-5 * S
            if inp["C_logical"] is not None:
                tol = tol + 1e-6 * np.abs(w.beta * inp["C_logical"][:rows].numpy().reshape(-1))
        else:
            tol = 4e-3 * S + 1e-6
        err = float(np.max(np.abs(got - ref) / np.maximum(tol, 1e-300)))
        cpu["sample_max_err_over_tol"] = err
        return cpu, err


# Configs timed after the headline, in the same process, each for at least
# SECONDARY_MIN_S (so a 50 ms clock sampler sees the load): the FP32 4096^3
# target and the MLP up-projection with its beta = 1 epilogue.
SECONDARY = ("f32_4096", "bf16_mlp")
SECONDARY_MIN_S = 0.6


def bench_ours(args):
    import torch
    import dense_gemm_08_gb300 as lib

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    w = resolve_workload(args)
    stream = torch.cuda.current_stream(device)
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    bus_id = nvml_bus_id(local)
    wb = Workbench(lib, w, device, stream)
    kernel, t_host = wb.warm(args.warmup)

    with NvmlSampler(bus_id, local) as nvml, ClockSampler(bus_id or local) as smi:
        elapsed_ms, kernel_names, launches, t0, t1 = wb.timed(args.steps, t_host, ws)
    clk = region_clocks(nvml.rows, getattr(smi, "rows", []), t0, t1)
    elapsed_ms = max_over_ranks(elapsed_ms, ws, device)
    ms_per_step = elapsed_ms / args.steps
    tflops = ws * w.flops * args.steps / (elapsed_ms * 1e-3) / 1e12

    # ---- end to end through the C ABI with host buffers
    # Every step copies its A and B (and C) from pinned host memory, runs the
    # GEMM and copies D back to pinned host memory.  Steps are pipelined over
    # three streams with two device buffer sets: step i+1's inputs travel in
    # while step i computes and step i-1's result travels out.
    e2e = None
    if not args.no_e2e:
        inp = wb.inp
        A, B, C, D = wb.rot[0]
        hA = inp["A"].pin_memory()
        hB = inp["B"].pin_memory()
        hC = inp["C"].pin_memory() if inp["C"] is not None else None
        hD = [torch.empty((w.M, w.N), dtype=torch.float32).pin_memory() for _ in range(2)]
        sets = [(A, B, C, D)]
        sets.append((torch.empty_like(A), torch.empty_like(B),
                     torch.empty_like(C) if C is not None else None, torch.empty_like(D)))
        s_in, s_mm, s_out = (torch.cuda.Stream(device) for _ in range(3))

        def run_e2e(n):
            ev_in = [torch.cuda.Event() for _ in range(n)]
            ev_mm = [torch.cuda.Event() for _ in range(n)]
            ev_out = [torch.cuda.Event() for _ in range(n)]
            t_start = torch.cuda.Event(enable_timing=True)
            t_end = torch.cuda.Event(enable_timing=True)
            t_start.record(s_in)
            for i in range(n):
                dA, dB, dC, dD = sets[i % 2]
                with torch.cuda.stream(s_in):
                    if i >= 2:
                        s_in.wait_event(ev_mm[i - 2])  # the GEMM that read this set is done
                    dA.copy_(hA, non_blocking=True)
                    dB.copy_(hB, non_blocking=True)
                    if hC is not None:
                        dC.copy_(hC, non_blocking=True)
                    ev_in[i].record(s_in)
                s_mm.wait_event(ev_in[i])
                if i >= 2:
                    s_mm.wait_event(ev_out[i - 2])  # this set's D has been copied out
                wb.fn(w.M, w.N, w.K, w.alpha, dA, inp["lda"], w.order_a, dB, inp["ldb"],
                      w.order_b, w.beta, dC, inp["ldc"], dD, w.N, w.order_cd, s_mm)
                ev_mm[i].record(s_mm)
                s_out.wait_event(ev_mm[i])
                with torch.cuda.stream(s_out):
                    hD[i % 2].copy_(dD, non_blocking=True)
                    ev_out[i].record(s_out)
            s_out.wait_event(ev_out[n - 1])
            t_end.record(s_out)
            torch.cuda.synchronize(device)
            return t_start.elapsed_time(t_end)

        e2e_steps = max(4, min(args.steps, 20))
        run_e2e(3)  # warm-up
        barrier(ws, device)
        e2e_ms = max_over_ranks(run_e2e(e2e_steps), ws, device)
        h2d = hA.numel() * hA.element_size() + hB.numel() * hB.element_size()
        if hC is not None:
            h2d += hC.numel() * 4
        e2e = {"value": ws * w.flops * e2e_steps / (e2e_ms * 1e-3) / 1e12, "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": hD[0].numel() * 4,
               "ms_per_step": e2e_ms / e2e_steps, "steps": e2e_steps,
               "pipelining": "3 streams (copy in / GEMM / copy out), 2 device buffer sets"}
        del sets, hA, hB, hC, hD

    # ---- the other targets, each timed in its own region of >= SECONDARY_MIN_S
    secondary = {}
    names = [] if args.secondary in ("", "none") or args.shape else args.secondary.split(",")
    for name in names:
        if name == w.name:
            continue
        from dense_gemm_08_gb300.inputs import WORKLOADS
        w2 = WORKLOADS[name]
        wb2 = Workbench(lib, w2, device, stream)
        k2, t_host2 = wb2.warm(max(args.warmup, 3))
        # calibrate the step time, then run enough steps for the minimum region
        cal_ms, _, _, _, _ = wb2.timed(5, t_host2, ws)
        steps2 = max(args.steps, int(SECONDARY_MIN_S / (cal_ms / 5 * 1e-3)) + 1)
        with NvmlSampler(bus_id, local) as nvml2, ClockSampler(bus_id or local) as smi2:
            el2, names2, launches2, u0, u1 = wb2.timed(steps2, t_host2, ws)
        clk2 = region_clocks(nvml2.rows, getattr(smi2, "rows", []), u0, u1)
        el2 = max_over_ranks(el2, ws, device)
        ms2 = el2 / steps2
        entry = {"metric": METRIC, "value": ws * w2.flops * steps2 / (el2 * 1e-3) / 1e12,
                 "unit": UNIT, "ms_per_step": ms2, "steps": steps2, "warmup": max(args.warmup, 3),
                 "dtype": w2.dtype, "config": workload_config(w2, l2=wb2.l2_note()),
                 "roofline": wb2.roofline(k2, ms2, el2 * 1e-3, clk2, sms),
                 "clocks": clk2, "gpu_launches": launches2, "kernels": sorted(names2)}
        if rank == 0 and not args.no_cpu_baseline:
            cpu2, err2 = wb2.spot_check(target_s=2.0)
            entry["sample_max_err_over_tol"] = err2
            entry["oracle_sample"] = cpu2["sample"]
        secondary[name] = entry
        del wb2
        torch.cuda.empty_cache()

    if rank != 0:
        if ws > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return None

    roof = wb.roofline(kernel, ms_per_step, elapsed_ms * 1e-3, clk, sms)
    cpu = None
    if not args.no_cpu_baseline:
        # the oracle's sample doubles as a parity spot check of the timed output
        cpu, _ = wb.spot_check(target_s=args.cpu_seconds, threads=args.cpu_threads)

    line = {
        "metric": METRIC, "value": tflops, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": w.dtype, "data": "synthetic",
        "config": workload_config(
            w, queue="timed steps enqueued behind a GPU-side delay, run back to back",
            l2=wb.l2_note(), parallelism=f"replicas x{ws}" if ws > 1 else "single GPU"),
        "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches,
        "kernels": sorted(kernel_names), "clocks": clk,
    }
    if secondary:
        line["secondary"] = secondary
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return line


# ---------------------------------------------------------- reference arm
def bench_reference(args):
    from dense_gemm_08_gb300.inputs import make_inputs
    ws, rank, _ = dist_env()
    if rank != 0:
        return None
    w = resolve_workload(args)
    inp = make_inputs(w, seed=0)
    per_step = max(0.5, min(10.0, args.ref_seconds / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        run_cpu_baseline(w, inp, target_s=per_step, threads=args.cpu_threads)
    t_total, flops_total, cores, rows_total = 0.0, 0.0, 0, 0
    for _ in range(args.steps):
        r = run_cpu_baseline(w, inp, target_s=per_step, threads=args.cpu_threads)
        t_total += r["seconds"]
        flops_total += 2.0 * r["_rows"] * w.N * w.K
        rows_total += r["_rows"]
        cores = r["cores"]
    value = flops_total / t_total / 1e12
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_total * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": workload_config(
            w, queue="oracle on the host cores, each step whole rows of D",
            parallelism="single process"),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{args.steps} steps, each whole rows of D (total {rows_total} "
                                   f"rows x {w.N}, K = {w.K}) sized to ~{per_step:.1f} s"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


# ------------------------------------------------- pipeline-depth sweep
def fit_saturating(S, T):
    """Least-squares fit of T = P * S / (S + kappa), the pipelined-throughput
    model of "High-Performance FP16 GEMM on NVIDIA Ada Lovelace via CUTLASS
    and WMMA" (pipeline-depth analysis).  For a fixed kappa the best P is
    linear least squares; kappa is searched on a log grid, then refined.
    Returns (P, kappa, rms)."""
    import math
    S = [float(x) for x in S]
    T = [float(x) for x in T]

    def fit_at(kappa):
        x = [s / (s + kappa) for s in S]
        P = sum(t * xi for t, xi in zip(T, x)) / sum(xi * xi for xi in x)
        rms = math.sqrt(sum((t - P * xi) ** 2 for t, xi in zip(T, x)) / len(T))
        return rms, P, kappa

    best = min(fit_at(10 ** (-3 + 6 * i / 6000)) for i in range(6001))
    lo, hi = best[2] / 1.01, best[2] * 1.01
    for _ in range(60):  # golden-section refinement around the grid minimum
        a, b = lo + 0.382 * (hi - lo), lo + 0.618 * (hi - lo)
        if fit_at(a)[0] < fit_at(b)[0]:
            hi = b
        else:
            lo = a
    rms, P, kappa = fit_at((lo + hi) / 2)
    return P, kappa, rms


def fit_littles_law(S, T):
    """Least-squares fit of T = min(P, b * S): each stage in flight covers a
    fixed slice of the load latency (Little's law) until the compute ceiling P.
    Tries every split of the depths (sorted) into a rising part, fitted by b
    through the origin, and a flat part, fitted by its mean.  Returns
    (P, b, rms)."""
    import math
    pts = sorted(zip((float(s) for s in S), (float(t) for t in T)))
    best = None
    for j in range(1, len(pts)):
        rise, flat = pts[:j], pts[j:]
        b = sum(s * t for s, t in rise) / sum(s * s for s, _ in rise)
        P = sum(t for _, t in flat) / len(flat)
        rms = math.sqrt(sum((t - min(P, b * s)) ** 2 for s, t in pts) / len(pts))
        if best is None or rms < best[2]:
            best = (P, b, rms)
    return best


def bench_sweep_stages(args):
    """--sweep-stages S1,S2,...: builds the library once per CTA-pair ring
    depth S (only the tensor-core unit recompiled: the direct-epilogue ring,
    which BF16 8192^3 runs, gets S stages, -DGEMM_TC_DIRECT_STAGES=S; the
    staged ring, which the MLP shape's beta = 1 needs, min(S, 6)) and times
    BF16 8192^3 and the MLP shape with each, in a fresh process per depth,
    over --sweep-reps rounds in rotated order; prints the median TFLOPS per
    depth and the two fits as one JSON line."""
    from concurrent.futures import ThreadPoolExecutor
    from dense_gemm_08_gb300 import _build

    stages = [int(x) for x in args.sweep_stages.split(",")]
    _build.build()
    with ThreadPoolExecutor(len(stages)) as ex:
        paths = list(ex.map(lambda S: _build.build_variant(
            f"stages{S}", {"GEMM_TC_DIRECT_STAGES": S, "GEMM_TC_PAIR_STAGES": min(S, 5)}),
            stages))
    libs = dict(zip(stages, paths))
    runs = {"bf16_8192": {S: [] for S in stages}, "bf16_mlp": {S: [] for S in stages}}
    clocks = {S: [] for S in stages}
    for rep in range(args.sweep_reps):
        order = stages[rep % len(stages):] + stages[:rep % len(stages)]
        for S in order:
            cmd = [sys.executable, os.path.abspath(__file__), "--workload", "bf16_8192",
                   "--secondary", "bf16_mlp", "--steps", str(args.steps), "--warmup",
                   str(args.warmup), "--no-e2e", "--no-cpu-baseline"]
            env = dict(os.environ, DENSE_GEMM_08_GB300_LIB=libs[S])
            out = subprocess.run(cmd, env=env, capture_output=True, text=True, check=True)
            line = json.loads(out.stdout.strip().splitlines()[-1])
            runs["bf16_8192"][S].append(line["value"])
            runs["bf16_mlp"][S].append(line["secondary"]["bf16_mlp"]["value"])
            clocks[S].append(line["clocks"].get("sm_mhz"))
    result = {"sweep": "pair ring depth", "stages": stages, "reps": args.sweep_reps,
              "steps": args.steps, "stage_kib_per_cta": 32}
    for wl, per in runs.items():
        med = [statistics.median(per[S]) for S in stages]
        P, kappa, rms = fit_saturating(stages, med)
        P2, b, rms2 = fit_littles_law(stages, med)
        result[wl] = {"tflops_median": med, "tflops_all": [per[S] for S in stages],
                      "fit_saturating": {"P": P, "kappa": kappa, "rms": rms},
                      "fit_littles_law": {"P": P2, "b_per_stage": b, "rms": rms2}}
    result["sm_mhz_median"] = [statistics.median([c for c in clocks[S] if c] or [0])
                               for S in stages]
    return result


# ------------------------------------------------------------- peak probes
# Dense BF16 tensor-core rate per SM and clock: a 128 x 256 x 16 MMA of one
# CTA (1,048,576 FLOP) every 128 cycles, 8192 FLOP per cycle per SM.
BF16_FLOP_PER_CLK_PER_SM = 8192


def bf16_formula_tflops(sms, mhz):
    """Dense BF16 tensor peak from the SM count and clock: SMs x 8192 x clock."""
    return sms * BF16_FLOP_PER_CLK_PER_SM * mhz * 1e6 / 1e12



def bench_probe(args):
    """--probe: the library's peak probes (tensor pipe, FP32 FMA pipe), timed
    with CUDA events on the launching stream; one JSON line, rank 0 only."""
    import torch
    import dense_gemm_08_gb300 as lib

    ws, rank, local = dist_env()
    if rank != 0:
        return None
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    stream = torch.cuda.current_stream(device)
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    reps = max(args.steps, 5)

    def timed(launch):
        for _ in range(args.warmup):
            launch()
        torch.cuda.synchronize(device)
        times, flops = [], 0.0
        for _ in range(reps):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            _, flops = launch()
            e1.record(stream)
            e1.synchronize()
            times.append(e0.elapsed_time(e1) * 1e-3)
        st = lib.gemm_last_device_status(stream)
        if st != lib.GEMM_OK:
            raise RuntimeError(f"probe device status {st}: {lib.gemm_status_string(st)}")
        med = statistics.median(times)
        return {"tflops": flops / med / 1e12, "ms": med * 1e3, "flops": flops}

    # each launch about 10 ms at 2 PFLOP/s (tensor) or 80 TFLOP/s (FMA)
    n_mma = int(0.010 * 2.0e15 / (2 ** 20 * sms))
    trips = int(0.010 * 80e12 / (2 * 8 * 16 * sms * 8 * 256))
    peaks, src = load_peaks()
    with ClockSampler(local) as clk:
        tc1 = timed(lambda: lib.gemm_probe_tc_bf16(1, n_mma, stream))
        tc2 = timed(lambda: lib.gemm_probe_tc_bf16(2, n_mma, stream))
        fma = timed(lambda: lib.gemm_probe_fma_f32(trips, stream))
    clocks = clock_summary(clk.rows)
    mhz = clocks["sm_mhz"] if clocks and clocks["sm_mhz"] else None
    max_mhz = clocks["sm_max_mhz"] if clocks and clocks["sm_max_mhz"] else 2070.0
    return {
        "probe": "peaks", "n_gpus": 1, "steps": reps, "warmup": args.warmup,
        "tc_bf16_pair": dict(tc2, n_mma=n_mma, mma="256x256x16 per CTA pair"),
        "tc_bf16_single": dict(tc1, n_mma=n_mma, mma="128x256x16 per CTA"),
        "fma_f32": dict(fma, trips=trips),
        "bf16_formula_tflops": {"at_max_clock": bf16_formula_tflops(sms, max_mhz),
                                "at_run_clock": bf16_formula_tflops(sms, mhz) if mhz else None,
                                "flop_per_clk_per_sm": BF16_FLOP_PER_CLK_PER_SM, "sms": sms},
        "measured_cublas_bf16_tflops": {"burst": peaks.get("bf16_tflops"),
                                        "sustained": peaks.get("bf16_tflops_sustained"),
                                        "source": src},
        "fp32_formula_tflops": {"at_max_clock": fp32_core_peak_tflops(sms, max_mhz),
                                "at_run_clock": fp32_core_peak_tflops(sms, mhz) if mhz else None,
                                "sms": sms},
        "clocks": clocks,
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="bf16_8192")
    ap.add_argument("--shape", default=None,
                    help="M,N,K overriding the workload's sizes (profiling on smaller cases)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-seconds", type=float, default=60.0)
    ap.add_argument("--cpu-threads", type=int, default=0,
                    help="host threads of the oracle (reference arm and CPU baseline); 0: all cores")
    ap.add_argument("--secondary", default=",".join(SECONDARY),
                    help="workloads timed after the headline, each in its own region "
                         "(comma list, or 'none')")
    ap.add_argument("--sweep-stages", default=None,
                    help="comma list of CTA-pair ring depths to build and time (2..7)")
    ap.add_argument("--sweep-reps", type=int, default=2)
    ap.add_argument("--probe", action="store_true",
                    help="time the library's peak probes instead of a GEMM workload")
    args = ap.parse_args(argv)
    args.warmup = max(args.warmup, 3)  # timing rule: at least 3 untimed warm-up steps
    if args.sweep_stages:
        line = bench_sweep_stages(args)
    elif args.probe:
        line = bench_probe(args)
    else:
        line = bench_reference(args) if args.impl == "reference" else bench_ours(args)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
