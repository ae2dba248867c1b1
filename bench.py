#!/usr/bin/env python3
"""Benchmark: sliding-window + sink attention on B300.

One step = one sliding-window prefill call over the B=4, T=8192, Hq=64, Hkv=8,
D=128, W=128 workload (bf16 q/k/v, fp32 sink, fp32 out + per-row LSE), inputs
resident in HBM.  ``value`` is algorithmic TFLOP/s (only in-window query/key
pairs count, 4*D FLOPs each).  The same JSON line also carries the ring-buffer
decode measurement (256 sequences, W=128, GB/s of algorithmic bytes), the
roofline of each kernel against the measured peaks, the end-to-end number
through host buffers, the CPU oracle baseline and the SM clocks seen.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

``--impl reference`` times the fp64 CPU oracle (the only reference for this
operation) on the host cores, on a bounded sample of the same workload.
Under torchrun (N > 1) every rank runs its own replica (no data exchange);
time is the max over ranks and ``value`` the total over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from hybrid_sliding_window_02_b300 import inputs as gen  # noqa: E402
from hybrid_sliding_window_02_b300 import work  # noqa: E402

METRIC = "SWA+sink prefill TFLOP/s & decode GB/s on 1 B300, as % of roofline vs CPU oracle"
PREFILL = dict(B=4, T=8192, Hq=64, Hkv=8, D=128, W=128)
DECODE = dict(B=256, Hq=64, Hkv=8, D=128, W=128)
VERIFY = dict(B=256, L=4, Hq=64, Hkv=8, D=128, W=128)
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
# sources each kernel is built from (its traffic record is void once they change)
KERNEL_SOURCES = {
    "swa_fwd_tc_kernel": ("csrc/tc_swa.cuh", "csrc/device_common.cuh"),
    "swa_fwd_tc_global_kernel": ("csrc/tc_global.cuh", "csrc/device_common.cuh"),
    "decode_tc_kernel": ("csrc/decode_tc.cuh", "csrc/device_common.cuh", "csrc/griddep.cuh"),
    "verify_tc_kernel": ("csrc/verify_tc.cuh", "csrc/device_common.cuh", "csrc/griddep.cuh"),
}


def workload_name(c):
    return (f"swa_sink_prefill B{c['B']} T{c['T']} Hq{c['Hq']} Hkv{c['Hkv']} D{c['D']} "
            f"W{c['W']} bf16->fp32+lse")


# ---------------------------------------------------------------------------
# distributed plumbing (replicas only)
# ---------------------------------------------------------------------------
class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            backend = "nccl" if torch.cuda.is_available() else "gloo"
            if backend == "nccl":
                torch.cuda.set_device(self.local_rank)
            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg is not None:
            if torch.cuda.is_available():
                self.pg.barrier(device_ids=[self.local_rank])
            else:
                self.pg.barrier()

    def max(self, x: float) -> float:
        return reduce_value(self.pg, x, "max")

    def sum(self, x: float) -> float:
        return reduce_value(self.pg, x, "sum")

    def close(self):
        if self.pg is not None:
            self.pg.destroy_process_group()


def job_rate(dist, units: float, ms: float):
    """Whole-job rate over replicas: the units all ranks processed divided by
    the slowest rank's time.  Returns (units per second, max ms)."""
    ms_max = dist.max(ms)
    return dist.sum(units) / (ms_max * 1e-3), ms_max


def reduce_value(pg, x: float, op: str) -> float:
    """Reduce a float over ranks (identity without a process group)."""
    if pg is None:
        return float(x)
    dev = torch.device("cuda", torch.cuda.current_device()) if (
        torch.cuda.is_available() and pg.get_backend() == "nccl") else torch.device("cpu")
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    pg.all_reduce(t, op=pg.ReduceOp.MAX if op == "max" else pg.ReduceOp.SUM)
    return float(t.item())


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class _NvmlLib:
    """The few NVML calls the sampler needs, through ctypes on the driver's
    libnvidia-ml (used when the pynvml module is not installed).  Reads only."""

    CLOCK_SM = 1

    def __init__(self, device_index: int):
        import ctypes
        self.ct = ctypes
        self.L = ctypes.CDLL("libnvidia-ml.so.1")
        if self.L.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit_v2 failed")
        self.h = ctypes.c_void_p()
        rc = -1
        try:  # match the CUDA device to its NVML handle by UUID
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
            rc = self.L.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.h))
        except Exception:
            rc = -1
        if rc != 0 and self.L.nvmlDeviceGetHandleByIndex_v2(device_index,
                                                            ctypes.byref(self.h)) != 0:
            raise RuntimeError("no NVML handle for the device")
        self._reasons = getattr(self.L, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.L.nvmlDeviceGetCurrentClocksThrottleReasons

    def sm_mhz(self):
        v = self.ct.c_uint()
        return v.value if self.L.nvmlDeviceGetClockInfo(self.h, self.CLOCK_SM,
                                                         self.ct.byref(v)) == 0 else None

    def sm_max_mhz(self):
        v = self.ct.c_uint()
        return v.value if self.L.nvmlDeviceGetMaxClockInfo(self.h, self.CLOCK_SM,
                                                            self.ct.byref(v)) == 0 else None

    def reasons(self):
        v = self.ct.c_ulonglong()
        return v.value if self._reasons(self.h, self.ct.byref(v)) == 0 else 0


class ClockSampler:
    """Samples the SM clock and clock-event (throttle) reasons while a timed
    region runs: through NVML (the pynvml module, else the driver's NVML
    library through ctypes) in a thread about every millisecond, or, if NVML
    is unavailable, from an ``nvidia-smi -lms`` subprocess."""

    REASONS = {
        "applications_clocks_setting": 0x2, "sw_power_cap": 0x4, "hw_slowdown": 0x8,
        "sync_boost": 0x10, "sw_thermal_slowdown": 0x20, "hw_thermal_slowdown": 0x40,
        "hw_power_brake_slowdown": 0x80,
    }
    SMI_FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.sw_power_cap,"
                  "clocks_event_reasons.hw_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                  "clocks_event_reasons.hw_thermal_slowdown")
    _nvml_cache = {}

    def __init__(self, device_index: int, period_s: float = 0.001):
        self.idx = device_index
        self.period = period_s
        self.samples = []
        self.reasons = set()
        self.max_mhz = None
        self.source = None
        self.error = None
        self._stop = threading.Event()
        self._thread = None
        self._proc = None
        self._nv = None
        try:
            self._nv = self._open(device_index)
            self.max_mhz = self._nv.sm_max_mhz()
            self.source = "nvml"
        except Exception as e:  # fall back to nvidia-smi
            self._nv = None
            self.error = f"nvml: {type(e).__name__}: {e}"
            self.source = "nvidia-smi"

    @classmethod
    def _open(cls, device_index):
        if device_index in cls._nvml_cache:
            return cls._nvml_cache[device_index]
        try:
            import pynvml
            pynvml.nvmlInit()
            try:
                uuid = str(torch.cuda.get_device_properties(device_index).uuid)
                h = pynvml.nvmlDeviceGetHandleByUUID(
                    uuid if uuid.startswith("GPU-") else "GPU-" + uuid)
            except Exception:
                h = pynvml.nvmlDeviceGetHandleByIndex(device_index)
            rf = (getattr(pynvml, "nvmlDeviceGetCurrentClocksEventReasons", None)
                  or getattr(pynvml, "nvmlDeviceGetCurrentClocksThrottleReasons"))

            class _Py:
                def sm_mhz(self):
                    return pynvml.nvmlDeviceGetClockInfo(h, pynvml.NVML_CLOCK_SM)

                def sm_max_mhz(self):
                    return pynvml.nvmlDeviceGetMaxClockInfo(h, pynvml.NVML_CLOCK_SM)

                def reasons(self):
                    return rf(h)
            nv = _Py()
        except ImportError:
            nv = _NvmlLib(device_index)
        cls._nvml_cache[device_index] = nv
        return nv

    def _run_nvml(self):
        nv = self._nv
        while not self._stop.is_set():
            try:
                mhz = nv.sm_mhz()
                if mhz is not None:
                    self.samples.append(float(mhz))
                mask = nv.reasons()
                for name, bit in self.REASONS.items():
                    if mask & bit:
                        self.reasons.add(name)
            except Exception as e:
                self.error = f"nvml sample: {e}"
            time.sleep(self.period)

    def __enter__(self):
        if self.source == "nvml":
            self._thread = threading.Thread(target=self._run_nvml, daemon=True)
            self._thread.start()
        else:
            import subprocess
            try:
                self._proc = subprocess.Popen(
                    ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.SMI_FIELDS}",
                     "--format=csv,noheader,nounits", "-lms", "50"],
                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            except Exception as e:
                self.error = (self.error or "") + f"; nvidia-smi: {e}"
        return self

    def __exit__(self, *exc):
        if self._thread is not None:
            self._stop.set()
            self._thread.join()
        if self._proc is not None:
            self._proc.terminate()
            out, _ = self._proc.communicate(timeout=10)
            names = ("sw_power_cap", "hw_slowdown", "sw_thermal_slowdown", "hw_thermal_slowdown")
            for line in out.splitlines():
                f = [x.strip() for x in line.split(",")]
                if len(f) < 6:
                    continue
                try:
                    self.samples.append(float(f[0]))
                    self.max_mhz = float(f[1])
                except ValueError:
                    continue
                for name, val in zip(names, f[2:6]):
                    if val.lower() == "active":
                        self.reasons.add(name)

    def median(self):
        return statistics.median(self.samples) if self.samples else None

    def summary(self):
        d = {"sm_mhz": self.median(), "sm_max_mhz": self.max_mhz,
             "reasons": sorted(self.reasons), "samples": len(self.samples),
             "source": self.source}
        if not self.samples and self.error:
            d["error"] = self.error
        return d


# ---------------------------------------------------------------------------
# peaks, traffic records
# ---------------------------------------------------------------------------
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def source_code_only(text: str) -> str:
    """C/CUDA source with comments and whitespace removed (string literals kept):
    what the traffic of a kernel depends on, so that editing a comment does not
    retire a recorded measurement."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        elif c == '"':
            j = i + 1
            while j < n and text[j] != '"':
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        else:
            if not c.isspace():
                out.append(c)
            i += 1
    return "".join(out)


def kernel_source_hash(kernel: str) -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "hybrid_sliding_window_02_b300", rel), encoding="utf-8") as f:
            h.update(source_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def traffic_shape(**dims) -> str:
    """The key a traffic record is stored under: the workload's sizes, e.g.
    "B4 T8192 Hq64 Hkv8 D128 W128"."""
    return " ".join(f"{k}{v}" for k, v in dims.items())


def recorded_traffic(kernel: str, shape: str, path: str = "", record: str = ""):
    """DRAM bytes (read + write) per launch of the bench workload, from the
    committed ncu summary ``profiles/dram_traffic.txt`` (or ``path``); None if
    absent, if the record was taken on another workload shape, or if the
    kernel's sources have changed since the counters were taken.  ``record``
    names a second record of the same kernel (another mode of it); it defaults
    to the kernel's name."""
    path = path or os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if kernel not in KERNEL_SOURCES or not os.path.exists(path):
        return None
    rec = {}
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#") or ":" not in line:
                continue
            key, val = line.split(":", 1)
            rec[key.strip()] = val.strip()
    record = record or kernel
    if rec.get(f"{record}.source_hash") != kernel_source_hash(kernel):
        return None
    if rec.get(f"{record}.shape") != shape:
        return None
    val = rec.get(f"{record}.bytes_per_launch")
    return int(float(val)) if val else None


# ---------------------------------------------------------------------------
# CPU oracle baseline
# ---------------------------------------------------------------------------
def oracle_rows_rate(q, k, v, sink, W, i0, ts):
    """Run the fp64 oracle on rows i0..i0+ts-1 (all heads) of batch entry 0 and
    return (seconds, FLOPs, rows).  Only the key range those rows read is
    copied to the host."""
    import oracle
    Hq, D = q.shape[2], q.shape[3]
    j0 = max(0, i0 - W + 1)
    qs, ks, vs = (x[0:1, j0:i0 + ts].cpu() for x in (q, k, v))
    rows = [[0, h, i - j0] for i in range(i0, i0 + ts) for h in range(Hq)]
    t0 = time.perf_counter()
    oracle.swa_sink_fwd_rows(qs, ks, vs, sink.cpu(), W, rows)
    dt = time.perf_counter() - t0
    npairs = sum(min(i + 1, W) for i in range(i0, i0 + ts))
    return dt, 4 * D * Hq * npairs, len(rows)


def cpu_oracle_sample(q, k, v, sink, W, target_s=12.0, i0=None):
    """Time the fp64 oracle on consecutive full-window rows of batch entry 0
    (all heads), sized for about target_s seconds of host work."""
    import oracle
    nthr = oracle.num_threads()
    T, Hq = q.shape[1], q.shape[2]
    i0 = min(W, T - 1) if i0 is None else i0
    ts = min(T - i0, 16)
    dt, flops, nrows = oracle_rows_rate(q, k, v, sink, W, i0, ts)
    while dt < target_s / 4 and ts < T - i0:
        ts = min(T - i0, int(ts * max(2.0, min(8.0, target_s / max(dt, 1e-3) / 2))))
        dt, flops, nrows = oracle_rows_rate(q, k, v, sink, W, i0, ts)
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": nthr, "kind": "oracle",
            "sample": f"batch entry 0, positions {i0}..{i0 + ts - 1}, all {Hq} heads "
                      f"({nrows} rows, {flops:.3e} FLOP) in {dt:.2f} s"}


def cpu_oracle_call(fn, units, unit, sample):
    """Time one oracle call over the whole workload of a line; ``units`` is the
    line's work (bytes or FLOPs) and ``unit`` its rate unit."""
    import oracle
    t0 = time.perf_counter()
    fn()
    dt = time.perf_counter() - t0
    scale = 1e9 if unit == "GB/s" else 1e12
    return {"value": units / dt / scale, "unit": unit, "cores": oracle.num_threads(),
            "kind": "oracle", "sample": f"{sample} in {dt:.2f} s"}


def cpu_global_layer(x, T):
    """The fp64 oracle on the global layer's last 128 positions (all heads:
    8192 rows, the longest ones), and the whole layer's time extrapolated from
    that rate by its exact pair count."""
    D, Hq = x.q.shape[3], x.q.shape[2]
    dt, flops, nrows = oracle_rows_rate(x.q, x.k, x.v, x.sink, T, T - 128, 128)
    full = work.prefill_flops(1, T, Hq, D, T)
    return flops / dt, (f"global layer: positions {T - 128}..{T - 1}, all {Hq} heads ({nrows} "
                        f"rows, {flops:.3e} FLOP) in {dt:.2f} s; the layer's "
                        f"{full:.3e} FLOP extrapolated at that rate")


def with_clocks(dev, fn):
    """Run fn under a clock sampler; returns (fn's result, clock summary)."""
    with ClockSampler(dev.index) as clk:
        r = fn()
    return r, clk.summary()


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------
def time_prefill(swa, x, c, steps, warmup, dist, stream):
    B, T, Hq, Hkv, D, W = (c[k] for k in ("B", "T", "Hq", "Hkv", "D", "W"))
    out = torch.empty(B, T, Hq, D, dtype=torch.float32, device=x.q.device)
    lse = torch.empty(B, Hq, T, dtype=torch.float32, device=x.q.device)
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            swa.swa_sink_fwd(x.q, x.k, x.v, x.sink, W, out, lse, stream=stream)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dist.barrier()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        # a short device-side wait ahead of the first event, so that the host
        # has queued the first launches before the stream reaches it: the
        # events then time the kernels, not the host's first enqueue
        if hasattr(torch.cuda, "_sleep"):
            torch.cuda._sleep(400_000)
        e0.record(stream)
        for s in range(steps):
            ev[s][0].record(stream)
            swa.swa_sink_fwd(x.q, x.k, x.v, x.sink, W, out, lse, stream=stream)
            ev[s][1].record(stream)
        e1.record(stream)
    torch.cuda.synchronize()
    dist.barrier()
    total_ms = e0.elapsed_time(e1)
    per_launch_ms = sum(a.elapsed_time(b) for a, b in ev) / steps
    return total_ms, per_launch_ms


def time_graph(call, sets, steps, warmup, stream, per_graph=32):
    """Mean device time (ms) of one call, launched back to back from a CUDA
    graph of ``per_graph`` calls rotating over ``sets`` (so that the host's
    per-call cost -- argument checks, tensor-map encoding, the launch -- does
    not set the pace of a call shorter than it)."""
    with torch.cuda.stream(stream):
        for i in range(warmup * len(sets)):
            call(sets[i % len(sets)])
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(per_graph):
            call(sets[i % len(sets)])
    reps = max(1, steps // per_graph)
    with torch.cuda.stream(stream):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    del g
    return e0.elapsed_time(e1) / (reps * per_graph)


def decode_line(swa, dev, stream, steps, hbm, cpu, nsets=4, c=None):
    """Decode calls rotating over input sets whose total exceeds L2."""
    c = c or DECODE
    B, Hq, Hkv, D, W = (c[k] for k in ("B", "Hq", "Hkv", "D", "W"))
    sets = [gen.decode_inputs(B, Hq, Hkv, D, W, seed=100 + i, device=dev) for i in range(nsets)]
    out = torch.empty(B, Hq, D, dtype=torch.float32, device=dev)
    lse = torch.empty(B, Hq, dtype=torch.float32, device=dev)

    def call(d):
        swa.swa_sink_decode(d.q, d.k_ring, d.v_ring, d.pos, d.sink, out, lse, stream=stream)

    ms, clocks = with_clocks(dev, lambda: time_graph(call, sets, steps, 3, stream))
    nbytes = work.decode_bytes(B, Hq, Hkv, D, W, 2)
    gbs = nbytes / (ms * 1e-3) / 1e9
    kernel = ("decode_tc_kernel" if swa.decode_path(B, Hq, Hkv, D, W) == "tc_decode"
              else "decode_kernel")
    line = {
        "workload": f"decode B{B} Hq{Hq} Hkv{Hkv} D{D} W{W} ring, bf16->fp32+lse, {nsets} sets "
                    "(>L2), graph of 32",
        "value": round(gbs, 1), "unit": "GB/s", "us_per_call": round(ms * 1e3, 2),
        "roofline": {"kernel": kernel, "bound": "hbm", "achieved": round(gbs, 1), "peak": hbm,
                     "unit": "GB/s", "frac": round(gbs / hbm, 4),
                     "bytes_per_launch": nbytes,
                     "traffic": recorded_traffic(kernel, traffic_shape(B=B, Hq=Hq, Hkv=Hkv, D=D,
                                                                       W=W))},
        "clocks": clocks,
    }
    if cpu:
        import oracle
        d = sets[0]
        hc = [t.cpu() for t in (d.q, d.k_ring, d.v_ring, d.pos, d.sink)]
        line["cpu_baseline"] = cpu_oracle_call(
            lambda: oracle.swa_sink_decode(*hc), nbytes, "GB/s", f"the whole call ({B} seqs)")
    return line


def rope_line(swa, dev, stream, reps, hbm, cpu, theta=10000.0):
    """RoPE of a prefill, in place: q and k of the headline workload rotated at
    positions 0 .. T-1 (rot_dim = D), two launches per step; inputs larger
    than L2."""
    c = PREFILL
    B, T, Hq, Hkv, D = (c[k] for k in ("B", "T", "Hq", "Hkv", "D"))
    x = gen.prefill_inputs(B, T, Hq, Hkv, D, seed=7, device=dev)
    pos0 = torch.zeros(B, dtype=torch.int64, device=dev)

    def call():
        swa.swa_rope(x.q, pos0, D, theta, stream=stream)
        swa.swa_rope(x.k, pos0, D, theta, stream=stream)

    ms, clocks = with_clocks(dev, lambda: _event_ms(call, reps, stream))
    nbytes = work.rope_bytes(B, T, Hq, D, 2) + work.rope_bytes(B, T, Hkv, D, 2)
    gbs = nbytes / (ms * 1e-3) / 1e9
    line = {
        "workload": f"RoPE in place of q [B{B} T{T} Hq{Hq} D{D}] and k [Hkv{Hkv}], bf16, rot_dim {D}, "
                    f"theta {theta:g}, positions 0..{T - 1}",
        "value": round(gbs, 1), "unit": "GB/s", "ms_per_step": round(ms, 4),
        "roofline": {"kernel": "rope_inplace_kernel", "bound": "hbm", "achieved": round(gbs, 1),
                     "peak": hbm, "unit": "GB/s", "frac": round(gbs / hbm, 4),
                     "bytes_per_step": nbytes, "traffic": None},
        "clocks": clocks,
    }
    if cpu:
        import oracle
        n = 512   # the first 512 positions of sequence 0, q and k
        qs, ks = x.q[:1, :n].cpu(), x.k[:1, :n].cpu()
        p0 = torch.zeros(1, dtype=torch.int64)
        line["cpu_baseline"] = cpu_oracle_call(
            lambda: (oracle.rope(qs, p0, D, theta), oracle.rope(ks, p0, D, theta)),
            work.rope_bytes(1, n, Hq, D, 2) + work.rope_bytes(1, n, Hkv, D, 2), "GB/s",
            f"q and k of positions 0..{n - 1} of sequence 0")
    return line


def decode_step_line(swa, dev, stream, steps, hbm, cpu, nsets=4, c=None, theta=10000.0):
    """One generated token per sequence: its k and v written into the ring
    (alone: ``swa_ring_append``; fused with the rotation of its q and k:
    ``swa_rope_append``), then decode of the rotated q.  Each part is timed on
    its own and the step as a whole, from CUDA graphs rotating over input sets
    whose total exceeds L2."""
    c = c or DECODE
    B, Hq, Hkv, D, W = (c[k] for k in ("B", "Hq", "Hkv", "D", "W"))
    sets = []
    for i in range(nsets):
        d = gen.decode_inputs(B, Hq, Hkv, D, W, seed=100 + i, device=dev)
        g = torch.Generator(device=dev).manual_seed(400 + i)
        kn = torch.randn(B, Hkv, D, generator=g, device=dev).to(torch.bfloat16)
        vn = torch.randn(B, Hkv, D, generator=g, device=dev).to(torch.bfloat16)
        sets.append((d, kn, vn, torch.empty_like(d.q)))
    out = torch.empty(B, Hq, D, dtype=torch.float32, device=dev)
    lse = torch.empty(B, Hq, dtype=torch.float32, device=dev)

    def append(x):
        d, kn, vn, _ = x
        swa.swa_ring_append(kn, vn, d.k_ring, d.v_ring, d.pos, stream=stream)

    def rope_append(x):
        d, kn, vn, qo = x
        swa.swa_rope_append(d.q, kn, vn, d.k_ring, d.v_ring, d.pos, D, theta, q_out=qo,
                            stream=stream)

    def step(x):
        rope_append(x)
        d, _, _, qo = x
        swa.swa_sink_decode(qo, d.k_ring, d.v_ring, d.pos, d.sink, out, lse, stream=stream)

    ms_app = time_graph(append, sets, steps, 3, stream)
    ms_rope = time_graph(rope_append, sets, steps, 3, stream)
    ms_step, clocks = with_clocks(dev, lambda: time_graph(step, sets, steps, 3, stream))
    b_app = work.append_bytes(B, Hkv, D, 2)
    b_rope = work.rope_append_bytes(B, Hq, Hkv, D, 2)
    b_step = b_rope + work.decode_bytes(B, Hq, Hkv, D, W, 2)
    gbs = b_step / (ms_step * 1e-3) / 1e9
    gbs_rope = b_rope / (ms_rope * 1e-3) / 1e9
    line = {
        "workload": f"decode step B{B} Hq{Hq} Hkv{Hkv} D{D} W{W}: rotate q, k and append k, v "
                    f"(rot_dim {D}, theta {theta:g}), then decode; bf16->fp32+lse, {nsets} sets "
                    "(>L2), graph of 32",
        "value": round(gbs, 1), "unit": "GB/s", "us_per_step": round(ms_step * 1e3, 2),
        "append_us": round(ms_app * 1e3, 2),
        "append_gbs": round(b_app / (ms_app * 1e-3) / 1e9, 1),
        "rope_append_us": round(ms_rope * 1e3, 2),
        # the fused rotate-and-append moves ~10 MB: a few microseconds at any
        # rate, so its fraction says more about launch latency than about HBM
        "roofline": {"kernel": "rope_append_kernel", "bound": "hbm", "achieved": round(gbs_rope, 1),
                     "peak": hbm, "unit": "GB/s", "frac": round(gbs_rope / hbm, 4),
                     "bytes_per_launch": b_rope, "traffic": None},
        "step_frac_of_hbm": round(gbs / hbm, 4),
        "clocks": clocks,
    }
    if cpu:
        import oracle
        d, kn, vn, _ = sets[0]
        hq, hk, hv, kr, vr, pos, sk = (t.cpu() for t in (d.q, kn, vn, d.k_ring, d.v_ring, d.pos,
                                                           d.sink))

        def host_step():
            p0 = pos.clamp(min=0)
            qr = torch.from_numpy(oracle.rope(hq.unsqueeze(1), p0, D, theta)[:, 0])
            kr_new = torch.from_numpy(oracle.rope(hk.unsqueeze(1), p0, D, theta)[:, 0])
            k_ring, v_ring = kr.double(), vr.double()
            for b in range(B):
                if int(pos[b]) >= 0:
                    k_ring[b, :, int(pos[b]) % W] = kr_new[b]
                    v_ring[b, :, int(pos[b]) % W] = hv[b].double()
            oracle.swa_sink_decode(qr, k_ring, v_ring, pos, sk)
        line["cpu_baseline"] = cpu_oracle_call(host_step, b_step, "GB/s",
                                               f"the whole step ({B} seqs)")
    return line


def verify_line(swa, dev, stream, steps, hbm, cpu, nsets=4, c=None):
    """Verify calls (L drafted tokens per sequence) rotating over input sets
    whose total exceeds L2."""
    c = c or VERIFY
    B, L, Hq, Hkv, D, W = (c[k] for k in ("B", "L", "Hq", "Hkv", "D", "W"))
    sets = [gen.verify_inputs(B, L, Hq, Hkv, D, W, seed=300 + i, device=dev)
            for i in range(nsets)]
    out = torch.empty(B, L, Hq, D, dtype=torch.float32, device=dev)
    lse = torch.empty(B, Hq, L, dtype=torch.float32, device=dev)

    def call(d):
        swa.swa_sink_verify(d.q, d.k_new, d.v_new, d.k_ring, d.v_ring, d.pos, d.sink, out, lse,
                            stream=stream)

    ms, clocks = with_clocks(dev, lambda: time_graph(call, sets, steps, 3, stream))
    nbytes = work.verify_bytes(B, L, Hq, Hkv, D, W, 2)
    gbs = nbytes / (ms * 1e-3) / 1e9
    kpath = swa.verify_path(B, L, Hq, Hkv, D, W)
    kernel = "verify_tc_kernel" if kpath == "tc_verify" else "verify_simt_kernel"
    line = {
        "workload": f"verify B{B} L{L} Hq{Hq} Hkv{Hkv} D{D} W{W} ring + {L} drafts, "
                    f"bf16->fp32+lse, {nsets} sets (>L2), graph of 32",
        "value": round(gbs, 1), "unit": "GB/s", "us_per_call": round(ms * 1e3, 2),
        "roofline": {"kernel": kernel, "bound": "hbm", "achieved": round(gbs, 1), "peak": hbm,
                     "unit": "GB/s", "frac": round(gbs / hbm, 4),
                     "bytes_per_launch": nbytes,
                     "traffic": recorded_traffic(kernel, traffic_shape(B=B, L=L, Hq=Hq, Hkv=Hkv,
                                                                       D=D, W=W))},
        "clocks": clocks,
    }
    if cpu:
        import oracle
        d = sets[0]
        hc = [t.cpu() for t in (d.q, d.k_new, d.v_new, d.k_ring, d.v_ring, d.pos, d.sink)]
        line["cpu_baseline"] = cpu_oracle_call(
            lambda: oracle.swa_sink_verify(*hc), nbytes, "GB/s", f"the whole call ({B}x{L})")
    return line


HYBRID = dict(T=32768, Hq=64, Hkv=8, D=128, W=128, n_swa=5, n_ga=1)


def time_hybrid(swa, dev, stream, reps, layers, Ws):
    """One hybrid block: the window layers then the global layer (W = T), each
    on its own seeded inputs, one sequence of T=32768.  Returns per-layer
    mean launch times (ms) measured with events on the launching stream."""
    T, Hq, D = HYBRID["T"], HYBRID["Hq"], HYBRID["D"]
    out = torch.empty(1, T, Hq, D, dtype=torch.float32, device=dev)
    lse = torch.empty(1, Hq, T, dtype=torch.float32, device=dev)

    def block(evs=None):
        for li, (x, W) in enumerate(zip(layers, Ws)):
            if evs is not None:
                evs[li][0].record(stream)
            swa.swa_sink_fwd(x.q, x.k, x.v, x.sink, W, out, lse, stream=stream)
            if evs is not None:
                evs[li][1].record(stream)

    with torch.cuda.stream(stream):
        for _ in range(2):
            block()
    torch.cuda.synchronize()
    per_layer = [0.0] * len(Ws)
    total = 0.0
    with torch.cuda.stream(stream):
        for _ in range(reps):
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in Ws]
            block(evs)
            torch.cuda.synchronize()
            for li, (a, b) in enumerate(evs):
                per_layer[li] += a.elapsed_time(b) / reps
            total += evs[0][0].elapsed_time(evs[-1][1]) / reps
    del out, lse
    return per_layer, total


def hybrid_line(swa, dev, stream, reps, peaks, cpu, n_swa=None, cpu_rates=None):
    c = dict(HYBRID)
    if n_swa is not None:
        c["n_swa"] = n_swa
    T, Hq, Hkv, D = c["T"], c["Hq"], c["Hkv"], c["D"]
    layers = gen.hybrid_block_inputs(T, Hq, Hkv, D, n_swa=c["n_swa"], n_ga=c["n_ga"], seed=200,
                                     device=dev)
    Ws = [c["W"]] * c["n_swa"] + [T] * c["n_ga"]
    (per_layer, total_ms), clocks = with_clocks(
        dev, lambda: time_hybrid(swa, dev, stream, reps, layers, Ws))
    fl = [work.prefill_flops(1, T, Hq, D, W) for W in Ws]
    ga_ms = sum(t for t, W in zip(per_layer, Ws) if W >= T) / max(1, c["n_ga"])
    ga_fl = fl[-1]
    ga_tf = ga_fl / (ga_ms * 1e-3) / 1e12
    swa_ms = sum(t for t, W in zip(per_layer, Ws) if W < T) / c["n_swa"]
    flop_ratio, kv_ratio = work.hybrid_reduction(T, c["W"], c["n_swa"], c["n_ga"])
    peak = float(peaks["bf16_tflops"])
    roof = {"kernel": "swa_fwd_tc_global_kernel", "bound": "tensor",
            "achieved": round(ga_tf, 1), "peak": peak,
            "unit": "TFLOP/s", "frac": round(ga_tf / peak, 4),
            "peak_source": "measured bf16_tflops (burst)",
            # the layer runs inside a seconds-long loop under the power
            # cap: its fraction of the sustained GEMM rate, for context
            "frac_of_sustained": round(ga_tf / float(peaks["bf16_tflops_sustained"]), 4),
            "flops_per_launch": ga_fl,
            "traffic": recorded_traffic("swa_fwd_tc_global_kernel",
                                        traffic_shape(B=1, T=T, Hq=Hq, Hkv=c["Hkv"], D=D, W=T))}
    if clocks.get("sm_mhz") and clocks.get("sm_max_mhz"):
        # time x clock: the layer's rate had it run at the maximum SM clock
        # throughout (the median clock of the line's timed region stands in
        # for the layer's own)
        roof["frac_at_max_clock"] = round(
            ga_tf / peak * clocks["sm_max_mhz"] / clocks["sm_mhz"], 4)
    line = {
        "workload": f"hybrid block {c['n_swa']}x SWA (W={c['W']}) + {c['n_ga']}x global "
                    f"(W=T), B1 T{T} Hq{Hq} Hkv{Hkv} D{D} bf16->fp32+lse",
        "value": round(sum(fl) / (total_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
        "ms_per_block": round(total_ms, 3), "reps": reps,
        "layer_ms": [round(t, 4) for t in per_layer],
        "swa_layer_ms": round(swa_ms, 4), "global_layer_ms": round(ga_ms, 4),
        "attention_flop_reduction_vs_all_global": round(flop_ratio, 3),
        "kv_cache_reduction_vs_all_global": round(kv_ratio, 3),
        "roofline": roof, "clocks": clocks,
    }
    if cpu:
        if cpu_rates is None:
            swa_s = cpu_oracle_sample(layers[0].q, layers[0].k, layers[0].v, layers[0].sink,
                                      c["W"], target_s=3.0)
            ga_rate, ga_sample = cpu_global_layer(layers[-1], T)
            cpu_rates = (swa_s, ga_rate, ga_sample)
        swa_s, ga_rate, ga_sample = cpu_rates
        cpu_s = sum(f / (swa_s["value"] * 1e12) for f, W in zip(fl, Ws) if W < T) + \
            sum(f / ga_rate for f, W in zip(fl, Ws) if W >= T)
        line["cpu_baseline"] = {
            "value": sum(fl) / cpu_s / 1e12, "unit": "TFLOP/s", "cores": swa_s["cores"],
            "kind": "oracle", "extrapolated": True, "block_s": round(cpu_s, 1),
            "sample": f"window layers: {swa_s['sample']} (layer 0); {ga_sample}"}
    del layers
    torch.cuda.empty_cache()
    return line, cpu_rates


SPARSE = dict(T=32768, Hq=64, Hkv=8, D=128, QB=64, topk=16)


def _event_ms(fn, reps, stream):
    with torch.cuda.stream(stream):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


LONG = dict(B=1, T=262144, Hq=64, Hkv=8, D=128, W=128)


def long_context_line(swa, dev, stream, reps, peaks, cpu):
    """The long-context sliding-window prefill: one sequence of T=262144 with
    every 97th key scaled by 8 (peaky scores) and sinks U(-4, 4)."""
    c = LONG
    B, T, Hq, Hkv, D, W = (c[k] for k in ("B", "T", "Hq", "Hkv", "D", "W"))
    x = gen.prefill_inputs(B, T, Hq, Hkv, D, seed=5, device=dev, sink_dist="uniform4",
                           peaky_every=97)
    out = torch.empty(B, T, Hq, D, dtype=torch.float32, device=dev)
    lse = torch.empty(B, Hq, T, dtype=torch.float32, device=dev)
    ms, clocks = with_clocks(dev, lambda: _event_ms(
        lambda: swa.swa_sink_fwd(x.q, x.k, x.v, x.sink, W, out, lse, stream=stream),
        reps, stream))
    flops = work.prefill_flops(B, T, Hq, D, W)
    nbytes = work.prefill_bytes(B, T, Hq, Hkv, D, 2)
    hbm = float(peaks["hbm_gbs"])
    gbs = nbytes / (ms * 1e-3) / 1e9
    line = {
        "workload": f"swa_sink_prefill B{B} T{T} Hq{Hq} Hkv{Hkv} D{D} W{W} bf16->fp32+lse, every "
                    f"97th key x8, sinks U(-4,4)",
        "value": round(flops / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
        "ms_per_call": round(ms, 4),
        "roofline": {"kernel": "swa_fwd_tc_kernel", "bound": "hbm", "achieved": round(gbs, 1),
                     "peak": hbm, "unit": "GB/s", "frac": round(gbs / hbm, 4),
                     "bytes_per_launch": nbytes},
        "clocks": clocks,
    }
    if cpu:
        line["cpu_baseline"] = cpu_oracle_sample(x.q, x.k, x.v, x.sink, W, target_s=3.0,
                                                 i0=T // 2)
    del x, out, lse
    torch.cuda.empty_cache()
    return line


def high_sparse_line(swa, dev, stream, reps, peaks, cpu):
    """High Sparse on one sequence of T=32768: the global layer with and
    without its block scores, the selection, and the sparse layer over the
    selected blocks of the shared K/V."""
    c = SPARSE
    T, Hq, Hkv, D, QB, topk = (c[k] for k in ("T", "Hq", "Hkv", "D", "QB", "topk"))
    x = gen.prefill_inputs(1, T, Hq, Hkv, D, seed=500, device=dev)
    q2 = gen.prefill_inputs(1, T, Hq, Hkv, D, seed=501, device=dev).q
    state = {}

    def glb():
        swa.swa_sink_fwd(x.q, x.k, x.v, x.sink, T, stream=stream)

    def glb_scores():
        state["bm"] = swa.swa_sink_fwd_scores(x.q, x.k, x.v, x.sink, T, stream=stream)[2]

    def sparse():
        swa.swa_sink_sparse_fwd(q2, x.k, x.v, x.sink, state["idx"], QB, stream=stream)

    def timed():
        ms_g = _event_ms(glb, reps, stream)
        ms_gs = _event_ms(glb_scores, reps, stream)
        ms_sel = _event_ms(lambda: state.__setitem__(
            "idx", swa.swa_topk_blocks(state["bm"], T, QB, topk, stream=stream)), reps, stream)
        return ms_g, ms_gs, ms_sel

    # a first pass makes the selection; the timed pass measures the pipeline
    # in order (the sparse layer right after the global layers, under the
    # power cap they bring on), then the sparse layer alone after one second
    # of idle; each with the clocks of its own timed region
    timed()
    sparse()
    (ms_g, ms_gs, ms_sel), _ = with_clocks(dev, timed)
    ms_sp, clocks = with_clocks(dev, lambda: _event_ms(sparse, reps, stream))
    time.sleep(1.0)
    ms_sp_first, clocks_idle = with_clocks(dev, lambda: _event_ms(sparse, reps, stream))
    # algorithmic work of the sparse layer: keys j <= i of the selected blocks
    idx = state["idx"][0].cpu().numpy()              # [Hkv, nqb, topk]
    pairs = 0
    for g in range(Hkv):
        for qb in range(idx.shape[1]):
            for kb in idx[g, qb]:
                if kb < 0:
                    continue
                i0, i1 = qb * QB, min(qb * QB + QB, T)
                j0 = int(kb) * 128
                for i in range(i0, i1):
                    pairs += max(0, min(i, j0 + 127) - j0 + 1)
    sp_flops = 4 * D * (Hq // Hkv) * pairs
    gl_flops = work.prefill_flops(1, T, Hq, D, T)
    peak = float(peaks["bf16_tflops"])
    tf = sp_flops / (ms_sp * 1e-3) / 1e12
    tf_first = sp_flops / (ms_sp_first * 1e-3) / 1e12
    line = {
        "workload": f"High Sparse B1 T{T} Hq{Hq} Hkv{Hkv} D{D}: global layer + block scores, "
                    f"top-{topk} blocks per {QB}-position query block, sparse layer on the "
                    "shared K/V",
        "global_ms": round(ms_g, 3), "global_with_scores_ms": round(ms_gs, 3),
        "score_overhead": round(ms_gs / ms_g - 1.0, 4),
        "select_ms": round(ms_sel, 4),
        "sparse_ms": round(ms_sp_first, 3), "sparse_ms_in_pipeline": round(ms_sp, 3),
        "sparse_tflops": round(tf_first, 1),
        "sparse_fraction_of_global_flops": round(sp_flops / gl_flops, 4),
        # the layer timed alone (after one second of idle) against the burst
        # peak; timed inside the pipeline (right after ~100 ms of global
        # layers) against the sustained one
        "roofline": {"kernel": "swa_fwd_tc_global_kernel (sparse mode)", "bound": "tensor",
                     "achieved": round(tf_first, 1), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(tf_first / peak, 4),
                     "peak_source": "measured bf16_tflops (burst), the layer timed alone",
                     "traffic": recorded_traffic(
                         "swa_fwd_tc_global_kernel",
                         traffic_shape(B=1, T=T, Hq=Hq, Hkv=Hkv, D=D, QB=QB, topk=topk),
                         record="swa_fwd_tc_global_kernel.sparse")},
        "in_pipeline": {"achieved": round(tf, 1), "unit": "TFLOP/s",
                        "peak": float(peaks["bf16_tflops_sustained"]),
                        "frac_of_sustained": round(tf / float(peaks["bf16_tflops_sustained"]), 4),
                        "frac_of_burst": round(tf / peak, 4)},
        "clocks": clocks_idle, "clocks_in_pipeline": clocks,
    }
    if clocks.get("sm_mhz") and clocks.get("sm_max_mhz"):
        # time x clock: the in-pipeline rate had the layer run at the maximum
        # SM clock
        line["in_pipeline"]["frac_of_burst_at_max_clock"] = round(
            tf / peak * clocks["sm_max_mhz"] / clocks["sm_mhz"], 4)
    if cpu:
        import oracle
        # rows 0..Ts-1 of the sparse layer are its first query blocks exactly
        Ts = 3072
        nqb = Ts // QB
        hc = [t[:, :Ts].cpu() for t in (q2, x.k, x.v)]
        ic = state["idx"][:, :, :nqb].cpu()
        pairs_s = 0
        for g in range(Hkv):
            for qb in range(nqb):
                for kb in ic[0, g, qb].tolist():
                    if kb >= 0:
                        pairs_s += sum(max(0, min(i, 128 * kb + 127) - 128 * kb + 1)
                                       for i in range(qb * QB, qb * QB + QB))
        fl_s = 4 * D * (Hq // Hkv) * pairs_s
        line["cpu_baseline"] = cpu_oracle_call(
            lambda: oracle.sparse_fwd(hc[0], hc[1], hc[2], x.sink.cpu(), ic, QB), fl_s,
            "TFLOP/s", f"sparse layer rows 0..{Ts - 1}, all {Hq} heads ({fl_s:.3e} FLOP)")
    del x, q2, state
    torch.cuda.empty_cache()
    return line


def bf16_out_line(swa, x, c, steps, dev, stream, peaks, cpu_headline):
    """The headline prefill with bf16 output (out rounded from fp32, lse fp32)."""
    B, T, Hq, Hkv, D, W = (c[k] for k in ("B", "T", "Hq", "Hkv", "D", "W"))
    out = torch.empty(B, T, Hq, D, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(B, Hq, T, dtype=torch.float32, device=dev)

    def timed():
        with torch.cuda.stream(stream):
            for _ in range(3):
                swa.swa_sink_fwd(x.q, x.k, x.v, x.sink, W, out, lse, stream=stream)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(steps):
                swa.swa_sink_fwd(x.q, x.k, x.v, x.sink, W, out, lse, stream=stream)
            e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / steps

    ms, clocks = with_clocks(dev, timed)
    nbytes = work.prefill_bytes(B, T, Hq, Hkv, D, 2, out_bytes=2)
    flops = work.prefill_flops(B, T, Hq, D, W)
    hbm = float(peaks["hbm_gbs"])
    gbs = nbytes / (ms * 1e-3) / 1e9
    line = {"workload": workload_name(c).replace("fp32+lse", "bf16 out + fp32 lse"),
            "value": round(flops / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
            "ms_per_call": round(ms, 4),
            "roofline": {"kernel": "swa_fwd_tc_kernel", "bound": "hbm", "achieved": round(gbs, 1),
                         "peak": hbm, "unit": "GB/s", "frac": round(gbs / hbm, 4),
                         "bytes_per_launch": nbytes},
            "clocks": clocks}
    if cpu_headline is not None:
        # the oracle computes the same rows whatever the output type
        line["cpu_baseline"] = dict(cpu_headline, sample="the headline line's sample (the "
                                    "same rows; the output type does not change the oracle)")
    return line


# other group sizes and draft counts on the tensor-core kernels (same window,
# head dimension and sequence counts as the main workloads)
WIDE_PREFILL = {"g4": dict(B=4, T=8192, Hq=32, Hkv=8, D=128, W=128),
                "g16": dict(B=4, T=8192, Hq=64, Hkv=4, D=128, W=128),
                "d64": dict(B=4, T=8192, Hq=64, Hkv=8, D=64, W=128)}
WIDE_DECODE = {"g4": dict(B=256, Hq=32, Hkv=8, D=128, W=128),
               "g16": dict(B=256, Hq=64, Hkv=4, D=128, W=128),
               "d64": dict(B=256, Hq=64, Hkv=8, D=64, W=128)}
WIDE_VERIFY = {"l8": dict(B=256, L=8, Hq=64, Hkv=8, D=128, W=128)}
WIDE_GLOBAL = {"d64": dict(B=1, T=16384, Hq=64, Hkv=8, D=64, W=16384),
               "g4": dict(B=1, T=16384, Hq=32, Hkv=8, D=128, W=16384)}


def wide_prefill_line(swa, c, steps, dev, stream, peaks, cpu=False):
    """Sliding-window prefill of another group size: HBM roofline."""
    B, T, Hq, Hkv, D, W = (c[k] for k in ("B", "T", "Hq", "Hkv", "D", "W"))
    x = gen.prefill_inputs(B, T, Hq, Hkv, D, seed=7, device=dev)
    out = torch.empty(B, T, Hq, D, dtype=torch.float32, device=dev)
    lse = torch.empty(B, Hq, T, dtype=torch.float32, device=dev)
    ms, clocks = with_clocks(dev, lambda: _event_ms(
        lambda: swa.swa_sink_fwd(x.q, x.k, x.v, x.sink, W, out, lse, stream=stream),
        steps, stream))
    nbytes = work.prefill_bytes(B, T, Hq, Hkv, D, 2)
    hbm = float(peaks["hbm_gbs"])
    gbs = nbytes / (ms * 1e-3) / 1e9
    kpath = swa.fwd_path(B, T, Hq, Hkv, D, W)
    line = {"workload": workload_name(c), "value": round(gbs, 1), "unit": "GB/s",
            "ms_per_call": round(ms, 4),
            "roofline": {"kernel": KERNEL_OF_PATH.get(kpath, kpath), "bound": "hbm",
                         "achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s",
                         "frac": round(gbs / hbm, 4), "bytes_per_launch": nbytes},
            "sm_mhz": clocks.get("sm_mhz")}
    if cpu:
        # the oracle's rate in the line's unit: bytes of the sampled rows' share
        smp = cpu_oracle_sample(x.q, x.k, x.v, x.sink, W, target_s=1.5)
        line["cpu_baseline"] = dict(smp, value=smp["value"] * 1e12 / work.prefill_flops(
            B, T, Hq, D, W) * nbytes / 1e9, unit="GB/s")
    del x, out, lse
    torch.cuda.empty_cache()
    return line


def wide_global_line(swa, c, steps, dev, stream, peaks, cpu=False):
    """Global layer (W = T) of another head dimension: tensor roofline, the
    burst peak (the call is timed alone), with the sustained one beside it."""
    B, T, Hq, Hkv, D, W = (c[k] for k in ("B", "T", "Hq", "Hkv", "D", "W"))
    x = gen.prefill_inputs(B, T, Hq, Hkv, D, seed=7, device=dev)
    out = torch.empty(B, T, Hq, D, dtype=torch.float32, device=dev)
    lse = torch.empty(B, Hq, T, dtype=torch.float32, device=dev)
    ms, clocks = with_clocks(dev, lambda: _event_ms(
        lambda: swa.swa_sink_fwd(x.q, x.k, x.v, x.sink, W, out, lse, stream=stream),
        steps, stream))
    flops = work.prefill_flops(B, T, Hq, D, W)
    tf = flops / (ms * 1e-3) / 1e12
    burst = float(peaks["bf16_tflops"])
    sust = float(peaks.get("bf16_tflops_sustained") or burst)
    kpath = swa.fwd_path(B, T, Hq, Hkv, D, W)
    line = {"workload": workload_name(c), "value": round(tf, 1), "unit": "TFLOP/s",
            "ms_per_call": round(ms, 4),
            "roofline": {"kernel": KERNEL_OF_PATH.get(kpath, kpath), "bound": "tensor",
                         "achieved": round(tf, 1), "peak": burst, "unit": "TFLOP/s",
                         "frac": round(tf / burst, 4), "flops_per_launch": flops,
                         "frac_of_sustained": round(tf / sust, 4)},
            "sm_mhz": clocks.get("sm_mhz")}
    if cpu:
        import oracle
        rate, sample = cpu_global_layer(x, T)
        line["cpu_baseline"] = {"value": rate / 1e12, "unit": "TFLOP/s",
                                "cores": oracle.num_threads(), "kind": "oracle", "sample": sample}
    del x, out, lse
    torch.cuda.empty_cache()
    return line


def run_only(args):
    """A few eager calls of one workload, for a profiler (``--only prefill_g4``,
    ``--only sparse_main`` and so on); prints one JSON line with the mean time
    of the timed calls."""
    import hybrid_sliding_window_02_b300 as swa
    swa.lib()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(device=dev)
    kind, name = args.only.split("_", 1)
    if kind == "prefill":
        c = PREFILL if name == "main" else WIDE_PREFILL[name]
        B, T, Hq, Hkv, D, W = (c[k] for k in ("B", "T", "Hq", "Hkv", "D", "W"))
        x = gen.prefill_inputs(B, T, Hq, Hkv, D, seed=7, device=dev)
        call = lambda: swa.swa_sink_fwd(x.q, x.k, x.v, x.sink, W, stream=stream)
    elif kind == "global":
        c = WIDE_GLOBAL[name]
        B, T, Hq, Hkv, D, W = (c[k] for k in ("B", "T", "Hq", "Hkv", "D", "W"))
        x = gen.prefill_inputs(B, T, Hq, Hkv, D, seed=7, device=dev)
        call = lambda: swa.swa_sink_fwd(x.q, x.k, x.v, x.sink, W, stream=stream)
    elif kind == "sparse":
        # the High Sparse workload: one scored global layer and the selection
        # (launched once each, before the timed calls), then the sparse layer
        c = SPARSE
        T, Hq, Hkv, D, QB, topk = (c[k] for k in ("T", "Hq", "Hkv", "D", "QB", "topk"))
        x = gen.prefill_inputs(1, T, Hq, Hkv, D, seed=500, device=dev)
        q2 = gen.prefill_inputs(1, T, Hq, Hkv, D, seed=501, device=dev).q
        bm = swa.swa_sink_fwd_scores(x.q, x.k, x.v, x.sink, T, stream=stream)[2]
        idx = swa.swa_topk_blocks(bm, T, QB, topk, stream=stream)
        call = lambda: swa.swa_sink_sparse_fwd(q2, x.k, x.v, x.sink, idx, QB, stream=stream)
    elif kind == "rope":
        # RoPE in place of the headline prefill's q and k (two launches)
        c = PREFILL
        B, T, Hq, Hkv, D = (c[k] for k in ("B", "T", "Hq", "Hkv", "D"))
        x = gen.prefill_inputs(B, T, Hq, Hkv, D, seed=7, device=dev)
        pos0 = torch.zeros(B, dtype=torch.int64, device=dev)

        def call():
            swa.swa_rope(x.q, pos0, D, 10000.0, stream=stream)
            swa.swa_rope(x.k, pos0, D, 10000.0, stream=stream)
    elif kind == "step":
        # one decode step: rotate the new token's q and k, append k and v, decode
        c = DECODE
        B, Hq, Hkv, D, W = (c[k] for k in ("B", "Hq", "Hkv", "D", "W"))
        d = gen.decode_inputs(B, Hq, Hkv, D, W, seed=100, device=dev)
        g = torch.Generator(device=dev).manual_seed(400)
        kn = torch.randn(B, Hkv, D, generator=g, device=dev).to(torch.bfloat16)
        vn = torch.randn(B, Hkv, D, generator=g, device=dev).to(torch.bfloat16)
        qo = torch.empty_like(d.q)

        def call():
            swa.swa_rope_append(d.q, kn, vn, d.k_ring, d.v_ring, d.pos, D, 10000.0, q_out=qo,
                                stream=stream)
            swa.swa_sink_decode(qo, d.k_ring, d.v_ring, d.pos, d.sink, stream=stream)
    elif kind == "decode":
        c = DECODE if name == "main" else WIDE_DECODE[name]
        d = gen.decode_inputs(*(c[k] for k in ("B", "Hq", "Hkv", "D", "W")), seed=100, device=dev)
        call = lambda: swa.swa_sink_decode(d.q, d.k_ring, d.v_ring, d.pos, d.sink, stream=stream)
    else:
        c = VERIFY if name == "main" else WIDE_VERIFY[name]
        v = gen.verify_inputs(*(c[k] for k in ("B", "L", "Hq", "Hkv", "D", "W")), seed=300,
                              device=dev)
        call = lambda: swa.swa_sink_verify(v.q, v.k_new, v.v_new, v.k_ring, v.v_ring, v.pos,
                                           v.sink, stream=stream)
    ms = _event_ms(call, args.steps, stream)
    return {"only": args.only, "workload": c, "ms_per_call": round(ms, 4)}


def time_e2e(swa, xh, c, steps, dev, stream):
    """Host (pinned) inputs -> device -> prefill -> host outputs, every step,
    through the library's host-buffer call (swa_sink_fwd_host: per chunk of
    positions, the copies in, the prefill and the copies out, with neighbouring
    chunks' copies overlapping).  The sink is a resident layer parameter."""
    B, T, Hq, Hkv, D, W = (c[k] for k in ("B", "T", "Hq", "Hkv", "D", "W"))
    sink_d = xh.sink.to(dev)
    out_h = torch.empty(B, T, Hq, D, dtype=torch.float32, pin_memory=True)
    lse_h = torch.empty(B, Hq, T, dtype=torch.float32, pin_memory=True)
    state = {"work": None}

    def step():
        _, _, state["work"] = swa.swa_sink_fwd_host(xh.q, xh.k, xh.v, sink_d, W, out_h, lse_h,
                                                    work=state["work"], stream=stream)

    step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    h2d = sum(t.numel() * t.element_size() for t in (xh.q, xh.k, xh.v))
    d2h = out_h.numel() * 4 + lse_h.numel() * 4
    del state
    return e0.elapsed_time(e1) / steps, h2d, d2h


KERNEL_OF_PATH = {"tc_swa": "swa_fwd_tc_kernel", "tc_global": "swa_fwd_tc_global_kernel",
                  "simt": "simt_fwd_kernel"}


def prefill_roofline(kpath, flops, nbytes, launch_ms, peaks, peak_src, shape=""):
    """Roofline of the prefill kernel: HBM-bound for the sliding window (fp32
    output dominates the bytes), tensor-bound for the global layer.  shape:
    the workload's sizes (traffic_shape), which select the traffic record."""
    kernel = KERNEL_OF_PATH.get(kpath, kpath)
    gbs = nbytes / (launch_ms * 1e-3) / 1e9
    tfs = flops / (launch_ms * 1e-3) / 1e12
    common = {"kernel": kernel, "launch_ms": round(launch_ms, 4),
              "algorithmic_bytes_per_launch": nbytes, "algorithmic_flops_per_launch": flops,
              "traffic": recorded_traffic(kernel, shape)}
    if kpath == "tc_global":
        peak = float(peaks["bf16_tflops"])
        return dict({"bound": "tensor", "achieved": round(tfs, 1), "peak": peak,
                     "unit": "TFLOP/s", "frac": round(tfs / peak, 4),
                     "peak_source": f"{peak_src} bf16_tflops (burst)",
                     "gbs": round(gbs, 1)}, **common)
    hbm = float(peaks["hbm_gbs"])
    return dict({"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s",
                 "frac": round(gbs / hbm, 4), "peak_source": f"{peak_src} hbm_gbs",
                 "tflops": round(tfs, 2),
                 "tensor_peak_frac": round(tfs / float(peaks["bf16_tflops"]), 4)}, **common)


def run_ours(args, dist):
    import hybrid_sliding_window_02_b300 as swa
    swa.lib()
    dev = torch.device("cuda", dist.local_rank)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(device=dev)
    c = dict(PREFILL, B=args.prefill[0], T=args.prefill[1])
    if args.window:
        c["W"] = args.window
    kpath = swa.fwd_path(c["B"], c["T"], c["Hq"], c["Hkv"], c["D"], c["W"])
    x = gen.prefill_inputs(c["B"], c["T"], c["Hq"], c["Hkv"], c["D"], seed=0, device=dev)
    flops = work.prefill_flops(c["B"], c["T"], c["Hq"], c["D"], c["W"])
    nbytes = work.prefill_bytes(c["B"], c["T"], c["Hq"], c["Hkv"], c["D"], 2)
    peaks, peak_src = load_peaks()
    hbm = float(peaks["hbm_gbs"])
    cpu = dist.rank == 0 and not args.no_cpu

    with ClockSampler(dev.index) as clk:
        total_ms, launch_ms = time_prefill(swa, x, c, args.steps, args.warmup, dist, stream)
    rate, total_ms = job_rate(dist, flops * args.steps, total_ms)
    ms_per_step = total_ms / args.steps
    value = rate / 1e12

    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s",
        "n_gpus": dist.world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": workload_name(c), "seed": 0,
                   "l2": f"inputs larger than L2 ({nbytes / 1e6:.0f} MB moved per step)",
                   "parallelism": f"replicas x{dist.world}"},
        "roofline": prefill_roofline(kpath, flops, nbytes, launch_ms, peaks, peak_src,
                                     traffic_shape(**{k: c[k] for k in ("B", "T", "Hq", "Hkv",
                                                                         "D", "W")})),
        "gpu_launches": args.steps,
        "clocks": clk.summary(),
    }
    if not args.no_e2e:
        xh = gen.PrefillInputs(*(t.cpu().pin_memory() for t in (x.q, x.k, x.v, x.sink)))
        e2e_ms, h2d, d2h = time_e2e(swa, xh, c, max(3, args.steps // 50), dev, stream)
        e2e_rate, e2e_ms = job_rate(dist, flops, e2e_ms)
        line["e2e"] = {"value": round(e2e_rate / 1e12, 3),
                       "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                       "ms_per_step": round(e2e_ms, 3)}
        del xh
    if cpu:
        line["cpu_baseline"] = cpu_oracle_sample(x.q, x.k, x.v, x.sink, c["W"],
                                                 target_s=args.cpu_seconds)
    # the other workloads; decode and verify come last so that they stay in
    # the tail of the line when only its end is kept
    line["prefill_bf16_out"] = bf16_out_line(swa, x, c, max(10, args.steps // 4), dev, stream,
                                             peaks, line.get("cpu_baseline"))
    if not args.no_hybrid:
        line["hybrid_block"], rates = hybrid_line(swa, dev, stream, args.hybrid_reps, peaks, cpu)
        # the 7:1 schedule of the later models: same kernels, seven window
        # layers per global layer (same per-layer CPU rates)
        line["hybrid_block_7to1"], _ = hybrid_line(swa, dev, stream, args.hybrid_reps, peaks,
                                                   cpu, n_swa=7, cpu_rates=rates)
        line["high_sparse"] = high_sparse_line(swa, dev, stream, args.hybrid_reps, peaks, cpu)
        line["long_context"] = long_context_line(swa, dev, stream, args.hybrid_reps, peaks, cpu)
    if not args.no_wide:
        wide = {}
        for name, wc in WIDE_PREFILL.items():
            wide["prefill_" + name] = wide_prefill_line(swa, wc, max(20, args.steps // 20), dev,
                                                        stream, peaks, cpu)
        for name, wc in WIDE_GLOBAL.items():
            wide["global_" + name] = wide_global_line(swa, wc, 5, dev, stream, peaks, cpu)
        for name, wc in WIDE_DECODE.items():
            d = decode_line(swa, dev, stream, args.decode_steps, hbm, cpu, c=wc)
            wide["decode_" + name] = {k: d[k] for k in ("workload", "value", "unit", "roofline",
                                                        "cpu_baseline") if k in d}
        for name, wc in WIDE_VERIFY.items():
            d = verify_line(swa, dev, stream, args.decode_steps, hbm, cpu, c=wc)
            wide["verify_" + name] = {k: d[k] for k in ("workload", "value", "unit", "roofline",
                                                        "cpu_baseline") if k in d}
        line["other_shapes"] = wide
    line["rope"] = rope_line(swa, dev, stream, max(20, args.steps // 20), hbm, cpu)
    line["decode_step"] = decode_step_line(swa, dev, stream, args.decode_steps, hbm, cpu)
    line["verify"] = verify_line(swa, dev, stream, args.decode_steps, hbm, cpu)
    line["decode"] = decode_line(swa, dev, stream, args.decode_steps, hbm, cpu)
    if swa.device_error() != 0:
        line["device_error"] = True
    return line


def run_reference(args, dist):
    """The fp64 CPU oracle, timed on the host cores, on bounded samples."""
    if dist.rank != 0:
        return None
    c = PREFILL
    # same recipe as the GPU arm's workload: one of its sequences
    x = gen.prefill_inputs(1, c["T"], c["Hq"], c["Hkv"], c["D"], seed=0)
    import oracle
    oracle.build()
    nthr = oracle.num_threads()
    # full-window rows per step, sized from a first timed sample so that the
    # whole run (warm-up and timed steps) takes about 90 s of host work, at
    # most 2 s a step
    i0 = c["W"]
    dt0, _, _ = oracle_rows_rate(x.q, x.k, x.v, x.sink, c["W"], i0, 64)
    target = min(2.0, max(0.02, 90.0 / max(1, args.steps + args.warmup)))
    ts = max(16, min(c["T"] - i0, int(target * 64 / max(dt0, 1e-6))))
    for s in range(args.warmup):
        oracle_rows_rate(x.q, x.k, x.v, x.sink, c["W"], i0, ts)
    tot, flops = 0.0, 0
    for s in range(args.steps):
        dt, f, _ = oracle_rows_rate(x.q, x.k, x.v, x.sink, c["W"], i0, ts)
        tot += dt
        flops = f
    dt = tot / args.steps
    value = flops / dt / 1e12
    sample = (f"per step: one sequence of the workload, positions {i0}..{i0 + ts - 1}, "
              f"all {c['Hq']} heads "
              f"({flops:.3e} FLOP)")
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": dist.world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_name(c), "seed": 0, "parallelism": "host cores"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": nthr, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--decode-steps", type=int, default=2000)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer measurement")
    ap.add_argument("--no-hybrid", action="store_true", help="skip the 5:1 hybrid-block line")
    ap.add_argument("--no-wide", action="store_true",
                    help="skip the lines of other group sizes and draft counts")
    ap.add_argument("--only", default="",
                    choices=[""] + [f"{k}_main" for k in ("prefill", "decode", "verify", "sparse", "rope",
                                                          "step")] +
                    [f"prefill_{n}" for n in WIDE_PREFILL] + [f"global_{n}" for n in WIDE_GLOBAL] +
                    [f"decode_{n}" for n in WIDE_DECODE] + [f"verify_{n}" for n in WIDE_VERIFY],
                    help="run only a few calls of one workload (for a profiler)")
    ap.add_argument("--hybrid-reps", type=int, default=5)
    ap.add_argument("--window", type=int, default=0,
                    help="window of the timed prefill (default 128; W >= T is a global layer); "
                         "for profiling other cases")
    ap.add_argument("--prefill", type=int, nargs=2, metavar=("B", "T"),
                    default=(PREFILL["B"], PREFILL["T"]),
                    help="prefill batch and length (default: the headline workload); other "
                         "values are for profiling small cases")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.only:
        print(json.dumps(run_only(args)), flush=True)
        return
    dist = Dist()
    try:
        line = run_reference(args, dist) if args.impl == "reference" else run_ours(args, dist)
        if dist.rank == 0 and line is not None:
            print(json.dumps(line), flush=True)
    finally:
        dist.close()


if __name__ == "__main__":
    main()
