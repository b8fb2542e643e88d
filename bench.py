#!/usr/bin/env python
"""Benchmark of the fused deinterleave + clamped SwiGLU + NVFP4 quantize step.

One step = one call of moe_swiglu_nvfp4_quantize (one kernel launch) over the
MoE decode/routing workload: 4096 tokens x top-8 of 256 experts = 32768 rows
in per-expert segments (device offsets), I = 2048, BF16 gate/up ~ N(0, 1.5^2),
L = 7. Inputs (306 MB) are larger than L2 (129 MB), and two input copies
alternate between steps. Metric: algorithmic GB/s (BF16 read + FP4 + scale
written) and rows/s; the roofline is HBM bandwidth.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints ONE JSON line on rank 0. Under torchrun (N > 1) every rank runs its own
copy of the workload (weak scaling, no data-path collective); the only
collectives are the barrier around the timed region and the max over ranks of
its duration.

--impl reference times the CPU oracle (test infrastructure, single-threaded
C) on a bounded sample of the same workload on rank 0.
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
sys.path.insert(0, ROOT)

METRIC = "fused SwiGLU+NVFP4 quant GB/s (rows/s) and % of GB300 HBM peak, 1 GPU"
UNIT = "GB/s"
HEADLINE = "ragged"
L2_BYTES = 129 * 2 ** 20
FALLBACK_HBM_GBS = 6800.0


# ---------------------------------------------------------------------------
# distributed plumbing (host side; tested with gloo on CPU)
# ---------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(seconds: float, group=None) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return seconds
    dev = "cuda" if dist.get_backend(group) == "nccl" else "cpu"
    t = torch.tensor([seconds], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    return float(t.item())


def aggregate_throughput(bytes_per_step: int, rows_per_step: int, steps: int,
                         max_seconds: float, world: int) -> dict:
    """Whole-job throughput: every rank processed its own batch each step."""
    return {
        "gbs": world * bytes_per_step * steps / max_seconds / 1e9,
        "rows_per_s": world * rows_per_step * steps / max_seconds,
        "ms_per_step": max_seconds * 1e3 / steps,
    }


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# ---------------------------------------------------------------------------
# measurement helpers
# ---------------------------------------------------------------------------

def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def code_without_comments(text: str) -> str:
    """C/C++/CUDA source with its comments removed and every run of
    whitespace collapsed to one space; string and character literals are
    kept as written."""
    out, i, n = [], 0, len(text)
    while i < n:
        ch = text[i]
        if ch in "\"'":                                  # literal: copy through its closing quote
            j = i + 1
            while j < n and text[j] != ch:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
            out.append(" ")
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(ch)
            i += 1
    return " ".join("".join(out).split())


def kernel_source_hash() -> str:
    """Hash of the code (comments and layout ignored) of the sources the
    activation-step kernels are compiled from (the C header holds
    declarations only)."""
    h = hashlib.sha256()
    for rel in ("moe_swiglu_epilogue_gb300/csrc/moe_nvfp4.cu",
                "moe_swiglu_epilogue_gb300/csrc/nvfp4_device.cuh"):
        with open(os.path.join(ROOT, rel), encoding="utf-8") as fh:
            h.update(code_without_comments(fh.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source; None otherwise."""
    p = os.path.join(ROOT, "profiles", "ncu_dram_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as fh:
        rec = json.load(fh)
    for r in rec.get("records", []):
        if (r.get("kernel") == kernel and r.get("workload") == workload
                and r.get("source_hash") == kernel_source_hash()):
            return r.get("dram_bytes_per_launch")
    return None


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 100 ms."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu = gpu_id
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu=timestamp,{self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100", "-f", self.path],
                stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        with open(self.path) as fh:
            for line in fh:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                    rows.append((ts, float(parts[2]), float(parts[3]), parts[6:10]))
                except ValueError:
                    continue
        os.unlink(self.path)
        inside = [r for r in rows if t0 - 1.0 <= r[0] <= t1 + 1.0] or rows
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i, v in enumerate(r[3]) if v == "Active"})
        return {"sm_mhz": statistics.median(r[1] for r in inside),
                "sm_max_mhz": max(r[2] for r in inside), "reasons": reasons,
                "samples": len(inside)}


# ---------------------------------------------------------------------------
# our implementation
# ---------------------------------------------------------------------------

class DirectCall:
    """Pre-marshalled C-ABI call (the binding's work done once), so the host
    enqueues launches faster than the ~50 us kernels run."""

    def __init__(self, fn, args):
        self.fn = fn
        self.args = args

    def __call__(self):
        rc = self.fn(*self.args)
        if rc != 0:
            raise RuntimeError(f"C-ABI call failed with code {rc}")


def make_call(lib, w, src, packed, sf, off, stream):
    P = ctypes.c_void_p
    s = P(stream.cuda_stream)
    if w.kind == "quantize":
        return DirectCall(lib.moe_nvfp4_quantize,
                          (P(src.data_ptr()), w.rows, w.width, P(packed.data_ptr()),
                           P(sf.data_ptr()), s))
    E = 0 if off is None else off.shape[0] - 1
    return DirectCall(lib.moe_swiglu_nvfp4_quantize,
                      (P(src.data_ptr()), w.rows, w.width, ctypes.c_float(w.clamp_L),
                       P(0 if off is None else off.data_ptr()), ctypes.c_int32(E),
                       P(packed.data_ptr()), P(sf.data_ptr()), s))


def device_buffers(w, torch, copies: int):
    srcs = [torch.from_numpy(w.data.view(np.int16)).cuda() for _ in range(copies)]
    packed = torch.empty((w.rows, w.width // 2), dtype=torch.uint8, device="cuda")
    sf = torch.empty((w.rows, w.width // 16), dtype=torch.uint8, device="cuda")
    off = None if w.offsets is None else torch.from_numpy(w.offsets).cuda()
    return srcs, packed, sf, off


def time_steps(torch, calls, steps: int, warmup: int, stream, flush=None):
    """Warm up, then time exactly `steps` launches back to back on the
    launching stream: one event before, one after (barrier + synchronize on
    both sides). Each step is one launch, so the mean launch duration is the
    region's duration / steps. With `flush` (small inputs that fit in L2),
    each launch is timed on its own event pair after an L2 flush instead."""
    for i in range(warmup):
        calls[i % len(calls)]()
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    t_begin = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    per = []
    wall0 = time.time()
    if flush is None:
        t_begin.record(stream)
        for i in range(steps):
            calls[i % len(calls)]()
        t_end.record(stream)
        torch.cuda.synchronize()
    else:
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        t_begin.record(stream)
        for i in range(steps):
            flush()
            starts[i].record(stream)
            calls[i % len(calls)]()
            ends[i].record(stream)
        t_end.record(stream)
        torch.cuda.synchronize()
        per = [s.elapsed_time(e) / 1e3 for s, e in zip(starts, ends)]
    barrier()
    torch.cuda.synchronize()
    wall1 = time.time()
    total_s = t_begin.elapsed_time(t_end) / 1e3
    if not per:
        per = [total_s / steps] * steps
    return total_s, per, wall0, wall1


def run_workload(torch, lib, M, W, name: str, steps: int, warmup: int, stream, copies=2,
                 cold_small=False):
    w = W.make(name)
    srcs, packed, sf, off = device_buffers(w, torch, copies)
    calls = [make_call(lib, w, s, packed, sf, off, stream) for s in srcs]
    flush = None
    if cold_small:
        scratch = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device="cuda")
        flush = lambda: scratch.fill_(1)       # evict the small input from L2
    with torch.cuda.stream(stream):
        total_s, per, w0, w1 = time_steps(torch, calls, steps, warmup, stream, flush)
    return w, total_s, per, w0, w1, (srcs, packed, sf, off, calls)


def launch_percentiles(torch, calls, n: int, stream):
    """Per-launch durations outside the timed region: each of n launches
    (inputs alternating as in the timed loop) between its own event pair;
    p10 / p50 / p90 in microseconds."""
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    with torch.cuda.stream(stream):
        for i in range(n):
            starts[i].record(stream)
            calls[i % len(calls)]()
            ends[i].record(stream)
    torch.cuda.synchronize()
    us = np.asarray([a.elapsed_time(b) * 1e3 for a, b in zip(starts, ends)])
    return [round(float(v), 2) for v in np.percentile(us, [10, 50, 90])]


def e2e_chunks(w, chunks: int):
    """Row ranges of the e2e pipeline. With expert offsets the chunks are
    groups of whole expert segments (each call gets its group's slice of
    the device offsets, so the ragged path runs end to end); otherwise
    equal row ranges. Returns [(row0, row1, expert0, expert1)]."""
    if w.offsets is None:
        b = np.linspace(0, w.rows, chunks + 1).astype(np.int64)
        return [(int(a), int(c), 0, 0) for a, c in zip(b[:-1], b[1:])]
    off = w.offsets.astype(np.int64)
    E = off.shape[0] - 1
    out, e0 = [], 0
    for k in range(1, chunks + 1):
        target = off[0] + (off[-1] - off[0]) * k // chunks
        e1 = E if k == chunks else int(np.searchsorted(off, target, side="left"))
        e1 = max(e1, e0)
        if e1 > e0:
            out.append((int(off[e0]), int(off[e1]), e0, e1))
        e0 = e1
    return out


def e2e_measure(torch, lib, w, stream, steps: int, chunks: int = 8):
    """Through the public C-ABI call with HOST buffers, pipelined the way a
    streaming caller would: the active rows are split into `chunks` ranges
    (whole expert segments when the workload has offsets); each is copied
    from pinned host memory on an upload stream, processed by one C-ABI call
    (with its slice of the device expert offsets) on the compute stream, and
    its outputs are read back on a download stream, so transfers in both
    directions overlap the kernels. Every step moves every active row's input
    and output; the timed region spans the first upload to the last
    download."""
    P = ctypes.c_void_p
    h_in = torch.from_numpy(w.data.view(np.int16)).pin_memory()
    h_packed = torch.empty((w.rows, w.width // 2), dtype=torch.uint8).pin_memory()
    h_sf = torch.empty((w.rows, w.width // 16), dtype=torch.uint8).pin_memory()
    d_in = torch.empty_like(h_in, device="cuda")
    d_packed = torch.empty_like(h_packed, device="cuda")
    d_sf = torch.empty_like(h_sf, device="cuda")
    d_off = None if w.offsets is None else torch.from_numpy(w.offsets).cuda()
    parts = e2e_chunks(w, chunks)
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    in_w = 2 * w.width if w.kind == "fused" else w.width          # BF16 values per input row
    calls = []
    for a, b, e0, e1 in parts:
        if w.kind == "quantize":
            calls.append(DirectCall(lib.moe_nvfp4_quantize,
                                    (P(d_in.data_ptr() + a * in_w * 2), b - a, w.width,
                                     P(d_packed.data_ptr() + a * (w.width // 2)),
                                     P(d_sf.data_ptr() + a * (w.width // 16)), P(stream.cuda_stream))))
        elif d_off is None:
            calls.append(DirectCall(lib.moe_swiglu_nvfp4_quantize,
                                    (P(d_in.data_ptr() + a * in_w * 2), b - a, w.width, ctypes.c_float(w.clamp_L),
                                     P(0), ctypes.c_int32(0), P(d_packed.data_ptr() + a * (w.width // 2)),
                                     P(d_sf.data_ptr() + a * (w.width // 16)), P(stream.cuda_stream))))
        else:                                     # whole buffers, this group's offsets
            calls.append(DirectCall(lib.moe_swiglu_nvfp4_quantize,
                                    (P(d_in.data_ptr()), w.rows, w.width, ctypes.c_float(w.clamp_L),
                                     P(d_off.data_ptr() + 4 * e0), ctypes.c_int32(e1 - e0),
                                     P(d_packed.data_ptr()), P(d_sf.data_ptr()), P(stream.cuda_stream))))
    ev_in = [torch.cuda.Event() for _ in calls]
    ev_k = [torch.cuda.Event() for _ in calls]
    ev_out = [torch.cuda.Event() for _ in calls]

    def step(first: bool):
        for i, (a, b, _, _) in enumerate(parts):
            if not first:
                s_in.wait_event(ev_k[i])               # the previous step's kernel read this range
            with torch.cuda.stream(s_in):
                d_in[a:b].copy_(h_in[a:b], non_blocking=True)
                ev_in[i].record(s_in)
            stream.wait_event(ev_in[i])
            if not first:
                stream.wait_event(ev_out[i])           # the previous step's outputs were read back
            calls[i]()
            ev_k[i].record(stream)
            s_out.wait_event(ev_k[i])
            with torch.cuda.stream(s_out):
                h_packed[a:b].copy_(d_packed[a:b], non_blocking=True)
                h_sf[a:b].copy_(d_sf[a:b], non_blocking=True)
                ev_out[i].record(s_out)

    for k in range(2):
        step(k == 0)
    torch.cuda.synchronize()
    barrier()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    done = torch.cuda.Event()
    ev0.record(s_in)
    for _ in range(steps):
        step(False)
    done.record(s_out)
    s_in.wait_event(done)
    ev1.record(s_in)
    torch.cuda.synchronize()
    secs = ev0.elapsed_time(ev1) / 1e3
    rows = sum(b - a for a, b, _, _ in parts)
    h2d = rows * in_w * 2
    d2h = rows * (w.width // 2 + w.width // 16)
    return secs, h2d, d2h, len(parts)


def describe(w) -> str:
    if w.name == "ragged":
        return (f"ragged: {w.meta['tokens']} tokens x top-{w.meta['topk']} of "
                f"{w.meta['experts']} experts = {w.active_rows} rows in per-expert segments "
                f"(device offsets), I={w.width}, gate/up BF16 ~ N(0,1.5^2), L={w.clamp_L}")
    what = "quantize-only x" if w.kind == "quantize" else "fused gu"
    extra = "" if w.kind == "quantize" else f", L={w.clamp_L}"
    return f"{w.name}: {what} [{w.rows}, {w.width}]{extra}"


def cpu_baseline(w, budget_s: float = 12.0):
    """The oracle, as it stands (single-threaded C), on a bounded sample of
    the workload: whole active rows in order until ~budget_s of CPU work."""
    import oracle
    oracle.build()
    r0 = 0 if w.offsets is None else int(w.offsets[0])
    r1 = w.rows if w.offsets is None else int(w.offsets[-1])
    per_row = (2 * w.width if w.kind == "quantize" else 4 * w.width) + w.width // 2 + w.width // 16
    t = time.perf_counter()
    probe = w.data[r0:r0 + 64]
    if w.kind == "quantize":
        oracle.quantize_nvfp4(probe)
    else:
        oracle.swiglu_quantize_nvfp4(probe, w.clamp_L)
    per_row_s = (time.perf_counter() - t) / 64
    n = int(min(r1 - r0, max(64, budget_s / max(per_row_s, 1e-9))))
    sample = w.data[r0:r0 + n]
    t = time.perf_counter()
    if w.kind == "quantize":
        oracle.quantize_nvfp4(sample)
    else:
        oracle.swiglu_quantize_nvfp4(sample, w.clamp_L)
    secs = time.perf_counter() - t
    return {"value": per_row * n / secs / 1e9, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{n} of {r1 - r0} active rows of the {w.name} workload "
                      f"(I={w.width}), one pass, {secs:.2f} s",
            "rows_per_s": n / secs}


def _oracle_rows_worker(job):
    """One row partition of the oracle run (a spawned process; the input is
    read from shared memory). Returns the seconds spent in the oracle."""
    shm_name, shape, kind, width, clamp_L, r0, r1 = job
    from multiprocessing import shared_memory
    sys.path.insert(0, ROOT)
    import oracle
    shm = shared_memory.SharedMemory(name=shm_name)
    try:
        data = np.ndarray(shape, dtype=np.uint16, buffer=shm.buf)
        rows = np.ascontiguousarray(data[r0:r1])
        t = time.perf_counter()
        if kind == "quantize":
            oracle.quantize_nvfp4(rows)
        else:
            oracle.swiglu_quantize_nvfp4(rows, clamp_L)
        return time.perf_counter() - t
    finally:
        shm.close()


def _oracle_warm(_):
    sys.path.insert(0, ROOT)
    import oracle
    oracle.build()
    return os.getpid()


def cpu_baseline_all_cores(w):
    """The same oracle over contiguous row partitions of every active row,
    one spawned process per host core (the input shared, not copied);
    wall time of the parallel region after the pool has started."""
    import multiprocessing as mp
    from multiprocessing import shared_memory
    import oracle
    oracle.build()
    cores = os.cpu_count() or 1
    r0 = 0 if w.offsets is None else int(w.offsets[0])
    r1 = w.rows if w.offsets is None else int(w.offsets[-1])
    per_row = (2 * w.width if w.kind == "quantize" else 4 * w.width) + w.width // 2 + w.width // 16
    shm = shared_memory.SharedMemory(create=True, size=w.data.nbytes)
    try:
        np.ndarray(w.data.shape, dtype=np.uint16, buffer=shm.buf)[...] = w.data
        bounds = np.linspace(r0, r1, cores + 1).astype(np.int64)
        jobs = [(shm.name, w.data.shape, w.kind, w.width, w.clamp_L, int(a), int(b))
                for a, b in zip(bounds[:-1], bounds[1:]) if b > a]
        with mp.get_context("spawn").Pool(len(jobs)) as pool:
            pool.map(_oracle_warm, range(len(jobs)))
            t = time.perf_counter()
            pool.map(_oracle_rows_worker, jobs)
            secs = time.perf_counter() - t
    finally:
        shm.close()
        shm.unlink()
    return {"value": per_row * (r1 - r0) / secs / 1e9, "unit": UNIT, "cores": len(jobs), "kind": "oracle",
            "sample": f"all {r1 - r0} active rows of the {w.name} workload (I={w.width}) over "
                      f"{len(jobs)} processes, {secs:.2f} s wall",
            "rows_per_s": (r1 - r0) / secs}


class L2Flush:
    """Evicts the L2 before a cold launch. "read" sweeps a buffer of twice
    the L2 with the library's read-only kernel, leaving clean lines (nothing
    to write back when the next kernel misses); "fill" writes the buffer
    with torch's fill_, leaving the L2 full of dirty lines that the next
    kernel's misses must write back first (what an application that just
    wrote other data would see)."""

    def __init__(self, torch, lib, stream):
        P = ctypes.c_void_p
        self.buf = torch.ones(2 * L2_BYTES, dtype=torch.uint8, device="cuda")
        self.sink = torch.zeros(4, dtype=torch.uint8, device="cuda")
        self.read = DirectCall(lib.moe_nvfp4_traffic_floor,
                               (P(self.buf.data_ptr()), 2 * L2_BYTES // 32, 16, 3, P(self.sink.data_ptr()),
                                P(0), P(stream.cuda_stream)))
        self.fill = lambda: self.buf.fill_(1)


def cold_launches(torch, stream, calls: dict, flush, n: int) -> dict:
    """Each call in `calls` launched n times, each launch after `flush` and
    between its own event pair on the launching stream; the calls take turns
    so that drift affects them alike. Returns seconds per launch by name."""
    ev = {k: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(n)] for k in calls}
    with torch.cuda.stream(stream):
        for i in range(n):
            for k, c in calls.items():
                flush()
                ev[k][i][0].record(stream)
                c()
                ev[k][i][1].record(stream)
    torch.cuda.synchronize()
    return {k: [a.elapsed_time(b) / 1e3 for a, b in v] for k, v in ev.items()}


def small_config(torch, lib, W, name: str, stream, flush: L2Flush, peak: float, n: int = 60) -> dict:
    """A workload that fits in L2 (configs 1 and 2), as single cold launches:
    the median launch after a read flush, beside the two floors measured the
    same way in the same loop -- a launch that does nothing, and a kernel
    with the step's loads and stores and none of its arithmetic in the
    step's own launch shape -- and the median after a fill flush. Then the
    hot-L2 graph of 100 launches (the input resident in L2; not HBM)."""
    P = ctypes.c_void_p
    w = W.make(name)
    srcs, packed, sf, off = device_buffers(w, torch, 1)
    s = P(stream.cuda_stream)
    call = make_call(lib, w, srcs[0], packed, sf, off, stream)
    packed2, sf2 = torch.empty_like(packed), torch.empty_like(sf)
    kind = 0 if w.kind == "fused" else 1
    copy = DirectCall(lib.moe_nvfp4_traffic_floor, (P(srcs[0].data_ptr()), w.rows, w.width, kind,
                                                    P(packed2.data_ptr()), P(sf2.data_ptr()), s))
    empty = DirectCall(lib.moe_nvfp4_traffic_floor, (P(0), 0, 0, 2, P(0), P(0), s))
    with torch.cuda.stream(stream):
        for _ in range(5):
            call(), copy(), empty(), flush.read()
    torch.cuda.synchronize()
    t = cold_launches(torch, stream, {"step": call, "copy": copy, "empty": empty}, flush.read, n)
    t_fill = cold_launches(torch, stream, {"step": call}, flush.fill, n)["step"]
    med = {k: statistics.median(v) for k, v in t.items()}
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(100):
            call()
    with torch.cuda.stream(stream):
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(10):
            g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
    nbytes = w.algorithmic_bytes()
    return {"cold_us": round(med["step"] * 1e6, 2), "floor_copy_us": round(med["copy"] * 1e6, 2),
            "floor_empty_us": round(med["empty"] * 1e6, 2),
            "vs_copy_floor": round(med["step"] / med["copy"], 3),
            "gbs": round(nbytes / med["step"] / 1e9, 1), "frac": round(nbytes / med["step"] / 1e9 / peak, 4),
            "cold_us_fill_flush": round(statistics.median(t_fill) * 1e6, 2),
            "hot_graph_us": round(e0.elapsed_time(e1) * 1e3 / 1000, 2)}


def traffic_floor_us(torch, lib, w, srcs, stream, steps: int) -> float:
    """Back-to-back mean launch time of the step's loads and stores without
    its arithmetic, in its launch shape, over the same alternating inputs
    (rows of the workload's active range; the offsets only bound it)."""
    P = ctypes.c_void_p
    r0 = 0 if w.offsets is None else int(w.offsets[0])
    rows = w.active_rows
    in_w = 2 * w.width if w.kind == "fused" else w.width
    kind = 0 if w.kind == "fused" else 1
    packed = torch.empty((rows, w.width // 2), dtype=torch.uint8, device="cuda")
    sf = torch.empty((rows, w.width // 16), dtype=torch.uint8, device="cuda")
    calls = [DirectCall(lib.moe_nvfp4_traffic_floor,
                        (P(x.data_ptr() + r0 * in_w * 2), rows, w.width, kind, P(packed.data_ptr()),
                         P(sf.data_ptr()), P(stream.cuda_stream))) for x in srcs]
    with torch.cuda.stream(stream):
        _, per, _, _ = time_steps(torch, calls, steps, 5, stream)
    return statistics.fmean(per)


def large_config(torch, lib, M, W, name: str, steps: int, warmup: int, stream, peak: float,
                 timed=None) -> dict:
    """A workload larger than L2, back to back (two input copies
    alternating): mean launch, the isolated per-launch median, and the
    traffic floor. `timed` reuses the headline's timed region."""
    if timed is None:
        timed = run_workload(torch, lib, M, W, name, steps, warmup, stream)
    w, total_s, per, _, _, keep = timed
    srcs, calls = keep[0], keep[4]
    p50 = launch_percentiles(torch, calls, 50, stream)[1] * 1e-6
    floor = traffic_floor_us(torch, lib, w, srcs, stream, min(steps, 200))
    mean_s = statistics.fmean(per)
    nbytes = w.algorithmic_bytes()
    return {"us": round(mean_s * 1e6, 2), "gbs": round(nbytes / mean_s / 1e9, 1),
            "frac": round(nbytes / mean_s / 1e9 / peak, 4), "p50_us": round(p50 * 1e6, 2),
            "p50_frac": round(nbytes / p50 / 1e9 / peak, 4), "floor_us": round(floor * 1e6, 2)}


def reevaluation_rates(torch, lib, W, name: str) -> dict:
    """How often the fused kernel's exact path ran on a workload (the counted
    variant, one launch): scale decisions per block, nibble decisions per
    element."""
    P = ctypes.c_void_p
    w = W.make(name)
    x = torch.from_numpy(w.data.view(np.int16)).cuda()
    packed = torch.empty((w.rows, w.width // 2), dtype=torch.uint8, device="cuda")
    sf = torch.empty((w.rows, w.width // 16), dtype=torch.uint8, device="cuda")
    cnt = torch.zeros(3, dtype=torch.int64, device="cuda")
    off = None if w.offsets is None else torch.from_numpy(w.offsets).cuda()
    rc = lib.moe_swiglu_nvfp4_quantize_counted(P(x.data_ptr()), w.rows, w.width, ctypes.c_float(w.clamp_L),
                                               P(0 if off is None else off.data_ptr()),
                                               0 if off is None else off.shape[0] - 1, P(packed.data_ptr()),
                                               P(sf.data_ptr()), P(cnt.data_ptr()),
                                               P(torch.cuda.current_stream().cuda_stream))
    assert rc == 0
    torch.cuda.synchronize()
    blocks, scales, nibbles = (int(v) for v in cnt.cpu())
    return {"scale_reeval_per_block": float(f"{scales / max(blocks, 1):.3g}"),
            "nibble_reeval_per_elem": float(f"{nibbles / max(16 * blocks, 1):.3g}")}


NOMINAL_HBM_GBS = 8000.0          # the "about 8 TB/s" GB300 HBM3e figure the target is stated against


def roofline(bytes_per_launch: int, per_launch_s, peak_gbs: float, peak_src: str, traffic):
    mean_s = statistics.fmean(per_launch_s)
    achieved = bytes_per_launch / mean_s / 1e9
    return {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak_gbs, "unit": "GB/s",
            "frac": round(achieved / peak_gbs, 4), "traffic": traffic,
            "peak_source": f"{peak_src} hbm_gbs (burst copy)",
            "frac_of_8tbs": round(achieved / NOMINAL_HBM_GBS, 4),
            "launch_us_mean": round(mean_s * 1e6, 2)}


EXTENSION_CASES = ("two_level_scale", "bf16_compat", "bf16_compat_scaled", "padded_segments", "compact_writer",
                   "dequantize")


def extension_measurements(torch, lib, M, W, stream, steps: int, warmup: int, peak: float,
                           only=None):
    """Launch time and algorithmic GB/s of the extensions on the ragged
    workload (dequantization on the prefill quantize-only outputs): the
    two-level scale, the BF16-compat mode (global scale 1 and 1.25), padded
    per-expert output (segments padded to 128 rows), the compact BF16 writer,
    the compact flow (writer + quantize-only of its output, the pages'
    planned pipeline) and dequantization. `only`: a subset of
    EXTENSION_CASES, measured alone."""
    P = ctypes.c_void_p
    FO = M.FusedOptions
    w = W.make("ragged")
    rows, I, L = w.rows, w.width, w.clamp_L
    s = P(stream.cuda_stream)
    srcs = [torch.from_numpy(w.data.view(np.int16)).cuda() for _ in range(2)]
    off = torch.from_numpy(w.offsets).cuda()
    E = off.shape[0] - 1
    packed = torch.empty((rows, I // 2), dtype=torch.uint8, device="cuda")
    sf = torch.empty((rows, I // 16), dtype=torch.uint8, device="cuda")
    # two compact tensors (the writer alternates between them), so that the
    # quantize-only leg reads one that is not left in L2 by the previous step
    compacts = [torch.empty((rows, I), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    counts = np.diff(w.offsets)
    out_off = np.concatenate([[0], np.cumsum(np.ceil(counts / 128).astype(np.int64) * 128)])
    out_rows = int(out_off[-1])
    out_off_t = torch.from_numpy(out_off.astype(np.int32)).cuda()
    packed_p = torch.empty((out_rows, I // 2), dtype=torch.uint8, device="cuda")
    sf_p = torch.empty((out_rows, I // 16), dtype=torch.uint8, device="cuda")
    opts = {
        "two_level_scale": FO(1.25, 0, None, rows),
        "bf16_compat": FO(1.0, 1, None, rows),
        "bf16_compat_scaled": FO(1.25, 1, None, rows),
        "padded_segments": FO(1.0, 0, out_off_t.data_ptr(), out_rows),
    }
    fused_bytes = w.algorithmic_bytes()
    writer_bytes = w.active_rows * (4 * I + 2 * I)
    quant_bytes = rows * (2 * I + I // 2 + I // 16)
    res = {}

    def measure(name, calls, nbytes, note):
        with torch.cuda.stream(stream):
            tot, per, _, _ = time_steps(torch, calls, steps, warmup, stream)
        mean_s = statistics.fmean(per)
        res[name] = {"launch_us_mean": round(mean_s * 1e6, 2),
                     "gbs": round(nbytes / mean_s / 1e9, 1),
                     "frac_of_peak": round(nbytes / mean_s / 1e9 / peak, 4), "bytes": nbytes,
                     "what": note}

    def want(name):
        return only is None or name in only

    for name, opt in opts.items():
        if not want(name):
            continue
        pk, sc = (packed_p, sf_p) if name == "padded_segments" else (packed, sf)
        calls = [DirectCall(lib.moe_swiglu_nvfp4_quantize_ex,
                            (P(x.data_ptr()), rows, I, ctypes.c_float(L), P(off.data_ptr()),
                             ctypes.c_int32(E), ctypes.byref(opt), P(pk.data_ptr()),
                             P(sc.data_ptr()), s)) for x in srcs]
        measure(name, calls, fused_bytes, "moe_swiglu_nvfp4_quantize_ex on the ragged workload")
    writer = [DirectCall(lib.moe_swiglu_bf16, (P(x.data_ptr()), rows, I, ctypes.c_float(L),
                                               P(off.data_ptr()), ctypes.c_int32(E),
                                               P(c.data_ptr()), s)) for x, c in zip(srcs, compacts)]
    if want("compact_writer"):
        measure("compact_writer", writer, writer_bytes, "moe_swiglu_bf16: gate/up -> BF16 [rows, I]")
    if only is not None and not want("dequantize"):
        return res
    if only is None:                                       # the compact flow: full runs only
        quants = [DirectCall(lib.moe_nvfp4_quantize, (P(c.data_ptr()), rows, I,
                                                      P(packed.data_ptr()), P(sf.data_ptr()), s))
                  for c in compacts]
        measure("quantize_of_compact", quants, quant_bytes,
                "moe_nvfp4_quantize of the BF16 tensor (two tensors, alternating)")

        class Both:
            def __init__(self, a, b):
                self.a, self.b = a, b

            def __call__(self):
                self.a()
                self.b()

        measure("compact_flow", [Both(c, q) for c, q in zip(writer, quants)], writer_bytes + quant_bytes,
                "compact writer + quantize-only of its output per step (bytes: both kernels)")
        res["compact_flow"]["vs_fused_time"] = None
    del srcs, compacts
    torch.cuda.empty_cache()
    if not want("dequantize"):
        return res
    wq = W.make("prefill_quantize")
    x = torch.from_numpy(wq.data.view(np.int16)).cuda()
    # two copies of the NVFP4 input, alternating between steps
    pqs = [torch.empty((wq.rows, wq.width // 2), dtype=torch.uint8, device="cuda") for _ in range(2)]
    sqs = [torch.empty((wq.rows, wq.width // 16), dtype=torch.uint8, device="cuda") for _ in range(2)]
    for pq, sq in zip(pqs, sqs):
        rc = lib.moe_nvfp4_quantize_scaled(P(x.data_ptr()), wq.rows, wq.width, ctypes.c_float(1.5),
                                           P(pq.data_ptr()), P(sq.data_ptr()), s)
        assert rc == 0
    del x
    outq = torch.empty((wq.rows, wq.width), dtype=torch.bfloat16, device="cuda")
    dqs = [DirectCall(lib.moe_nvfp4_dequantize, (P(pq.data_ptr()), P(sq.data_ptr()), wq.rows, wq.width,
                                                 ctypes.c_float(1.5), P(outq.data_ptr()), s))
           for pq, sq in zip(pqs, sqs)]
    measure("dequantize", dqs, wq.rows * (wq.width // 2 + wq.width // 16 + 2 * wq.width),
            "moe_nvfp4_dequantize, global scale 1.5, [65536, 3072] (two inputs, alternating)")
    return res


GEMM_CASES = (("l1_gemm_decode", 256, 4096, 10), ("l1_gemm_prefill", 256, 32768, 5))


def gemm_measurements(torch, lib, M, W, stream, hbm_peak: float, cases=GEMM_CASES, warmup=3,
                      unfused=True):
    """The L1 GEMM with the step in its epilogue (BF16 operands, H = 7168,
    I = 2048, top-8 of 256 experts) on two row sets sharing one seeded weight
    tensor: 4096 tokens (32768 rows, ~128 per expert: the weights dominate
    the bytes, so HBM bounds it) and 32768 tokens (262144 rows, ~1024 per
    expert: the tensor cores bound it). Beside each, the unfused flow the
    pages' pipeline used: a cuBLAS batched BF16 GEMM over per-expert padded
    rows writing gu, then the fused activation kernel on gu."""
    P = ctypes.c_void_p
    s = P(stream.cuda_stream)
    H, I = 7168, 2048
    tflops_peak = None
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            tflops_peak = float(json.load(fh).get("bf16_tflops") or 0) or None
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    res = {}
    w1 = wq = ws = w1_experts = None
    for name, E, tokens, steps in cases:
        if w1_experts != E:
            w1 = wq = ws = None
            torch.cuda.empty_cache()
            w1_np = W.gemm_weights(E, H, I)
            w1 = torch.from_numpy(w1_np.view(np.int16)).cuda()
            w1_experts = E
            del w1_np
            # the same weights in NVFP4 (our quantize-only kernel writes the layout the GEMM reads)
            wq, ws = M.moe_nvfp4_quantize(w1.view(E * 2 * I, H), stream=stream)
            torch.cuda.synchronize()
        x_np, offsets = W.gemm_rows(tokens, E, 8, H)
        x = torch.from_numpy(x_np.view(np.int16)).cuda()
        off = torch.from_numpy(offsets).cuda()
        rows = x_np.shape[0]
        active_rows = int(offsets[-1]) - int(offsets[0])
        del x_np
        pk = torch.empty((rows, I // 2), dtype=torch.uint8, device="cuda")
        sc = torch.empty((rows, I // 16), dtype=torch.uint8, device="cuda")
        call = DirectCall(lib.moe_l1_gemm_swiglu_nvfp4,
                          (P(x.data_ptr()), P(w1.data_ptr()), rows, H, I, ctypes.c_float(7.0),
                           P(off.data_ptr()), ctypes.c_int32(E), P(pk.data_ptr()), P(sc.data_ptr()),
                           P(status.data_ptr()), s))
        with torch.cuda.stream(stream):
            _, per, _, _ = time_steps(torch, [call], steps, warmup, stream)
        fused_s = statistics.fmean(per)
        entry = {"rows": rows, "tokens": tokens, "H": H, "I": I, "experts": E}
        active_experts = int(np.count_nonzero(np.diff(offsets.astype(np.int64)) > 0))
        nbytes = active_rows * (2 * H + I // 2 + I // 16) + active_experts * 2 * I * H * 2
        flops = 2 * active_rows * H * 2 * I
        call4 = DirectCall(lib.moe_l1_gemm_w4_swiglu_nvfp4,
                           (P(x.data_ptr()), P(wq.data_ptr()), P(ws.data_ptr()), rows, H, I, ctypes.c_float(7.0),
                            P(off.data_ptr()), ctypes.c_int32(E), P(pk.data_ptr()), P(sc.data_ptr()),
                            P(status.data_ptr()), s))
        with torch.cuda.stream(stream):
            _, per4, _, _ = time_steps(torch, [call4], steps, warmup, stream)
        w4_s = statistics.fmean(per4)
        nbytes4 = active_rows * (2 * H + I // 2 + I // 16) + active_experts * 2 * I * (H // 2 + H // 16)
        entry["w4_nvfp4_weights"] = {
            "launch_us_mean": round(w4_s * 1e6, 1), "bytes": nbytes4,
            "gbs": round(nbytes4 / w4_s / 1e9, 1), "frac_of_hbm_peak": round(nbytes4 / w4_s / 1e9 / hbm_peak, 4),
            "tflops": round(flops / w4_s / 1e12, 1),
            "frac_of_bf16_peak": None if tflops_peak is None else round(flops / w4_s / 1e12 / tflops_peak, 4),
            "vs_bf16_weights_time": round(w4_s / fused_s, 3),
            "what": "moe_l1_gemm_w4_swiglu_nvfp4: the same weights quantized to NVFP4 (0.5625 B each)"}
        res[name] = entry
        entry.update({
            "launch_us_mean": round(fused_s * 1e6, 1),
            "gbs": round(nbytes / fused_s / 1e9, 1), "frac_of_hbm_peak": round(nbytes / fused_s / 1e9 / hbm_peak, 4),
            "tflops": round(flops / fused_s / 1e12, 1),
            "frac_of_bf16_peak": None if tflops_peak is None else round(flops / fused_s / 1e12 / tflops_peak, 4),
            "bytes": nbytes, "flops": flops,
            "bound": "hbm" if nbytes / hbm_peak > flops / 1e3 / (tflops_peak or 1e30) else "tensor",
            "what": "moe_l1_gemm_swiglu_nvfp4 (BF16 x, w1; NVFP4 out); peaks: measured hbm_gbs, bf16_tflops (burst)",
        })
        if not unfused:
            del x, pk, sc
            continue
        # the pages' two unfused flows with this GEMM: gu (2I BF16) then the
        # fused activation kernel; the compact SwiGLU (I BF16) then quantize-only
        gu_o = torch.empty((rows, 2 * I), dtype=torch.bfloat16, device="cuda")
        sw_o = torch.empty((rows, I), dtype=torch.bfloat16, device="cuda")
        gemm_gu = DirectCall(lib.moe_l1_gemm_bf16,
                             (P(x.data_ptr()), P(w1.data_ptr()), rows, H, I, ctypes.c_float(7.0),
                              P(off.data_ptr()), ctypes.c_int32(E), ctypes.c_int32(0), P(gu_o.data_ptr()),
                              P(status.data_ptr()), s))
        act = DirectCall(lib.moe_swiglu_nvfp4_quantize,
                         (P(gu_o.data_ptr()), rows, I, ctypes.c_float(7.0), P(off.data_ptr()),
                          ctypes.c_int32(E), P(pk.data_ptr()), P(sc.data_ptr()), s))
        gemm_sw = DirectCall(lib.moe_l1_gemm_bf16,
                             (P(x.data_ptr()), P(w1.data_ptr()), rows, H, I, ctypes.c_float(7.0),
                              P(off.data_ptr()), ctypes.c_int32(E), ctypes.c_int32(1), P(sw_o.data_ptr()),
                              P(status.data_ptr()), s))
        qnt = DirectCall(lib.moe_nvfp4_quantize,
                         (P(sw_o.data_ptr()), rows, I, P(pk.data_ptr()), P(sc.data_ptr()), s))

        class Pair:
            def __init__(self, a, b):
                self.a, self.b = a, b

            def __call__(self):
                self.a()
                self.b()
        with torch.cuda.stream(stream):
            _, per_g, _, _ = time_steps(torch, [Pair(gemm_gu, act)], steps, 2, stream)
            _, per_c, _, _ = time_steps(torch, [Pair(gemm_sw, qnt)], steps, 2, stream)
        entry["ours_gu_then_activation_us"] = round(statistics.fmean(per_g) * 1e6, 1)
        entry["ours_compact_then_quantize_us"] = round(statistics.fmean(per_c) * 1e6, 1)
        del gu_o, sw_o
        torch.cuda.empty_cache()
        # unfused: per-expert padded rows, cuBLAS batched GEMM to BF16 gu, then the activation step
        cnt = np.diff(offsets.astype(np.int64))
        mx = int(cnt.max())
        xp = torch.zeros((E, mx, H), dtype=torch.bfloat16, device="cuda")
        xb = x.view(torch.bfloat16)
        for e in range(E):
            xp[e, :cnt[e]] = xb[int(offsets[e]):int(offsets[e + 1])]
        gu = torch.empty((E, mx, 2 * I), dtype=torch.bfloat16, device="cuda")
        w1t = w1.view(torch.bfloat16).view(E, 2 * I, H).transpose(1, 2)
        gu2 = gu.view(E * mx, 2 * I)
        pk2 = torch.empty((E * mx, I // 2), dtype=torch.uint8, device="cuda")
        sc2 = torch.empty((E * mx, I // 16), dtype=torch.uint8, device="cuda")

        class Unfused:
            def __call__(self):
                torch.bmm(xp, w1t, out=gu)
                M.moe_swiglu_nvfp4_quantize(gu2, 7.0, None, pk2, sc2, stream=stream)
        with torch.cuda.stream(stream):
            _, per_u, _, _ = time_steps(torch, [Unfused()], steps, 2, stream)
        unfused_s = statistics.fmean(per_u)
        torch.cuda.synchronize()
        entry["unfused_cublas_plus_activation_us"] = round(unfused_s * 1e6, 1)
        entry["fused_vs_unfused_time"] = round(fused_s / unfused_s, 3)
        del x, pk, sc, xp, gu, gu2, pk2, sc2
        torch.cuda.empty_cache()
    torch.cuda.synchronize()
    assert int(status.item()) == 0, "a GEMM wait expired"
    del w1, wq, ws
    torch.cuda.empty_cache()
    return res


def config_of(w, world: int) -> dict:
    """The `config` object of both arms' JSON lines: the same workload gives
    the same dict."""
    return {"workload": describe(w), "rows": w.rows, "width": w.width, "experts": w.meta.get("experts"),
            "bytes_per_step": w.algorithmic_bytes(),
            "l2": f"inputs ({w.data.nbytes / 1e6:.0f} MB) larger than L2 (129 MB); 2 input copies alternate",
            "parallelism": f"{world} independent replica(s), no collective on the path"}


def measure_configs(torch, lib, M, W, args, stream, peak: float) -> dict:
    """Configurations 1, 2, 4 and 5 of the step, compact: 1 and 2 (they fit
    in L2) as cold single launches beside their floors; 4 and 5 back to back
    with the isolated per-launch median and the traffic floor, also as
    quantize-only on the same shape (where the scale saturates), and 5 with
    the rates at which the exact path ran on its tie blocks. Configuration 3
    is the headline, timed after these (on a GPU that has left its idle
    clocks) and added by the caller."""
    steps, warm = min(args.steps, 200), min(args.warmup, 20)
    keep = ("us", "gbs", "frac", "p50_frac", "floor_us")
    out = {}
    flush = L2Flush(torch, lib, stream)
    out["1"] = {"w": "quantize-only 128x2048", **small_config(torch, lib, W, "quantize", stream, flush, peak)}
    out["2"] = {"w": "fused 512x2048", **small_config(torch, lib, W, "fused", stream, flush, peak)}
    del flush
    torch.cuda.empty_cache()
    for key, name, label in (("4", "prefill", "prefill 65536x3072"), ("5", "edge", "edge 16384x4096")):
        out[key] = {"w": label, **large_config(torch, lib, M, W, name, steps, warm, stream, peak)}
        torch.cuda.empty_cache()
    for key, name in (("4", "prefill_quantize"), ("5", "edge_quantize")):
        r = large_config(torch, lib, M, W, name, steps, warm, stream, peak)
        out[key]["quantize_only"] = {k: r[k] for k in keep}
        torch.cuda.empty_cache()
    out["5"].update(reevaluation_rates(torch, lib, W, "edge"))
    return out


def main_ours(args):
    import torch
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    import moe_swiglu_epilogue_gb300 as M
    from moe_swiglu_epilogue_gb300 import build, workloads as W
    if rank == 0 or world == 1:
        build.build()
    barrier()
    lib = M.load_library()
    stream = torch.cuda.Stream()
    peak, peak_src = measured_peaks()
    visible = [v for v in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if v.strip()]
    gpu_id = visible[local] if local < len(visible) else str(local)

    # the other configurations run in single-GPU runs only, before the
    # headline's timed region
    configs = None
    if not args.no_extra and world == 1:
        configs = measure_configs(torch, lib, M, W, args, stream, peak)

    sampler = ClockSampler(gpu_id)
    sampler.start()
    headline = run_workload(torch, lib, M, W, args.workload, args.steps, args.warmup, stream)
    sampler.stop()
    w, total_s, per, w0, w1, keep = headline
    clocks = sampler.summary(w0, w1)
    pcts = launch_percentiles(torch, keep[4], 100, stream)
    max_s = max_over_ranks(total_s)
    agg = aggregate_throughput(w.algorithmic_bytes(), w.active_rows, args.steps, max_s, world)
    if configs is not None and w.name == "ragged":
        head = large_config(torch, lib, M, W, w.name, args.steps, args.warmup, stream, peak, timed=headline)
        configs = {"1": configs["1"], "2": configs["2"], "3": {"w": "ragged 32768x2048", **head},
                   "4": configs["4"], "5": configs["5"]}

    e2e_steps = max(3, min(args.steps, args.e2e_steps))
    e2e_s, h2d, d2h, n_chunks = e2e_measure(torch, lib, w, stream, e2e_steps)
    e2e_max = max_over_ranks(e2e_s)
    e2e = {"value": round(world * w.algorithmic_bytes() * e2e_steps / e2e_max / 1e9, 2),
           "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
           "how": f"{n_chunks} C-ABI calls per step on expert groups (device offsets), pinned host "
                  "buffers, uploads/kernels/downloads pipelined on 3 streams"}

    kernel = "nvfp4_quantize_kernel" if w.kind == "quantize" else "swiglu_nvfp4_kernel"
    roof = roofline(w.algorithmic_bytes(), per, peak, peak_src, recorded_traffic(kernel, w.name))
    roof["launch_us_p10_p50_p90"] = pcts

    del headline, keep
    torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = cpu_baseline(w)
        allc = cpu_baseline_all_cores(w)
        cpu["all_cores"] = {"value": round(allc["value"], 3), "cores": allc["cores"]}
        cpu["value"] = round(cpu["value"], 4)
        cpu.pop("rows_per_s", None)
    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": round(agg["gbs"], 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(agg["ms_per_step"], 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded; no dataset)",
        "config": config_of(w, world),
        "rows_per_s": round(agg["rows_per_s"], 1),
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": args.steps,
        "clocks": clocks,
        "configs": configs,
    }
    print(json.dumps(line, separators=(",", ":")), flush=True)


def main_reference(args):
    """The oracle on the host cores, same metric and workload, bounded
    per-step sample; rank 0 only."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    from moe_swiglu_epilogue_gb300 import workloads as W
    oracle.build()
    w = W.make(args.workload)
    r0 = 0 if w.offsets is None else int(w.offsets[0])
    r1 = w.rows if w.offsets is None else int(w.offsets[-1])
    per_row = w.algorithmic_bytes() // max(1, w.active_rows)

    def run(a, n):
        if w.kind == "quantize":
            oracle.quantize_nvfp4(w.data[a:a + n])
        else:
            oracle.swiglu_quantize_nvfp4(w.data[a:a + n], w.clamp_L)

    t = time.perf_counter()
    run(r0, 32)
    per_row_s = (time.perf_counter() - t) / 32
    budget = args.reference_budget_s
    n = int(max(1, min(r1 - r0, budget / (args.steps + args.warmup) / max(per_row_s, 1e-9))))
    for i in range(args.warmup):
        run(r0 + (i * n) % max(1, r1 - r0 - n + 1), n)
    t = time.perf_counter()
    for i in range(args.steps):
        run(r0 + (i * n) % max(1, r1 - r0 - n + 1), n)
    secs = time.perf_counter() - t
    value = per_row * n * args.steps / secs / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(secs * 1e3 / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64/f32 (oracle)",
        "data": "synthetic (seeded; no dataset)",
        "config": config_of(w, world),
        "rows_per_step_sample": n,
        "rows_per_s": round(n * args.steps / secs, 1),
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"{n} consecutive active rows per step"},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def parse(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=HEADLINE,
                    choices=["ragged", "fused", "prefill", "edge", "quantize", "prefill_quantize",
                             "edge_quantize"])
    ap.add_argument("--e2e-steps", type=int, default=30)
    ap.add_argument("--no-extra", action="store_true", help="skip the other configurations")
    ap.add_argument("--gemm-case", default=None, metavar="EXPERTS:TOKENS|all",
                    help="time only the L1 GEMM with the step in its epilogue (top-8 routing, "
                         "H=7168, I=2048) at this size, or 'all' for the decode and prefill cases "
                         "beside the unfused flows, and print its JSON record")
    ap.add_argument("--extension", default=None, choices=EXTENSION_CASES + ("all",),
                    help="time only this extension of the activation step on the ragged "
                         "workload ('all': every one, and the compact flow) and print its JSON record")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--reference-budget-s", type=float, default=90.0)
    return ap.parse_args(argv)


def main_gemm_case(args):
    """--gemm-case: the fused L1 GEMM alone at one size (one JSON record)."""
    import torch
    torch.cuda.set_device(0)
    import moe_swiglu_epilogue_gb300 as M
    from moe_swiglu_epilogue_gb300 import build, workloads as W
    build.build()
    lib = M.load_library()
    stream = torch.cuda.Stream()
    peak, _ = measured_peaks()
    if args.gemm_case == "all":
        res = gemm_measurements(torch, lib, M, W, stream, peak)
    else:
        E, tokens = (int(v) for v in args.gemm_case.split(":"))
        res = gemm_measurements(torch, lib, M, W, stream, peak,
                                cases=((f"l1_gemm_{E}x{tokens}", E, tokens, args.steps),),
                                warmup=args.warmup, unfused=False)
    print(json.dumps(res), flush=True)


def main_extension_case(args):
    """--extension: one extension of the activation step alone (one JSON record)."""
    import torch
    torch.cuda.set_device(0)
    import moe_swiglu_epilogue_gb300 as M
    from moe_swiglu_epilogue_gb300 import build, workloads as W
    build.build()
    lib = M.load_library()
    stream = torch.cuda.Stream()
    peak, _ = measured_peaks()
    only = None if args.extension == "all" else (args.extension,)
    res = extension_measurements(torch, lib, M, W, stream, args.steps, args.warmup, peak, only=only)
    if only is None:                  # the compact flow beside the fused step on the same box
        w, tot, per, _, _, keep = run_workload(torch, lib, M, W, "ragged", args.steps, args.warmup, stream)
        del keep
        res["fused_step_us"] = round(statistics.fmean(per) * 1e6, 2)
        res["compact_flow"]["vs_fused_time"] = round(res["compact_flow"]["launch_us_mean"] / res["fused_step_us"], 3)
    print(json.dumps(res), flush=True)


def main(argv=None):
    args = parse(argv)
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    if args.gemm_case is not None and args.impl == "ours":
        main_gemm_case(args)
    elif args.extension is not None and args.impl == "ours":
        main_extension_case(args)
    elif args.impl == "reference":
        main_reference(args)
    else:
        main_ours(args)


if __name__ == "__main__":
    main()
