#!/usr/bin/env python
"""Throughput of the in-place partial interleaved rotary embedding on GB300.

One step = the forward on x followed by the backward on a gradient of the
same shape (two launches), over the largest configuration: fp32 x of shape
(4, 8192, 32, 128) whose slice [34, 98) is rotated, with one cos/sin row per
(batch, position) of shape (4, 8192, 1, 64).  Inputs are seeded synthetic
data (N(0, 1) activations and gradients, a base-10000 cos/sin table over
per-batch position offsets) resident in HBM before timing; x and grad
(537 MB each) exceed the 129 MB L2, so no flush is needed between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                    [--split tokens|replica] [--strong]

Prints ONE JSON line on rank 0.  `value` is the algorithmic bytes of all
ranks (slice bytes read + written plus the unique cos/sin bytes, per launch)
divided by the slowest rank's device time, over the median of several timed
regions of K steps each.  Under torchrun the ranks split the tokens of one
workload (data parallel, no collective on the data path, only reductions of
the timings): by default the global workload has B x world batches, so each
GPU holds the named workload's size (weak scaling); --strong splits the
named workload itself; --split replica gives every rank its own copy.

`--impl reference` times the CPU oracle on the host cores instead, on a
bounded sample of the same workload, with the same metric.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import platform
import re
import statistics
import subprocess
import sys
import threading
import time
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from place_partial_rope_gb300 import synth  # noqa: E402

METRIC = "in-place partial RoPE fwd/bwd achieved HBM GB/s and % of GB300 peak"
HEADLINE = "large_unaligned"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e, nominal
CSRC = os.path.join(ROOT, "place_partial_rope_gb300", "csrc")
PROFILES = os.path.join(ROOT, "profiles")


# --------------------------------------------------------------------------
# small utilities
# --------------------------------------------------------------------------

def strip_c_comments(text: str) -> str:
    """C/C++ source without its comments and with whitespace runs collapsed
    (string and character literals kept as they are)."""
    out, i, n = [], 0, len(text)
    while i < n:
        ch = text[i]
        if ch in "\"'":
            j = i + 1
            while j < n and text[j] != ch:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(ch)
            i += 1
    return " ".join("".join(out).split())


# The files that define the kernels' device code.  The host planner and the
# launcher are left out: they choose among the kernel instances, and a
# traffic line names the instance it was measured on.
KERNEL_SOURCES = ("fast_div.h", "rope_internal.h", "rope_kernels.cuh", "rope_kernels_bf16.cu",
                  "rope_kernels_fp16.cu", "rope_kernels_fp32.cu")


def kernel_source_hash(read=None) -> str:
    """Hash of the kernels' device-code sources with comments and layout
    removed, to tell whether stored ncu counters still describe the code that
    runs.  `read(name)` returns a file's text (default: the file in CSRC)."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        if read is None:
            with open(os.path.join(CSRC, f), encoding="utf-8") as fh:
                text = fh.read()
        else:
            text = read(f)
        h.update(f.encode() + b"\0" + strip_c_comments(text).encode())
    return h.hexdigest()[:16]


def stored_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary (a `traffic:` line
    in profiles/*.md), or None when there is none for the current kernel
    sources."""
    if not os.path.isdir(PROFILES):
        return None
    pat = re.compile(r"traffic:\s*kernel=(\S+)\s+workload=(\S+)\s+source_sha=(\S+)\s+"
                     r"dram_bytes_per_launch=(\d+)")
    src = kernel_source_hash()
    for name in sorted(os.listdir(PROFILES)):
        if not name.endswith(".md"):
            continue
        with open(os.path.join(PROFILES, name)) as f:
            for line in f:
                m = pat.search(line)
                if m and m.group(1) == kernel and m.group(2) == workload and m.group(3) == src:
                    return int(m.group(4))
    return None


def kernel_name(plan, dtype: str, direction: int) -> str:
    """The template instance a plan runs, as ncu names it (without spaces)."""
    ctype = {"fp32": "float", "bf16": "__nv_bfloat16", "fp16": "__half"}[dtype]
    scalar = "true" if plan.path == 2 else "false"
    rhead = "true" if plan.r_per_head else "false"
    return (f"rope_partial_kernel<{ctype},{plan.vec_bytes},{scalar},{plan.heads_per_thread},"
            f"{direction},{rhead}>")


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# --------------------------------------------------------------------------
# clocks during the timed region (NVML through ctypes; nvidia-smi fallback)
# --------------------------------------------------------------------------

REASON_BITS = [(0x1, "gpu_idle"), (0x2, "applications_clocks_setting"), (0x4, "sw_power_cap"),
               (0x8, "hw_slowdown"), (0x10, "sync_boost"), (0x20, "sw_thermal_slowdown"),
               (0x40, "hw_thermal_slowdown"), (0x80, "hw_power_brake_slowdown"),
               (0x100, "display_clock_setting")]


class ClockSampler:
    """Samples the SM clock and the clock-event reasons while running."""

    def __init__(self, torch_device: int, interval_s: float = 0.002):
        self.interval = interval_s
        self.samples = []
        self.max_mhz = None
        self.source = None
        self._stop = threading.Event()
        self._thread = None
        self._proc = None
        self._nvml = None
        try:
            self._init_nvml(torch_device)
            self.source = "nvml"
        except Exception:
            self._nvml = None
            self.source = "nvidia-smi"

    def _init_nvml(self, torch_device):
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        count = ctypes.c_uint()
        lib.nvmlDeviceGetCount_v2(ctypes.byref(count))
        handle = ctypes.c_void_p()
        index = 0
        try:
            want = str(torch.cuda.get_device_properties(torch_device).uuid).lower().replace("gpu-", "")
            buf = ctypes.create_string_buffer(96)
            for i in range(count.value):
                h = ctypes.c_void_p()
                lib.nvmlDeviceGetHandleByIndex_v2(i, ctypes.byref(h))
                lib.nvmlDeviceGetUUID(h, buf, 96)
                if buf.value.decode().lower().replace("gpu-", "") == want:
                    index = i
                    break
        except Exception:
            index = 0
        if lib.nvmlDeviceGetHandleByIndex_v2(index, ctypes.byref(handle)) != 0:
            raise RuntimeError("no NVML handle")
        mx = ctypes.c_uint()
        lib.nvmlDeviceGetMaxClockInfo(handle, 1, ctypes.byref(mx))  # 1 = SM clock
        self.max_mhz = mx.value
        self._reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
        self._nvml, self._handle = lib, handle

    def _loop(self):
        lib, h = self._nvml, self._handle
        clk, rs = ctypes.c_uint(), ctypes.c_ulonglong()
        while not self._stop.is_set():
            if lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0:
                self._reasons_fn(h, ctypes.byref(rs))
                self.samples.append((clk.value, rs.value))
            time.sleep(self.interval)

    def start(self):
        if self._nvml is not None:
            self._thread = threading.Thread(target=self._loop, daemon=True)
            self._thread.start()
        else:
            try:
                self._proc = subprocess.Popen(
                    ["nvidia-smi", "--query-gpu=clocks.sm,clocks.max.sm,clocks_event_reasons.active",
                     "--format=csv,noheader,nounits", "-lms", "100"],
                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            except Exception:
                self._proc = None

    def stop(self) -> dict:
        if self._thread is not None:
            self._stop.set()
            self._thread.join()
        elif self._proc is not None:
            self._proc.terminate()
            out, _ = self._proc.communicate()
            for line in out.splitlines():
                parts = [p.strip() for p in line.split(",")]
                try:
                    self.samples.append((int(parts[0]), int(parts[2], 16)))
                    self.max_mhz = int(parts[1])
                except (ValueError, IndexError):
                    pass
        mhz = [s for s, _ in self.samples]
        mask = 0
        for _, r in self.samples:
            mask |= r
        reasons = [name for bit, name in REASON_BITS if mask & bit]
        return {"sm_mhz": float(statistics.median(mhz)) if mhz else None,
                "sm_max_mhz": self.max_mhz, "reasons": reasons, "samples": len(mhz),
                "source": self.source}


# --------------------------------------------------------------------------
# distributed plumbing (timing only; the data path has no collective)
# --------------------------------------------------------------------------

def dist_env():
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def reduce_timing(elapsed_s: float, units: float, world: int, device=None):
    """Max of the ranks' elapsed times and the sum of their work units."""
    if world == 1:
        return elapsed_s, units
    import torch.distributed as dist
    t = torch.tensor([elapsed_s], dtype=torch.float64, device=device)
    u = torch.tensor([units], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# --------------------------------------------------------------------------
# CPU oracle timing (the reference arm and the cpu_baseline leg)
# --------------------------------------------------------------------------

def oracle_sample(w, x, r1, r2, g, tokens: int):
    """The first `tokens` tokens (flattened b, s order) of a workload, as a
    (1, tokens, N, D) tensor with the cos/sin row of each token gathered
    beside it; also the number of distinct cos/sin rows those tokens use."""
    B, S, N, D = w.shape
    xs = np.ascontiguousarray(x.reshape(1, B * S, N, D)[:, :tokens])
    gs = np.ascontiguousarray(g.reshape(1, B * S, N, D)[:, :tokens]) if g is not None else None
    t = np.arange(tokens)
    b_idx, s_idx = t // S, t % S

    def gather(r):
        rb = b_idx if r.shape[0] > 1 else np.zeros_like(b_idx)
        rs = s_idx if r.shape[1] > 1 else np.zeros_like(s_idx)
        return np.ascontiguousarray(r[rb, rs][None])  # (1, tokens, Nr, L)

    keys = set(zip((b_idx if r1.shape[0] > 1 else 0 * b_idx).tolist(),
                   (s_idx if r1.shape[1] > 1 else 0 * s_idx).tolist()))
    return xs, gather(r1), gather(r2), gs, len(keys) * r1.shape[2]


def oracle_step(pool, cores, xs, c, s, gs, w):
    """One step of the oracle on a sample: forward over x, backward over
    grad, the tokens split across `cores` threads (the oracle's C calls
    release the GIL; the oracle itself is unchanged)."""
    import oracle
    T = xs.shape[1]
    cuts = np.linspace(0, T, cores + 1).astype(int)
    parts = [(a, b) for a, b in zip(cuts[:-1], cuts[1:]) if b > a]

    def run(args):
        fn, arr, a, b = args
        return fn(arr[:, a:b], c[:, a:b], s[:, a:b], w.dtype, w.start, w.end)

    list(pool.map(run, [(oracle.fwd, xs, a, b) for a, b in parts]))
    if gs is not None:
        list(pool.map(run, [(oracle.bwd, gs, a, b) for a, b in parts]))


def sample_bytes(w, tokens: int, r_rows: int) -> int:
    """Algorithmic bytes of one oracle step over `tokens` positions of batch
    0 (r_rows distinct cos/sin rows), for each direction of the workload."""
    e = synth.ELEM_BYTES[w.dtype]
    N = w.shape[2]
    return len(w.directions) * (2 * tokens * N * w.L * e + 2 * r_rows * w.L * e)


def time_oracle(w, x, r1, r2, g, steps: int, warmup: int, budget_s: float, min_s: float = 0.0):
    """Times the oracle over a sample of the workload: at least `steps`
    steps, more (up to 1000) until about `min_s` seconds of wall time, and
    the sample shrunk if `steps + warmup` of it would pass `budget_s`."""
    import oracle
    oracle.build()
    cores = host_cores()
    tokens = max(1, w.tokens // 4)  # a quarter of the workload's tokens
    xs, c, s, gs, r_rows = oracle_sample(w, x, r1, r2, g, tokens)
    with ThreadPoolExecutor(max_workers=cores) as pool:
        t0 = time.perf_counter()
        oracle_step(pool, cores, xs, c, s, gs, w)
        one = time.perf_counter() - t0
        if one * (steps + warmup) > budget_s:  # shrink the sample to fit the budget
            tokens = max(64, int(tokens * budget_s / (one * (steps + warmup))))
            xs, c, s, gs, r_rows = oracle_sample(w, x, r1, r2, g, tokens)
        for _ in range(max(0, warmup - 1)):
            oracle_step(pool, cores, xs, c, s, gs, w)
        times = []
        while len(times) < steps or (sum(times) < min_s and len(times) < 1000):
            t0 = time.perf_counter()
            oracle_step(pool, cores, xs, c, s, gs, w)
            times.append(time.perf_counter() - t0)
        steps = len(times)
    per_step = sample_bytes(w, tokens, r_rows)
    total = sum(times)
    dirs = " + ".join({"fwd": "forward", "bwd": "backward"}[d] for d in w.directions)
    sample = (f"{dirs} of the CPU oracle over the first {tokens} of {w.tokens} tokens of the "
              f"{w.name} workload ({tokens} x {w.shape[2]} rows of {w.L} {w.dtype} lanes), tokens "
              f"split across {cores} threads; {steps} steps")
    return {"value": per_step * steps / total / 1e9, "unit": "GB/s", "cores": cores,
            "kind": "oracle", "sample": sample, "ms_per_step": 1e3 * total / steps}


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else platform)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.processor() or platform.machine()


def oracle_per_workload(names=("small_model", "gqa", "mla_decode_q", "large_unaligned"),
                        sample_bytes_target: int = 16 * 2**20, reps: int = 5) -> dict:
    """The oracle on each large workload and direction, on one thread and on
    all host cores: the median of `reps` runs over a sample of the
    workload's first tokens (about `sample_bytes_target` algorithmic bytes
    per run).  A baseline only."""
    import oracle
    oracle.build()
    cores = host_cores()
    out = {}
    with ThreadPoolExecutor(max_workers=cores) as pool:
        for name in names:
            w = synth.WORKLOADS[name]
            x, r1, r2, g = synth.workload_inputs(w)
            per_tok = 2 * w.shape[2] * w.L * synth.ELEM_BYTES[w.dtype]
            tokens = int(min(w.tokens, max(1, sample_bytes_target // per_tok)))
            xs, c, s, gs, r_rows = oracle_sample(w, x, r1, r2, g, tokens)
            nbytes = sample_bytes(w, tokens, r_rows) // len(w.directions)
            cuts = np.linspace(0, tokens, cores + 1).astype(int)
            parts = [(a, b) for a, b in zip(cuts[:-1], cuts[1:]) if b > a]
            entry = {"sample_tokens": tokens, "of_tokens": w.tokens}
            for d in w.directions:
                fn = oracle.fwd if d == "fwd" else oracle.bwd
                arr = xs if d == "fwd" else gs

                def one():
                    fn(arr, c, s, w.dtype, w.start, w.end)

                def many():
                    list(pool.map(lambda ab: fn(arr[:, ab[0]:ab[1]], c[:, ab[0]:ab[1]],
                                                s[:, ab[0]:ab[1]], w.dtype, w.start, w.end), parts))

                res = {}
                for label, f in (("1_thread", one), (f"{cores}_threads", many)):
                    f()
                    ts = []
                    for _ in range(reps):
                        t0 = time.perf_counter()
                        f()
                        ts.append(time.perf_counter() - t0)
                    res[label + "_GB/s"] = round(nbytes / statistics.median(ts) / 1e9, 3)
                entry[d] = res
            out[name] = entry
            del x, g
    return out


# --------------------------------------------------------------------------
# the GPU arm
# --------------------------------------------------------------------------

def dram_floor_bytes(w) -> int:
    """The fewest DRAM bytes one launch can move for this layout: every
    row's slice read in whole 64-byte DRAM atoms and written in whole
    32-byte sectors (the granularities the ncu counters show on this GPU:
    352.3 MB read for the large fp32 shape's 256-byte slices at byte 136),
    plus the unique cos and sin bytes.  Rows start at multiples of the row
    pitch from a 256-byte aligned base."""
    e = synth.ELEM_BYTES[w.dtype]
    B, S, N, D = w.shape
    rows, pitch, off, length = B * S * N, D * e, w.start * e, w.L * e

    def touched(lo: int, hi: int, g: int) -> int:
        return 0 if hi <= lo else ((hi + g - 1) // g - lo // g) * g

    period = 256 // math.gcd(pitch, 256)
    per = [touched(r * pitch + off, r * pitch + off + length, 64) +
           touched(r * pitch + off, r * pitch + off + length, 32) for r in range(period)]
    body = sum(per) * (rows // period) + sum(per[:rows % period])
    return body + 2 * int(np.prod(w.r_shape)) * e


def workload_config(w, l2_bytes: int = 132 * 2**20) -> dict:
    step = ("forward on x then backward on grad (2 launches)" if "bwd" in w.directions
            else "forward on x (1 launch)")
    xbytes = int(np.prod(w.shape)) * synth.ELEM_BYTES[w.dtype]
    big = w.algorithmic_bytes() > 1.5 * l2_bytes
    l2 = (f"inputs larger than L2 ({xbytes / 1e6:.0f} MB per tensor, {w.algorithmic_bytes() / 1e6:.0f} "
          f"MB touched per launch vs {l2_bytes / 1e6:.0f} MB L2): no flush between steps" if big else
          f"NOT larger than L2 ({w.algorithmic_bytes() / 1e6:.1f} MB touched per launch vs "
          f"{l2_bytes / 1e6:.0f} MB L2): steps run partly from L2, so this is not an HBM figure")
    return {"workload": f"{w.name}: {w.description}; one step = {step}",
            "x_shape": list(w.shape), "partial_slice": [w.start, w.end], "r_shape": list(w.r_shape),
            "algorithmic_bytes_per_launch": w.algorithmic_bytes(), "l2": l2,
            "parallelism": "one independent copy of the workload per GPU"}


def l2_flusher(device):
    """Flush L2 without leaving it dirty: write a buffer 2.5x the L2 size,
    then read another of that size, so the next kernel starts with none of
    its own lines cached and pays no write-back of the flush's lines."""
    size = torch.cuda.get_device_properties(device).L2_cache_size
    n = int(2.5 * size) // 4 + 1
    wbuf = torch.empty(n, dtype=torch.float32, device=device)
    rbuf = torch.ones(n, dtype=torch.float32, device=device)

    def flush():
        wbuf.fill_(1.0)
        torch.sum(rbuf)
    return flush


def time_launches(fn, n: int, flush=None):
    """Median device time (s) of n launches, each bracketed by its own events;
    the L2 flush (if any) runs outside the events and keeps the GPU busy
    while the host queues the launch."""
    evs = []
    for _ in range(n):
        if flush is not None:
            flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        evs.append((a, b))
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) for a, b in evs) / 1e3


def time_back_to_back(fn, n: int, reps: int = 5):
    """Per-launch device time (s) of n launches back to back between two
    events; the median of `reps` repetitions."""
    out = []
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(n):
            fn()
        b.record()
        torch.cuda.synchronize()
        out.append(a.elapsed_time(b) / 1e3 / n)
    return statistics.median(out)


def time_graph(make_call, n: int, reps: int = 5):
    """Per-launch time of n launches captured in one CUDA graph and replayed
    (no host launch cost; the data stays in L2 when it fits)."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call = make_call()  # marshalled on the capture stream
        for _ in range(n):
            call()
    g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        g.replay()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / 1e3 / (n * reps)


def breakdown(device, peak):
    """Per named workload and direction: cold (L2-flushed) device time per
    launch, GB/s and fraction of peak; steady back-to-back time where the
    bytes a launch touches exceed 1.5x the L2; and the per-launch time of a
    replayed CUDA graph of 20 launches."""
    from place_partial_rope_gb300 import binding
    flush = l2_flusher(device)
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    out = {}
    for name, w in synth.WORKLOADS.items():
        x, r1, r2, g = synth.workload_inputs(w)
        xd = synth.to_torch(x, w.dtype).to(device)
        gd = synth.to_torch(g, w.dtype).to(device) if g is not None else None
        c = synth.to_torch(r1, w.dtype).to(device)
        s = synth.to_torch(r2, w.dtype).to(device)
        entry = {}
        for d in w.directions:
            buf = xd if d == "fwd" else gd
            prep = binding.prepare_fwd if d == "fwd" else binding.prepare_bwd
            call = prep(buf, c, s, w.start, w.end)
            for _ in range(3):
                call()
            t = time_launches(call, 50, flush)
            gbs = w.algorithmic_bytes() / t / 1e9
            e = {"cold_us": round(t * 1e6, 2), "cold_GB/s": round(gbs, 1),
                 "cold_frac": round(gbs / peak, 4)}
            if w.algorithmic_bytes() > 1.5 * l2:
                tb = time_back_to_back(call, 50)
                e["steady_us"] = round(tb * 1e6, 2)
                e["steady_frac"] = round(w.algorithmic_bytes() / tb / 1e9 / peak, 4)
                e["of_record"] = "steady_frac"
            else:
                e["of_record"] = "cold_frac"
            e["graph_us"] = round(time_graph(lambda: prep(buf, c, s, w.start, w.end), 20) * 1e6, 2)
            if w.algorithmic_bytes() < l2:
                e["graph_l2_resident"] = True
            entry[d] = e
        out[name] = entry
        del xd, gd, c, s
    out["fused_qk"] = qk_breakdown(device, peak, flush)
    out["half_split"] = half_breakdown(device, peak, flush, l2)
    out["positions"] = positions_breakdown(device, peak, flush, l2)
    out["odd_start"] = odd_breakdown(device, peak, flush, l2)
    torch.cuda.empty_cache()
    out["e2e_gqa"] = e2e_aligned(device)
    mark_above_peak(out)
    out["notes"] = {
        "cold": "one launch after an L2 flush, between its own events; the end event fires with "
                "part of the launch's writes still dirty in L2, so a cold window under-counts DRAM "
                "write time and a cold fraction can pass 1.0 (listed under above_peak)",
        "steady": "launches back to back on inputs larger than 1.5x L2: the HBM figure of record "
                  "where it is given (of_record names the figure of record per entry)",
        "graph": "per-launch time of a replayed CUDA graph of 20 launches; graph_l2_resident "
                 "marks shapes whose bytes fit in L2, so the replay runs from L2, not HBM",
        "e2e_gqa": "the zero-copy host-buffer calls on the GQA shape (its slices are 128-byte "
                   "aligned), against the host link's own copy rates measured in the same run"}
    return out


def mark_above_peak(d):
    """List, per entry, the cold fractions above 1.0 (under `above_peak`)."""
    if not isinstance(d, dict):
        return
    for k, v in list(d.items()):
        if isinstance(v, dict):
            mark_above_peak(v)
        elif (k.endswith("frac") and "steady" not in k and "floor" not in k
              and isinstance(v, (int, float)) and v > 1.0):
            d.setdefault("above_peak", []).append(k)


def host_link_rates(device, nbytes: int = 256 * 2**20) -> dict:
    """The host link's copy rates between page-locked host memory and the
    device: host to device alone, device to host alone, and both at once
    (two streams)."""
    h1 = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    h2 = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    d1 = torch.empty(nbytes, dtype=torch.uint8, device=device)
    d2 = torch.empty(nbytes, dtype=torch.uint8, device=device)
    s1, s2 = torch.cuda.Stream(device), torch.cuda.Stream(device)

    def rate(both: bool, h2d: bool, reps: int = 5) -> float:
        ts = []
        for _ in range(reps):
            torch.cuda.synchronize(device)
            t = time.perf_counter()
            if both or h2d:
                with torch.cuda.stream(s1):
                    d1.copy_(h1, non_blocking=True)
            if both or not h2d:
                with torch.cuda.stream(s2):
                    h2.copy_(d2, non_blocking=True)
            torch.cuda.synchronize(device)
            ts.append(time.perf_counter() - t)
        return round((2 if both else 1) * nbytes / statistics.median(ts) / 1e9, 1)

    rate(False, True, 1)
    return {"h2d_GB/s": rate(False, True), "d2h_GB/s": rate(False, False),
            "both_GB/s": rate(True, True), "bytes_each": nbytes}


def e2e_aligned(device) -> dict:
    """The e2e measurement on the GQA shape (aligned 128-byte slices), with
    the host link's own copy rates beside it."""
    from place_partial_rope_gb300 import binding, shard
    w = synth.WORKLOADS["gqa"]
    ri = shard.rank_inputs(w, 0, 1)
    out = e2e_measure(w, ri, device, 10, binding, shard, 1)
    out["host_link"] = host_link_rates(device)
    out["frac_of_concurrent_copy"] = round(out["value"] / out["host_link"]["both_GB/s"], 4)
    return out


def odd_breakdown(device, peak, flush, l2):
    """Odd slice starts, forward, per launch: on the gqa shape (fp16, one
    cos/sin row per position) [1, 65) (32 pairs per row), [1, 63) (31: the
    row's last lane stores part of its vector), [5, 69) (element 1 of an
    8-byte vector) and [3, 45) (21 pairs from element 3 of a vector); on the
    large fp32 shape (per-batch position offsets) [1, 65) and [3, 67).  A
    start at element 1 of a 16- or 8-byte vector runs the odd-start kernel
    (path 4, a lane per aligned vector of x), [3, 45) the element path
    (path 2).  Such a slice touches one more 64-byte DRAM atom per row than
    an aligned one, so each entry also gives the layout's DRAM floor and the
    fraction of it."""
    import dataclasses
    from place_partial_rope_gb300 import binding
    out = {}
    for name, cases in (("gqa", ((1, 65), (1, 63), (5, 69), (3, 45))),
                        ("large_unaligned", ((1, 65), (3, 67)))):
        w0 = synth.WORKLOADS[name]
        x = synth.normal(w0.shape, w0.dtype, w0.seed)
        xd = synth.to_torch(x, w0.dtype).to(device)
        pos = synth.positions(w0)
        for st, en in cases:
            if not wanted(f"{name} [{st},{en})"):
                continue
            L = en - st
            w = dataclasses.replace(w0, start=st, end=en, r_shape=w0.r_shape[:3] + (L,))
            r1, r2 = synth.rope_table(pos, L, w.dtype)
            c, s = synth.to_torch(r1, w.dtype).to(device), synth.to_torch(r2, w.dtype).to(device)
            call = binding.prepare_fwd(xd, c, s, st, en)
            plan = binding.rope_partial_plan(xd, c, s, st, en)
            for _ in range(3):
                call()
            t = time_launches(call, 50, flush)
            nbytes = w.algorithmic_bytes()
            floor = nbytes / dram_floor_bytes(w)
            entry = {"path": int(plan.path), "vec_bytes": int(plan.vec_bytes),
                     "lanes_per_row": int(plan.chunks_per_row),
                     "heads_per_thread": int(plan.heads_per_thread),
                     "cold_us": round(t * 1e6, 2), "cold_frac": round(nbytes / t / 1e9 / peak, 4),
                     "floor_frac": round(floor, 4)}
            if nbytes > 1.5 * l2:
                tb = time_back_to_back(call, 50)
                entry["steady_us"] = round(tb * 1e6, 2)
                entry["steady_frac"] = round(nbytes / tb / 1e9 / peak, 4)
                entry["steady_frac_of_floor"] = round(nbytes / tb / 1e9 / peak / floor, 4)
            out[f"{name} [{st},{en})"] = {"fwd": entry}
            del c, s
        del xd
    return out


def positions_breakdown(device, peak, flush, l2):
    """cos/sin computed in the kernel from int32 positions (no table read)
    on the three large shapes, forward, per launch (interleave mode; the
    gqa and large fp32 shapes also in half-split mode).  The fraction is of
    the bytes the positions call moves (the slice read + written, plus 4
    bytes per position)."""
    from place_partial_rope_gb300 import binding
    out = {}
    for name, modes in (("gqa", ("interleave", "half")), ("mla_decode_q", ("interleave",)),
                        ("large_unaligned", ("interleave", "half"))):
        if not wanted(name):
            continue
        w = synth.WORKLOADS[name]
        x = synth.normal(w.shape, w.dtype, w.seed)
        pos = np.ascontiguousarray(synth.positions(w)[..., 0], dtype=np.int32)
        xd = synth.to_torch(x, w.dtype).to(device)
        pd = torch.from_numpy(pos).to(device)
        nbytes = 2 * w.slice_elems() * synth.ELEM_BYTES[w.dtype] + pos.nbytes
        for mode in modes:
            call = binding.PreparedPos("fwd", xd, pd, w.start, w.end, mode=mode)
            for _ in range(3):
                call()
            t = time_launches(call, 50, flush)
            e = {"cold_us": round(t * 1e6, 2), "cold_frac": round(nbytes / t / 1e9 / peak, 4)}
            if nbytes > 1.5 * l2:
                tb = time_back_to_back(call, 50)
                e["steady_us"] = round(tb * 1e6, 2)
                e["steady_frac"] = round(nbytes / tb / 1e9 / peak, 4)
            out[name if mode == "interleave" else f"{name}/half"] = {"fwd": e}
        del xd, pd
    return out


# `--section ... --case TEXT` runs only the entries whose label holds TEXT.
CASE = None


def wanted(label: str) -> bool:
    return CASE is None or CASE in label


def half_breakdown(device, peak, flush, l2):
    """The half-split rotary mode (pairs (i, i + L/2)) on the gqa and large
    fp32 shapes with a half-layout cos/sin table, forward, per launch.  Their
    rows are 8 and 32 accesses per half pair, so a lane's partner access
    comes from another lane (rope_partial_half_lanes_kernel); the large
    shape's [0, 96) has 12 per half and runs both halves in one thread
    (rope_partial_half_kernel)."""
    import dataclasses
    from place_partial_rope_gb300 import binding
    out = {}
    L0 = synth.WORKLOADS["large_unaligned"]
    cases = (("gqa", synth.WORKLOADS["gqa"]), ("large_unaligned", L0),
             ("large_unaligned [0,96)", dataclasses.replace(L0, start=0, end=96,
                                                            r_shape=L0.r_shape[:3] + (96,))))
    for name, w in cases:
        if not wanted(name):
            continue
        x = synth.normal(w.shape, w.dtype, w.seed)
        r1, r2 = synth.rope_table(synth.positions(w), w.L, w.dtype, layout="half")
        xd = synth.to_torch(x, w.dtype).to(device)
        c, s = synth.to_torch(r1, w.dtype).to(device), synth.to_torch(r2, w.dtype).to(device)
        call = binding.prepare_fwd(xd, c, s, w.start, w.end, mode="half")
        plan = binding.rope_partial_plan(xd, c, s, w.start, w.end, 0, "half")
        for _ in range(3):
            call()
        t = time_launches(call, 50, flush)
        tb = time_back_to_back(call, 50)
        out[name] = {"fwd": {"kernel": "half_lanes" if plan.path == 3 else "half",
                             "cold_us": round(t * 1e6, 2),
                             "cold_frac": round(w.algorithmic_bytes() / t / 1e9 / peak, 4),
                             "steady_us": round(tb * 1e6, 2),
                             "steady_frac": round(w.algorithmic_bytes() / tb / 1e9 / peak, 4)}}
        del xd, c, s
    return out


def qk_breakdown(device, peak, flush):
    """The fused query + key MLA-decode call against two single launches
    (query, then key), cold, per call."""
    from place_partial_rope_gb300 import binding
    w = synth.WORKLOADS["mla_decode_q"]
    q, k, r1, r2 = synth.qk_inputs()
    qd, kd = synth.to_torch(q, w.dtype).to(device), synth.to_torch(k, w.dtype).to(device)
    c, s = synth.to_torch(r1, w.dtype).to(device), synth.to_torch(r2, w.dtype).to(device)
    ks = synth.QK_KEY_SLICE
    fused = binding.PreparedQK("fwd", qd, kd, c, s, (w.start, w.end), ks)
    one_q = binding.prepare_fwd(qd, c, s, w.start, w.end)
    one_k = binding.prepare_fwd(kd, c, s, ks[0], ks[1])

    def separate():
        one_q()
        one_k()

    for _ in range(3):
        fused()
        separate()
    tf = time_launches(fused, 50, flush)
    ts = time_launches(separate, 50, flush)
    nbytes = synth.qk_algorithmic_bytes()
    out = {"fwd": {"fused_cold_us": round(tf * 1e6, 2), "separate_cold_us": round(ts * 1e6, 2),
                   "fused_GB/s": round(nbytes / tf / 1e9, 1),
                   "fused_frac": round(nbytes / tf / 1e9 / peak, 4),
                   "what": "query (4096,1,128,192) [0,64) + key (4096,1,1,64) [0,64), bf16, one "
                           "cos/sin row per token: one fused launch vs query then key"}}
    del qd, kd, fused, one_q, one_k

    # a GQA pair: the gqa query with 4 key heads of the same rows
    g = synth.WORKLOADS["gqa"]
    q = synth.normal(g.shape, g.dtype, g.seed)
    k = synth.normal(g.shape[:2] + (4,) + g.shape[3:], g.dtype, g.seed + 600)
    r1, r2 = synth.rope_table(synth.positions(g), g.L, g.dtype)
    qd, kd = synth.to_torch(q, g.dtype).to(device), synth.to_torch(k, g.dtype).to(device)
    c, s = synth.to_torch(r1, g.dtype).to(device), synth.to_torch(r2, g.dtype).to(device)
    fused = binding.PreparedQK("fwd", qd, kd, c, s, (g.start, g.end), (g.start, g.end))
    one_q = binding.prepare_fwd(qd, c, s, g.start, g.end)
    one_k = binding.prepare_fwd(kd, c, s, g.start, g.end)
    for _ in range(3):
        fused()
        separate()
    tf = time_launches(fused, 50, flush)
    ts = time_launches(separate, 50, flush)
    tfb, tsb = time_back_to_back(fused, 50), time_back_to_back(separate, 25)
    e = synth.ELEM_BYTES[g.dtype]
    nbytes = 2 * (qd.numel() + kd.numel()) // g.shape[3] * g.L * e + 2 * r1.size * e
    out["gqa_fwd"] = {"fused_cold_us": round(tf * 1e6, 2), "separate_cold_us": round(ts * 1e6, 2),
                      "fused_steady_us": round(tfb * 1e6, 2), "separate_steady_us": round(tsb * 1e6, 2),
                      "fused_frac": round(nbytes / tf / 1e9 / peak, 4),
                      "fused_steady_frac": round(nbytes / tfb / 1e9 / peak, 4),
                      "what": "query (32,2048,16,128) + key (32,2048,4,128), slices [0,64), fp16, "
                              "cos/sin (1,2048,1,64): one fused launch vs query then key"}
    return out


def reduce_regions(elapsed, units: float, world: int, device=None):
    """Per timed region the slowest rank's elapsed time, and the sum of the
    ranks' work units per region."""
    if world == 1:
        return list(elapsed), units
    import torch.distributed as dist
    t = torch.tensor(elapsed, dtype=torch.float64, device=device)
    u = torch.tensor([units], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return [float(v) for v in t.tolist()], float(u.item())


def region_count(first_s: float, world: int, device=None, min_regions: int = 5,
                 min_total_s: float = 0.1, max_regions: int = 200) -> int:
    """How many K-step regions to time: at least 5, and enough for about
    100 ms of timed work (the same count on every rank)."""
    t, _ = reduce_timing(first_s, 0.0, world, device)
    return max(min_regions, min(max_regions, math.ceil(min_total_s / max(t, 1e-9))))


def rank_calls(binding, shard, ri, bufs, tables, w, host=False):
    """One step of a rank: each direction of the workload over each run of
    the rank's share (one library call per run), forward first."""
    calls = []
    for d in w.directions:
        buf = bufs[d]
        if host:
            prep = binding.prepare_fwd_host if d == "fwd" else binding.prepare_bwd_host
        else:
            prep = binding.prepare_fwd if d == "fwd" else binding.prepare_bwd
        for run, (c, s) in zip(ri.share.runs, tables):
            calls.append(prep(shard.run_block(buf, ri.share, run), c, s, w.start, w.end))
    return calls


def gpu_arm(args):
    world, rank, local = dist_env()
    from place_partial_rope_gb300 import binding, build, shard
    build.build()  # no-op when the in-tree library is current
    lib = binding.load_library()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)

    w = synth.WORKLOADS[args.workload]
    peak, peak_kind = hbm_peak()
    # The rank's inputs: its share of the tokens (rows of x and grad, and
    # its tokens' cos/sin rows), one run per contiguous block.  With one
    # rank that is the named workload itself.
    if args.split == "tokens":
        ri = shard.rank_inputs(w, rank, world, weak=not args.strong)
    else:
        ri = shard.rank_inputs(w, 0, 1)
    share = ri.share
    xd = synth.to_torch(ri.x, w.dtype).to(device)
    gd = synth.to_torch(ri.g, w.dtype).to(device) if ri.g is not None else None
    tabs = [(synth.to_torch(c, w.dtype).to(device), synth.to_torch(s, w.dtype).to(device))
            for c, s in ri.tables]
    stream = torch.cuda.current_stream(device)
    plan = (binding.rope_partial_plan(shard.run_block(xd, share, share.runs[0]), *tabs[0], w.start,
                                      w.end) if share.runs else None)

    # Arguments are marshalled once: one ctypes call (about 4 us of host
    # time) per launch, below the time a launch of the large workloads takes.
    calls = rank_calls(binding, shard, ri, {"fwd": xd, "bwd": gd}, tabs, w)
    ndir = len(w.directions)
    per_launch = ri.algorithmic_bytes()  # one direction over the rank's runs
    bytes_step = ndir * per_launch
    # kernel launches per step (a call whose work index would pass 2^31
    # launches once per piece)
    launches_step = ndir * sum(int(binding.rope_partial_plan(
        shard.run_block(xd, share, run), c, s, w.start, w.end).launches)
        for run, (c, s) in zip(share.runs, tabs))

    for _ in range(args.warmup):
        for call in calls:
            call()
    K = args.steps
    # Each timed region holds K steps and nothing else: an event at each end.
    # Launches carry programmatic dependent launch, so each one's launch and
    # ramp overlap the previous one's tail; an event between two launches
    # would serialise them and add its own ~1.7 us.  The region is timed
    # several times (at least 5, and about 100 ms of work in all); the
    # median is reported, and the clock sampler runs across all of them.
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local)
    elapsed = []

    def region():
        barrier(world)
        torch.cuda.synchronize(device)
        t0.record(stream)
        for _ in range(K):
            for call in calls:
                call()
        t1.record(stream)
        torch.cuda.synchronize(device)
        elapsed.append(t0.elapsed_time(t1) / 1e3)

    sampler.start()
    region()
    nreg = region_count(elapsed[0], world, device)
    for _ in range(nreg - 1):
        region()
    clocks = sampler.stop()
    barrier(world)

    reg_max, total_bytes = reduce_regions(elapsed, bytes_step * K, world, device)
    _, total_elems = reduce_timing(0.0, float(ndir * share.tokens * w.shape[2] * w.L * K), world,
                                   device)
    med = statistics.median(reg_max)
    value = total_bytes / med / 1e9 if med > 0 else 0.0
    regions = {"count": nreg, "steps_each": K, "median_ms": round(med * 1e3, 4),
               "min_ms": round(min(reg_max) * 1e3, 4), "max_ms": round(max(reg_max) * 1e3, 4),
               "spread": round((max(reg_max) - min(reg_max)) / med, 4),
               "note": "value and ms_per_step use the median region (slowest rank per region)"}

    # Each direction timed alone, between its own events, after the timed
    # regions (these serialise the launches); the slower one names the
    # dominant kernel, whose average launch duration over the timed region is
    # the median region's time over its launches (the step is nothing but
    # these launches, back to back).
    nl = len(calls)
    Ki = min(K, 50)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * nl * Ki)]
    for i in range(Ki):
        for j, call in enumerate(calls):
            ev[2 * (nl * i + j)].record(stream)
            call()
            ev[2 * (nl * i + j) + 1].record(stream)
    torch.cuda.synchronize(device)
    runs_per_dir = max(1, len(share.runs))
    iso_call = [statistics.mean(ev[2 * (nl * i + j)].elapsed_time(ev[2 * (nl * i + j) + 1]) / 1e3
                                for i in range(Ki)) for j in range(nl)] if nl else []
    isolated = [sum(iso_call[k * runs_per_dir:(k + 1) * runs_per_dir]) for k in range(ndir)] \
        if nl else [0.0] * ndir
    dom = max(range(ndir), key=lambda j: isolated[j])
    kname = kernel_name(plan, w.dtype, dom) if plan is not None else None
    avg = med / (ndir * K)
    achieved = per_launch / avg / 1e9 if (per_launch and avg > 0) else 0.0
    traffic = stored_traffic(kname, w.name) if (kname and world == 1) else None
    floor = dram_floor_bytes(w)
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": traffic,
                "peak_source": f"{peak_kind} (HBM copy bandwidth, MEASURED_PEAKS.json hbm_gbs)"
                if peak_kind == "measured" else "fallback 6.8 TB/s",
                "frac_of_nominal": round(achieved / NOMINAL_HBM_GBS, 4),
                "nominal_peak": NOMINAL_HBM_GBS,
                "target_basis": "the >= 80 % target is judged on frac (of the measured copy "
                                "rate); frac_of_nominal divides by the nominal HBM3e bandwidth",
                "kernel": kname, "kernel_avg_us": round(avg * 1e6, 2),
                "timing": "average launch duration over the median timed region: its elapsed "
                          "time (CUDA events at its two ends) over its launches, which are only "
                          "this workload's forward and backward kernels back to back",
                "isolated_avg_us": {d: round(isolated[j] * 1e6, 2)
                                    for j, d in enumerate(w.directions)},
                "algorithmic_bytes_per_launch": per_launch,
                "dram_floor_bytes_per_launch": floor,
                "floor_frac": round(w.algorithmic_bytes() / floor, 4),
                "frac_of_floor": round(achieved / peak * floor / w.algorithmic_bytes(), 4),
                "floor_note": "the fewest DRAM bytes the layout allows (64-byte read atoms, "
                              "32-byte write sectors per row's slice, plus cos/sin); floor_frac "
                              "is the highest frac reachable at the measured copy rate",
                "traffic_note": "dram bytes read + written per launch, from the committed ncu "
                                "summary of the same kernel sources (cold L2; part of the writes "
                                "are still in L2 when the kernel ends)" if traffic else
                                "no ncu summary for the current kernel sources"}

    e2e = e2e_measure(w, ri, device, min(K, 20), binding, shard, world)
    ceiling = dense_rmw_ceiling(xd)
    wg = ri.workload
    split = ("tokens" if args.split == "tokens" else "replica")
    config = workload_config(w, torch.cuda.get_device_properties(device).L2_cache_size)
    if split == "tokens":
        config["parallelism"] = (
            f"data-parallel token split over {world} GPU(s), no collective on the data path: "
            f"global x {list(wg.shape)}, rank r rotates its tokens [t0, t1) of the "
            f"{wg.shape[0]} x {wg.shape[1]} grid with its own cos/sin rows "
            f"({'strong' if args.strong else 'weak'} scaling)")
        config["split"] = {"mode": "tokens", "global_shape": list(wg.shape),
                           "global_r_shape": list(wg.r_shape), "rank0_tokens": [share.t0, share.t1]
                           if rank == 0 else None, "runs_rank0": len(share.runs)}
    else:
        config["parallelism"] = "one independent copy of the workload per GPU (replicas)"
    out = {"metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
           "steps": K, "warmup": args.warmup, "ms_per_step": round(1e3 * med / K, 5),
           "higher_is_better": True, "scaling": "strong" if args.strong else "weak",
           "vs_baseline": None, "dtype": w.dtype,
           "data": "synthetic: seeded N(0,1) activations and gradients, base-10000 cos/sin table "
                   "at the workload's seeded positions",
           "config": config,
           "frac_of_peak": round(value / world / peak, 4),
           "gelem_per_s": round(total_elems / med / 1e9, 2) if med > 0 else 0.0,
           "roofline": roofline, "e2e": e2e,
           "gpu_launches": K * launches_step,
           "timed_regions": regions,
           "clocks": clocks, "ceiling": ceiling,
           "plan": {"vec_bytes": plan.vec_bytes, "heads_per_thread": plan.heads_per_thread,
                    "blocks": plan.blocks, "threads_per_block": plan.threads_per_block,
                    "launches_per_call": plan.launches, "runs_per_direction": len(share.runs)}
           if plan is not None else None}
    if rank == 0:
        out["workloads"] = breakdown(device, peak)
    if rank == 0 and world == 1:
        x, g = ri.x.reshape(w.shape), (ri.g.reshape(w.shape) if ri.g is not None else None)
        r1, r2 = ri.tables[0]
        out["cpu_baseline"] = time_oracle(w, x, r1, r2, g, steps=20, warmup=1, budget_s=60.0, min_s=10.0)
        out["cpu_baseline"].pop("ms_per_step", None)
        out["cpu_baseline"]["cpu_model"] = cpu_model()
        out["cpu_baseline"]["workloads"] = oracle_per_workload()
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    _ = lib
    return 0


def dense_rmw_ceiling(xd, n: int = 20) -> dict:
    """Context for the roofline: torch's own in-place elementwise op over the
    WHOLE x tensor (every byte read and written, fully contiguous), timed
    back to back like the steps.  It is the practical HBM ceiling of an
    in-place read-modify-write on this GPU; the rotation touches only the
    slice bytes, so its achievable fraction is lower by the DRAM atoms its
    rows cannot use."""
    xd.mul_(1.0)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(n):
        xd.mul_(1.0)
    b.record()
    torch.cuda.synchronize()
    t = a.elapsed_time(b) / 1e3 / n
    return {"op": "torch x.mul_(1.0) over all of x (in place)", "us": round(t * 1e6, 2),
            "GB/s": round(2 * xd.numel() * xd.element_size() / t / 1e9, 1)}


def e2e_measure(w, ri, device, steps: int, binding, shard, world: int = 1):
    """The same metric end to end, with inputs and results in host memory.

    Headline (zero copy): the rank's x, grad and cos/sin rows stay in
    page-locked host memory; every step calls the *_host entry points (one
    per run of the rank's tokens), whose kernel reads the slice bytes and
    cos/sin rows across the host link (NVLink-C2C on Grace-Blackwell) and
    writes the rotated slice back into the host buffers.  The bytes crossing
    the link are counted from the tensors' slices.  For comparison,
    `copy_path` copies the whole tensors to device buffers, runs the
    launches there, and copies x and grad back.  With several ranks each
    moves its own tokens over its own link; the value is all ranks' bytes
    over the slowest rank's time."""
    e = synth.ELEM_BYTES[w.dtype]
    share = ri.share
    has_bwd = ri.g is not None
    hx = synth.to_torch(ri.x, w.dtype).pin_memory()
    hg = synth.to_torch(ri.g, w.dtype).pin_memory() if has_bwd else None
    htabs = [(synth.to_torch(c, w.dtype).pin_memory(), synth.to_torch(s, w.dtype).pin_memory())
             for c, s in ri.tables]
    ndir = len(w.directions)
    algo = ndir * ri.algorithmic_bytes()

    def timed(step):
        """Per-step time of the slowest rank, and the job's GB/s."""
        step()
        torch.cuda.synchronize(device)
        barrier(world)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(steps):
            step()
        b.record()
        torch.cuda.synchronize(device)
        t, total = reduce_timing(a.elapsed_time(b) / 1e3, algo * steps, world, device)
        return t / steps, (total / t / 1e9 if t > 0 else 0.0)

    zc = rank_calls(binding, shard, ri, {"fwd": hx, "bwd": hg}, htabs, w, host=True)

    def zero_copy_step():
        for call in zc:
            call()

    t_zc, gbs_zc = timed(zero_copy_step)
    slice_bytes = share.tokens * w.shape[2] * w.L * e
    r_bytes = sum((c.numel() + s.numel()) * e for c, s in htabs)
    r_whole = sum(c.nbytes + s.nbytes for c, s in htabs)

    dx = torch.empty_like(hx, device=device)
    dtabs = [(torch.empty_like(c, device=device), torch.empty_like(s, device=device))
             for c, s in htabs]
    ox = torch.empty_like(hx).pin_memory()
    dg = torch.empty_like(hg, device=device) if has_bwd else None
    og = torch.empty_like(hg).pin_memory() if has_bwd else None
    dev_calls = rank_calls(binding, shard, ri, {"fwd": dx, "bwd": dg}, dtabs, w)

    def copy_step():
        dx.copy_(hx, non_blocking=True)
        if has_bwd:
            dg.copy_(hg, non_blocking=True)
        for (dc, ds), (hc, hs) in zip(dtabs, htabs):
            dc.copy_(hc, non_blocking=True)
            ds.copy_(hs, non_blocking=True)
        for call in dev_calls:
            call()
        ox.copy_(dx, non_blocking=True)
        if has_bwd:
            og.copy_(dg, non_blocking=True)

    t_cp, gbs_cp = timed(copy_step)
    return {"value": round(gbs_zc, 2), "unit": "GB/s",
            "h2d_bytes_per_step": ndir * slice_bytes + r_bytes,
            "d2h_bytes_per_step": ndir * slice_bytes, "steps": steps,
            "ms_per_step": round(t_zc * 1e3, 3),
            "path": "zero copy: rope_partial_inplace_{fwd,bwd}_host on page-locked host tensors; "
                    "the kernel reads the slices and cos/sin over the host link and writes the "
                    "rotated slices back in place (one stream, synchronised at the end)",
            "copy_path": {"value": round(gbs_cp, 2), "unit": "GB/s",
                          "ms_per_step": round(t_cp * 1e3, 3),
                          "h2d_bytes_per_step": hx.nbytes * ndir + r_whole,
                          "d2h_bytes_per_step": hx.nbytes * ndir,
                          "path": "whole tensors copied host->device, the launches on device "
                                  "buffers, x and grad copied back (one stream)"}}


SECTIONS = {
    "fused_qk": lambda dev, peak, flush, l2: qk_breakdown(dev, peak, flush),
    "half_split": half_breakdown,
    "positions": positions_breakdown,
    "odd_start": odd_breakdown,
}


def run_section(name: str, case=None) -> int:
    """One part of the breakdown on cuda:0, alone, so that a profiler sees
    only its launches (with `case`, only its entries whose label holds it)."""
    global CASE
    CASE = case
    from place_partial_rope_gb300 import build
    build.build()
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    peak, _ = hbm_peak()
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    out = SECTIONS[name](device, peak, l2_flusher(device), l2)
    print(json.dumps({"section": name, "result": out}), flush=True)
    return 0


def reference_arm(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    w = synth.WORKLOADS[args.workload]
    x, r1, r2, g = synth.workload_inputs(w)
    base = time_oracle(w, x, r1, r2, g, steps=args.steps, warmup=args.warmup, budget_s=150.0)
    out = {"impl": "reference", "metric": METRIC, "value": round(base["value"], 4), "unit": "GB/s",
           "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(base["ms_per_step"], 3), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
           "data": "synthetic: seeded N(0,1) activations and gradients, base-10000 cos/sin table",
           "config": workload_config(w, torch.cuda.get_device_properties(0).L2_cache_size
                                     if torch.cuda.is_available() else 132 * 2**20),
           "cpu_baseline": {k: base[k] for k in ("value", "unit", "cores", "kind", "sample")},
           "e2e": {"value": round(base["value"], 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    out["cpu_baseline"]["value"] = out["value"]
    print(json.dumps(out), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--workload", choices=sorted(synth.WORKLOADS), default=HEADLINE,
                    help="named configuration a step runs (default: the largest)")
    ap.add_argument("--split", choices=["tokens", "replica"], default="tokens",
                    help="tokens (default): the ranks split one workload's tokens, B x world "
                         "batches under weak scaling; replica: every rank runs its own copy of "
                         "the named workload")
    ap.add_argument("--strong", action="store_true",
                    help="with --split tokens: split the named workload itself (strong scaling)")
    ap.add_argument("--section", choices=sorted(SECTIONS),
                    help="run only this part of the per-workload breakdown and print its JSON "
                         "(for profiling one kernel kind; not a bench line)")
    ap.add_argument("--case", help="with --section: only the entries whose label holds this text")
    args = ap.parse_args()
    if args.section:
        return run_section(args.section, args.case)
    if args.warmup < 3 and args.impl == "native":
        args.warmup = 3
    world = dist_env()[0]
    if args.gpus != world:
        print(f"bench.py: --gpus {args.gpus} but {world} rank(s) were launched (N > 1 runs under "
              f"torch.distributed.run with one rank per GPU); reporting the {world} that run",
              file=sys.stderr)
    if args.impl == "reference":
        return reference_arm(args)
    return gpu_arm(args)


if __name__ == "__main__":
    sys.exit(main())
