#!/usr/bin/env python3
"""Benchmark of the GB300 exact-attention path; prints ONE JSON line (rank 0).

A step is one fa_fwd call (the whole prefill path: tile scheduling, TMA loads,
S = QK^T, masking, online softmax, lazy O correction, P V, epilogue) over the
headline workload, the largest single-GPU one: the long causal MHA prefill
B=1, H=16, N=M=32768, d=128, bf16 (4.4 TFLOP per call); inputs (402 MB) are
resident in HBM and L2 is flushed (a 256 MiB write, then a 256 MiB read, so
that no dirty line is left to write back) between steps.
Each step is timed with CUDA events on the launching stream.  The line also
carries:
  roofline      the prefill kernel against the measured dense bf16 peak;
  e2e           the same metric through the public API with pinned host
                buffers, host->device inputs and device->host O/LSE inside the
                timed region;
  decode        split-KV decode (B=2, H=8, M=65536, d=128, chunk 128) in HBM
                GB/s against the measured copy bandwidth;
  workloads     every workload's time and roofline fraction;
  cpu_baseline  the fp64 CPU oracle, as it stands, on a bounded sample of
                the headline workload, and (per_config) of every workload,
                with the host's core count and CPU model;
  clocks        nvidia-smi samples taken during the timed regions.

--impl reference times the oracle (the only other implementation of the
method here) on the host cores, same metric and workload, a bounded sample per
step.  With --gpus N > 1 (torchrun, one process per GPU) every rank runs its
own replica of the workload (independent problems, no collective on the data
path): value = N * work / max-over-ranks time, scaling "weak".
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = ("fwd attention TFLOPS (4·B·H·N·M·d, causal halved) and decode "
          "HBM GB/s, % roofline")
HEADLINE = "prefill_causal_h16_n32768_bf16"
DECODE = "decode_b2_h8_m65536_f16"
FLUSH_BYTES = 256 << 20
L2_BYTES = 129 << 20      # GB300 L2; inputs larger than this need no flush between steps
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ---------------------------------------------------------------------------
# process group (torchrun) helpers -- host logic, testable with gloo on CPU
# ---------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, local, world


def init_dist(world: int, backend: str):
    if world <= 1:
        return None
    import torch.distributed as dist
    if not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(value: float, dist, device=None) -> float:
    """The largest value any rank holds (the job's time is its slowest rank's)."""
    if dist is None:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_throughput(units_per_rank: float, world: int, max_seconds: float) -> float:
    """Whole-job throughput: every rank's units over the slowest rank's time."""
    return units_per_rank * world / max_seconds


# ---------------------------------------------------------------------------
# peaks, clocks, traffic
# ---------------------------------------------------------------------------

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


KERNEL_SOURCES = {
    "prefill_kernel": ["fa_prefill.cu", "fa_device.cuh", "fa_internal.h"],
    "decode_chunk_kernel": ["fa_decode_kernel.cuh", "fa_decode.cu", "fa_device.cuh",
                            "fa_internal.h"],
    "decode_merge_kernel": ["fa_decode_kernel.cuh", "fa_decode.cu", "fa_device.cuh",
                            "fa_internal.h"],
    "backward_kernel": ["fa_backward.cu", "fa_device.cuh", "fa_internal.h"],
}


def _code_only(text: str) -> str:
    """C++ source without its comments and blank lines (string literals in these
    files hold no comment markers)."""
    import re
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def kernel_source_digest(kernel: str) -> str:
    """Short hash of the code (comments left out) of the files a kernel is
    compiled from: an edit to a comment does not void a recorded capture."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "exact_attention_05_gb300", "csrc")
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(name.encode())
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, kernel: str):
    """DRAM bytes per launch from the committed ncu summary, or None if absent or
    taken on a different version of the kernel sources."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    try:
        lines = open(path).read().splitlines()
    except OSError:
        return None
    digest = kernel_source_digest(kernel)
    for line in lines:
        parts = line.split()
        if len(parts) >= 4 and not line.startswith("#") and parts[0] == workload \
                and parts[1] == kernel and parts[2] == digest:
            return float(parts[3])
    return None


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples every 200 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.out = None

    def __enter__(self):
        self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.gpu)], stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        time.sleep(0.3)
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        self.out.flush()
        return False

    def summary(self):
        try:
            with open(self.out.name) as f:
                rows = [r.split(",") for r in f.read().splitlines() if r.strip()]
            os.unlink(self.out.name)
        except OSError:
            rows = []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        samples = []
        for r in rows:
            try:
                vals = [x.strip() for x in r]
                samples.append((float(vals[1]), float(vals[2]), float(vals[3]), float(vals[4]),
                                vals[5:9]))
            except (ValueError, IndexError):
                continue
        if not samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        loaded = [s for s in samples if s[3] >= 50.0] or samples
        reasons = sorted({names[i] for s in loaded for i, v in enumerate(s[4])
                          if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median(s[0] for s in loaded),
                "sm_max_mhz": max(s[1] for s in samples),
                "power_w_max": max(s[2] for s in samples),
                "reasons": reasons, "samples": len(samples), "samples_under_load": len(loaded)}


# ---------------------------------------------------------------------------
# GPU timing
# ---------------------------------------------------------------------------

def time_calls(torch, fn, steps, warmup, flush=None, dist=None):
    """Per-call device times (ms) with CUDA events on the current stream; the
    optional flush runs between calls, outside the event pairs."""
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        if flush is not None:
            flush()
        fn()
    torch.cuda.synchronize()
    barrier(dist)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for s, e in ev:
        if flush is not None:
            flush()
        s.record(stream)
        fn()
        e.record(stream)
    torch.cuda.synchronize()
    barrier(dist)
    torch.cuda.synchronize()
    return [s.elapsed_time(e) for s, e in ev]


def bench_prefill(torch, fa, w, steps, warmup, flush, dist=None):
    from exact_attention_05_gb300.workloads import workload_inputs
    q, k, v = (t.cuda() for t in workload_inputs(w))
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.Hq, w.N), dtype=torch.float32, device="cuda")

    def call():
        fa.fa_fwd(q, k, v, o, lse, w.B, w.Hq, w.Hkv, w.N, w.M, w.d, int(w.causal), w.scale,
                  w.dtype)

    times = time_calls(torch, call, steps, warmup, flush, dist)
    if fa.fa_get_last_device_status() != fa.FA_OK:
        raise RuntimeError(f"{w.name}: a device-side wait expired")
    return times


def bench_backward(torch, fa, w, steps, warmup, flush, dist=None):
    """fa_bwd on a prefill workload: O and LSE come from one untimed fa_fwd; dO is
    iid N(0, 1) in the workload's type.  Algorithmic FLOPs: 2.5x the forward's
    (five GEMMs of 2*N*M*d per head instead of two)."""
    from exact_attention_05_gb300.workloads import make_dout, workload_inputs
    q, k, v = (t.cuda() for t in workload_inputs(w))
    dout = make_dout(w.B, w.N, w.Hq, w.d, w.dtype, w.seed + 7).cuda()
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.Hq, w.N), dtype=torch.float32, device="cuda")
    fa.fa_fwd(q, k, v, o, lse, w.B, w.Hq, w.Hkv, w.N, w.M, w.d, int(w.causal), w.scale, w.dtype)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)

    def call():
        fa.fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, w.B, w.Hq, w.Hkv, w.N, w.M, w.d,
                  int(w.causal), w.scale, w.dtype)

    times = time_calls(torch, call, steps, warmup, flush, dist)
    if fa.fa_get_last_device_status() != fa.FA_OK:
        raise RuntimeError(f"{w.name}: a device-side wait expired (backward)")
    return times


def decode_call(torch, fa, w, single_launch=False):
    """Device-resident inputs of a decode workload and a zero-argument call of
    the entry point that serves it: fa_decode (or fa_decode_fused with
    ``single_launch``) for contiguous 16-bit K/V, fa_decode_fp8 for e4m3 K/V,
    fa_decode_paged for a paged cache."""
    from exact_attention_05_gb300.workloads import workload_decode_inputs
    host = workload_decode_inputs(w)
    if w.page > 0:
        host.pop("k")
        host.pop("v")
    x = {name: t.cuda() for name, t in host.items()}
    o = torch.empty_like(x["q"])
    lse = torch.empty((w.B, w.Hq), dtype=torch.float32, device="cuda")
    if w.kv == "e4m3":
        if single_launch:
            raise ValueError("the single launch is built for contiguous 16-bit K/V")
        return lambda: fa.fa_decode_fp8(x["q"], x["k"], x["v"], x["k_scale"], x["v_scale"], o,
                                        lse, w.B, w.Hq, w.Hkv, w.M, w.d, w.chunk, w.scale,
                                        w.dtype)
    if w.page > 0:
        if single_launch:
            raise ValueError("the single launch is built for contiguous 16-bit K/V")
        bt = x["block_table"]
        return lambda: fa.fa_decode_paged(x["q"], x["k_cache"], x["v_cache"], bt, x["seq_lens"],
                                          o, lse, w.B, w.Hq, w.Hkv, w.M,
                                          x["k_cache"].shape[0], w.page, bt.shape[1], w.d,
                                          w.chunk, w.scale, w.dtype)
    fn = fa.fa_decode_fused if single_launch else fa.fa_decode
    return lambda: fn(x["q"], x["k"], x["v"], o, lse, w.B, w.Hq, w.Hkv, w.M, w.d, w.chunk,
                      w.scale, w.dtype)


def bench_decode(torch, fa, w, steps, warmup, flush, dist=None, single_launch=False):
    call = decode_call(torch, fa, w, single_launch)
    times = time_calls(torch, call, steps, warmup, flush, dist)
    if fa.fa_get_last_device_status() != fa.FA_OK:
        raise RuntimeError(f"{w.name}: a device-side wait expired")
    return times


def bench_decode_single_launch(torch, fa, w, steps, warmup, flush, dist=None):
    return bench_decode(torch, fa, w, steps, warmup, flush, dist, single_launch=True)


def bench_e2e_decode(torch, fa, w, steps, warmup):
    """Public API with pinned host buffers: H2D of q/k/v, fa_decode, D2H of o/lse."""
    from exact_attention_05_gb300.workloads import workload_inputs
    qh, kh, vh = (t.pin_memory() for t in workload_inputs(w))
    qd, kd, vd = (torch.empty_like(t, device="cuda") for t in (qh, kh, vh))
    od = torch.empty_like(qd)
    lsed = torch.empty((w.B, w.Hq), dtype=torch.float32, device="cuda")
    oh = torch.empty_like(qh).pin_memory()
    lseh = torch.empty((w.B, w.Hq), dtype=torch.float32).pin_memory()

    def call():
        qd.copy_(qh, non_blocking=True)
        kd.copy_(kh, non_blocking=True)
        vd.copy_(vh, non_blocking=True)
        fa.fa_decode(qd, kd, vd, od, lsed, w.B, w.Hq, w.Hkv, w.M, w.d, w.chunk, w.scale, w.dtype)
        oh.copy_(od, non_blocking=True)
        lseh.copy_(lsed, non_blocking=True)

    times = time_calls(torch, call, steps, warmup)
    h2d = sum(t.numel() * t.element_size() for t in (qh, kh, vh))
    d2h = oh.numel() * oh.element_size() + lseh.numel() * lseh.element_size()
    return times, h2d, d2h


def bench_e2e_prefill(torch, fa, w, steps, warmup):
    """Public API on pinned host buffers: fa_fwd_host copies q/k/v in, runs the
    forward and copies o/lse back, chunk by chunk with the transfers overlapping
    the kernels; every byte crosses the link inside the timed region."""
    from exact_attention_05_gb300.workloads import workload_inputs
    qh, kh, vh = (t.pin_memory() for t in workload_inputs(w))
    oh = torch.empty_like(qh).pin_memory()
    lseh = torch.empty((w.B, w.Hq, w.N), dtype=torch.float32).pin_memory()

    def call():
        fa.fa_fwd_host(qh, kh, vh, oh, lseh, w.B, w.Hq, w.Hkv, w.N, w.M, w.d, int(w.causal),
                       w.scale, w.dtype)

    times = time_calls(torch, call, steps, warmup)
    h2d = sum(t.numel() * t.element_size() for t in (qh, kh, vh))
    d2h = oh.numel() * oh.element_size() + lseh.numel() * lseh.element_size()
    return times, h2d, d2h


# ---------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline and the reference arm)
# ---------------------------------------------------------------------------

def oracle_sample(w, heads: int, rows: int = 0):
    """A bounded sample of workload w for the oracle: batch 0, the first `heads`
    query heads (with their kv heads) and either every query row or, with
    `rows`, the first `rows` of them (with causal masking those rows see only
    keys 0..rows-1, so the sample is exactly that prefix of the workload).
    Returns a callable that runs it and the sample's algorithmic FLOPs (the
    workload's own convention: 4*rows*keys*d per head, halved when causal)."""
    import oracle
    from exact_attention_05_gb300.workloads import bits, workload_inputs
    q, k, v = workload_inputs(w)
    g = w.Hq // w.Hkv
    if heads % g:
        raise ValueError("sample must cover whole GQA groups")
    kvh = heads // g
    n = w.N if rows <= 0 else min(rows, w.N)
    m = min(n, w.M) if (w.causal and n < w.N) else w.M
    qs = bits(q[:1, :n, :heads].contiguous())
    ks = bits(k[:1, :m, :kvh].contiguous())
    vs = bits(v[:1, :m, :kvh].contiguous())
    flops = 4.0 * heads * n * m * w.d / (2.0 if w.causal else 1.0)

    def run():
        oracle.attention(qs, ks, vs, w.dtype, w.causal, w.scale)

    return run, flops


# Query rows per step of the reference arm: about a second of fp64 work on 16
# host cores (every row for the workloads smaller than that).
REFERENCE_ROWS = 16384


def cpu_model() -> str:
    """The host CPU's model name (lscpu on Arm hosts, /proc/cpuinfo elsewhere)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


def cpu_baseline(w, target_s: float = 12.0):
    """The oracle on a sample of prefill workload w: whole GQA groups of batch 0,
    every query row, as many groups as fit in about target_s seconds (at least one)."""
    import oracle
    oracle.build()
    g = w.Hq // w.Hkv
    run, flops = oracle_sample(w, g)
    t0 = time.perf_counter()
    run()
    t1 = time.perf_counter() - t0
    groups = max(1, min(w.Hq // g, int(target_s / max(t1, 1e-6))))
    heads = groups * g
    if heads > g:
        run, flops = oracle_sample(w, heads)
        t0 = time.perf_counter()
        run()
        t1 = time.perf_counter() - t0
    full = heads == w.Hq and w.B == 1
    return {"value": flops / t1 / 1e12, "unit": "TFLOP/s", "cores": oracle.num_threads(),
            "cpu": cpu_model(), "kind": "oracle", "seconds": t1,
            "seconds_full_workload": t1 * w.flops / flops,
            "full_workload_time": "measured" if full else "extrapolated by FLOPs",
            "sample": f"batch 0, query heads 0..{heads - 1} of {w.Hq} (all {w.N} rows), fp64, "
                      f"{t1:.2f} s"}


def cpu_baseline_decode(w):
    """The oracle on a whole 16-bit decode workload (its fp64 pass is short)."""
    import oracle
    from exact_attention_05_gb300.workloads import bits, workload_inputs
    oracle.build()
    q, k, v = workload_inputs(w)
    qb, kb, vb = bits(q), bits(k), bits(v)
    t0 = time.perf_counter()
    oracle.attention(qb, kb, vb, w.dtype, False, w.scale)
    t1 = time.perf_counter() - t0
    return {"value": w.decode_bytes / t1 / 1e9, "unit": "GB/s", "cores": oracle.num_threads(),
            "cpu": cpu_model(), "kind": "oracle", "seconds": t1,
            "seconds_full_workload": t1, "full_workload_time": "measured",
            "sample": f"the whole workload (B={w.B}, Hq={w.Hq}, M={w.M}), fp64, {t1:.2f} s"}


def cpu_baseline_all(target_s: float = 3.0):
    """The oracle timed on every 16-bit workload of the table (a bounded sample of
    each prefill workload, the whole of each decode workload)."""
    from exact_attention_05_gb300.workloads import WORKLOADS
    out = {}
    for name, wl in WORKLOADS.items():
        if wl.kv != "16bit" or wl.page:
            continue
        try:
            out[name] = cpu_baseline_decode(wl) if wl.kind == "decode" else \
                cpu_baseline(wl, target_s)
        except Exception as exc:  # the CPU leg never decides the GPU numbers
            out[name] = {"value": None, "sample": f"failed: {exc}"}
    return out


def latency_breakdown(torch, fa, flush, reps: int = 200):
    """Where the time of a small call goes, for the two latency-bound workloads
    (the N=256 prefill and the M=512 decode): the device time of one call after
    an L2 flush (CUDA events around it, as the table times it); the device time
    per call of `reps` calls back to back (events around all of them: the
    launches then overlap the previous kernel's tail); the host time to enqueue
    one call (the C entry point through the binding, no synchronisation); and
    the device time per replay of the same calls captured in a CUDA graph."""
    from exact_attention_05_gb300.workloads import WORKLOADS, workload_inputs
    out = {}
    for name in ("prefill_mha_n256_d64_f16", "decode_b1_h8_m512_f16"):
        w = WORKLOADS[name]
        if w.kind == "prefill":
            q, k, v = (t.cuda() for t in workload_inputs(w))
            o = torch.empty_like(q)
            lse = torch.empty((w.B, w.Hq, w.N), dtype=torch.float32, device="cuda")

            def call():
                fa.fa_fwd(q, k, v, o, lse, w.B, w.Hq, w.Hkv, w.N, w.M, w.d, int(w.causal),
                          w.scale, w.dtype)

            # the same call straight into the C ABI with the pointers and the stream
            # handle resolved once: the host cost of the library alone
            lib = fa.load_library()
            args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), w.B,
                    w.Hq, w.Hkv, w.N, w.M, w.d, int(w.causal), w.scale, w.dtype,
                    torch.cuda.current_stream().cuda_stream)

            def abi_call():
                lib.fa_fwd(*args)
            launches = 1
        else:
            call = decode_call(torch, fa, w)
            abi_call = None
            launches = 2
        single = statistics.median(time_calls(torch, call, 50, 5, flush))
        for _ in range(10):
            call()
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        for _ in range(reps):
            call()
        e.record()
        torch.cuda.synchronize()
        chained = s.elapsed_time(e) / reps
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(reps):
            call()
        host = (time.perf_counter() - t0) / reps * 1e3
        torch.cuda.synchronize()
        host_abi = None
        if abi_call is not None:
            t0 = time.perf_counter()
            for _ in range(reps):
                abi_call()
            host_abi = (time.perf_counter() - t0) / reps * 1e3
            torch.cuda.synchronize()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            call()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=side):  # the stream the warm-up call used
            for _ in range(10):
                call()
        graph.replay()
        torch.cuda.synchronize()
        s.record()
        for _ in range(reps // 10):
            graph.replay()
        e.record()
        torch.cuda.synchronize()
        graphed = s.elapsed_time(e) / (reps // 10 * 10)
        if fa.fa_get_last_device_status() != fa.FA_OK:
            raise RuntimeError(f"{name}: a device-side wait expired")
        out[name] = {"launches_per_call": launches, "flushed_single_call_us": single * 1e3,
                     "back_to_back_us_per_call": chained * 1e3,
                     "host_enqueue_us_per_call": host * 1e3,
                     "host_enqueue_abi_us_per_call": None if host_abi is None else host_abi * 1e3,
                     "cuda_graph_us_per_call": graphed * 1e3}
    return out


def run_reference(args, rank, world):
    """The reference arm: the oracle as it stands on the host cores."""
    if rank != 0:
        return 0
    import oracle
    from exact_attention_05_gb300.workloads import WORKLOADS, DTYPE_NAME
    oracle.build()
    w = WORKLOADS[args.workload]
    g = w.Hq // w.Hkv
    if w.kind == "decode":
        # one step is the whole decode workload (a short fp64 pass)
        from exact_attention_05_gb300.workloads import bits, workload_inputs
        q, k, v = workload_inputs(w)
        qb, kb, vb = bits(q), bits(k), bits(v)

        def run():
            oracle.attention(qb, kb, vb, w.dtype, False, w.scale)

        units, per, unit = w.decode_bytes, 1e9, "GB/s"
        sample = f"the whole workload (B={w.B}, Hq={w.Hq}, M={w.M}) per step, fp64"
    else:
        rows = REFERENCE_ROWS
        run, units = oracle_sample(w, g, rows)
        per, unit = 1e12, "TFLOP/s"
        n = min(rows, w.N)
        what = f"all {w.N} rows" if n == w.N else \
            f"query rows 0..{n - 1} of {w.N}, the causal prefix" if w.causal else \
            f"query rows 0..{n - 1} of {w.N}"
        sample = f"batch 0, query heads 0..{g - 1} of {w.Hq} ({what}) per step, fp64"
    for _ in range(max(0, args.warmup)):
        run()
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        run()
        times.append(time.perf_counter() - t0)
    mean_s = sum(times) / len(times)
    value = units / mean_s / per
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": unit,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": mean_s * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w),
        "cpu_baseline": {"value": value, "unit": unit, "cores": oracle.num_threads(),
                         "cpu": cpu_model(), "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config(w):
    from exact_attention_05_gb300.workloads import DTYPE_NAME
    cfg = {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "N": w.N, "M": w.M, "d": w.d,
           "dtype": DTYPE_NAME[w.dtype], "causal": w.causal, "scale": w.scale}
    if w.kind == "decode":
        cfg["chunk"] = w.chunk
        if w.kv != "16bit":
            cfg["kv"] = w.kv
        if w.page:
            cfg["page"] = w.page
    if w.peaky_frac:
        cfg["peaky_k_rows"] = w.peaky_frac
    return cfg


# ---------------------------------------------------------------------------
# main
# ---------------------------------------------------------------------------

def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    from exact_attention_05_gb300.workloads import WORKLOADS as _W
    headline_ok = sorted(n for n, x in _W.items() if x.kv == "16bit" and x.page == 0)
    ap.add_argument("--workload", default=HEADLINE, choices=headline_ok,
                    help="the timed workload (the FP8 and paged decode workloads are timed "
                         "in the per-workload table)")
    ap.add_argument("--profile", choices=["prefill", "backward", "decode", "decode_single",
                                          "decode_fp8", "decode_paged"],
                    default=None,
                    help="run only --warmup + --steps calls of one operation on --workload "
                         "(or the long decode workload; decode_fp8 and decode_paged take the "
                         "long e4m3 and paged decode workloads) and print nothing else: the "
                         "command the ncu summaries under profiles/ are taken with")
    ap.add_argument("--latency", action="store_true",
                    help="print only the latency breakdown of the two small workloads "
                         "(flushed single call, back-to-back calls, host enqueue, CUDA graph)")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the per-workload table, decode line and CPU baseline")
    args = ap.parse_args(argv)
    rank, local, world = dist_env()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3

    if args.impl == "reference":
        return run_reference(args, rank, world)

    import torch
    import exact_attention_05_gb300 as fa
    from exact_attention_05_gb300 import build as fa_build
    from exact_attention_05_gb300.workloads import WORKLOADS

    torch.cuda.set_device(local)
    dist = init_dist(world, "nccl")
    if rank == 0 or not os.path.exists(fa_build.LIB_PATH):
        fa_build.build()
    barrier(dist)
    fa.load_library()
    peaks, peak_src = load_peaks()
    w = WORKLOADS[args.workload]
    flush_buf = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    flush_read = torch.zeros(FLUSH_BYTES // 4, dtype=torch.int32, device="cuda")
    flush_ctr = [0]

    def flush():
        # write a buffer larger than L2, then read another one: L2 is left
        # holding clean lines of neither input, so the timed call neither hits
        # its inputs in L2 nor pays for writing back the flush's dirty lines
        flush_ctr[0] = (flush_ctr[0] + 1) & 0xFF
        flush_buf.fill_(flush_ctr[0])
        flush_read.max()

    if args.latency:
        if rank == 0:
            print(json.dumps({"latency": latency_breakdown(torch, fa, flush)}), flush=True)
        if dist is not None:
            dist.destroy_process_group()
        return 0

    if args.profile is not None:
        wp = WORKLOADS[DECODE] if args.profile.startswith("decode") and w.kind != "decode" else w
        if args.profile == "decode_fp8":
            wp = WORKLOADS["decode_fp8_b2_h8_m65536_f16"]
        elif args.profile == "decode_paged":
            wp = WORKLOADS["decode_paged_b2_h8_m65536_p16_f16"]
        fn = {"prefill": bench_prefill, "backward": bench_backward, "decode": bench_decode,
              "decode_single": bench_decode_single_launch, "decode_fp8": bench_decode,
              "decode_paged": bench_decode}[args.profile]
        times = fn(torch, fa, wp, args.steps, args.warmup, flush, dist)
        if rank == 0:
            print(f"profile {args.profile} {wp.name}: {len(times)} timed calls, "
                  f"median {statistics.median(times) * 1e3:.1f} us", flush=True)
        if dist is not None:
            dist.destroy_process_group()
        return 0

    is_decode = w.kind == "decode"
    # work units of one step: FLOPs (prefill) or HBM bytes (decode), and their scale
    units, per = (w.decode_bytes, 1e9) if is_decode else (w.flops, 1e12)
    extras = {}
    with ClockSampler(torch.cuda.current_device()) as clocks:
        if is_decode:
            times = bench_decode(torch, fa, w, args.steps, args.warmup,
                                 flush if units < 2 * L2_BYTES else None, dist)
        else:
            times = bench_prefill(torch, fa, w, args.steps, args.warmup, flush, dist)
        mean_ms = sum(times) / len(times)
        mean_ms_max = max_over_ranks(mean_ms, dist, device="cuda")
        value = aggregate_throughput(units, world, mean_ms_max * 1e-3) / per

        e2e_steps = max(3, min(args.steps, 20))
        e2e_fn = bench_e2e_decode if is_decode else bench_e2e_prefill
        e2e_times, h2d, d2h = e2e_fn(torch, fa, w, e2e_steps, 3)
        e2e_ms = max_over_ranks(sum(e2e_times) / len(e2e_times), dist, device="cuda")
        e2e_value = aggregate_throughput(units, world, e2e_ms * 1e-3) / per

        if not args.no_extras:
            wd = WORKLOADS[DECODE]
            dt = bench_decode(torch, fa, wd, max(3, min(args.steps, 50)), 3, None, dist)
            d_ms = max_over_ranks(sum(dt) / len(dt), dist, device="cuda")
            d_gbs = wd.decode_bytes / (d_ms * 1e-3) / 1e9
            extras["decode"] = {
                "workload": wd.name, "ms_per_call": d_ms, "value": d_gbs * world,
                "unit": "GB/s", "launches_per_call": 2,
                "roofline": {"bound": "hbm", "achieved": d_gbs, "peak": peaks["hbm_gbs"],
                             "unit": "GB/s", "frac": d_gbs / peaks["hbm_gbs"],
                             "traffic": recorded_traffic(wd.name, "decode_chunk_kernel"),
                             "peak_source": peak_src,
                             "note": "achieved over the whole call (chunk + merge kernels)"},
            }
            st = bench_decode_single_launch(torch, fa, wd, max(3, min(args.steps, 50)), 3, None,
                                            dist)
            s_ms = max_over_ranks(sum(st) / len(st), dist, device="cuda")
            s_gbs = wd.decode_bytes / (s_ms * 1e-3) / 1e9
            extras["decode"]["single_launch"] = {
                "ms_per_call": s_ms, "value": s_gbs * world, "unit": "GB/s",
                "launches_per_call": 1, "frac": s_gbs / peaks["hbm_gbs"]}
            table = {}
            for name, wl in WORKLOADS.items():
                n = max(3, min(args.steps, 20 if wl.flops < 1e12 else 5))
                if wl.kind == "prefill":
                    tt = bench_prefill(torch, fa, wl, n, 3, flush if wl.flops < 1e12 else None,
                                       dist)
                    ms = max_over_ranks(statistics.median(tt), dist, device="cuda")
                    tf = wl.flops / (ms * 1e-3) / 1e12
                    table[name] = {"ms": ms, "TFLOP/s": tf, "frac": tf / peaks["bf16_tflops"]}
                    tb = bench_backward(torch, fa, wl, n, 3, flush if wl.flops < 1e12 else None,
                                        dist)
                    msb = max_over_ranks(statistics.median(tb), dist, device="cuda")
                    tfb = 2.5 * wl.flops / (msb * 1e-3) / 1e12
                    table[name]["backward"] = {"ms": msb, "TFLOP/s": tfb,
                                               "frac": tfb / peaks["bf16_tflops"],
                                               "launches_per_call": 3}
                else:
                    fl = flush if wl.decode_bytes < 2 * L2_BYTES else None
                    tt = bench_decode(torch, fa, wl, n, 3, fl, dist)
                    ms = max_over_ranks(statistics.median(tt), dist, device="cuda")
                    gbs = wl.decode_bytes / (ms * 1e-3) / 1e9
                    table[name] = {"ms": ms, "GB/s": gbs, "frac": gbs / peaks["hbm_gbs"],
                                   "kv": wl.kv, "page": wl.page}
                    if wl.kv != "e4m3" and wl.page == 0:
                        ts = bench_decode_single_launch(torch, fa, wl, n, 3, fl, dist)
                        ms1 = max_over_ranks(statistics.median(ts), dist, device="cuda")
                        gbs1 = wl.decode_bytes / (ms1 * 1e-3) / 1e9
                        table[name]["single_launch"] = {"ms": ms1, "GB/s": gbs1,
                                                        "frac": gbs1 / peaks["hbm_gbs"]}
            extras["workloads"] = table
    clk = clocks.summary()

    if rank == 0 and world == 1 and not args.no_extras:
        try:
            extras["cpu_baseline"] = cpu_baseline_decode(w) if is_decode else cpu_baseline(w)
        except Exception as exc:  # the CPU leg never decides the GPU numbers
            extras["cpu_baseline"] = {"value": None, "unit": "GB/s" if is_decode else "TFLOP/s",
                                      "cores": None, "kind": "oracle", "sample": f"failed: {exc}"}
        extras["cpu_baseline"]["per_config"] = cpu_baseline_all()

    from exact_attention_05_gb300.workloads import DTYPE_NAME
    achieved = units / (mean_ms_max * 1e-3) / per
    if is_decode:
        unit = "GB/s"
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": unit,
                "frac": achieved / peaks["hbm_gbs"],
                "traffic": recorded_traffic(w.name, "decode_chunk_kernel"),
                "peak_source": f"{peak_src} HBM copy",
                "note": "achieved over the whole call (chunk + merge kernels)"}
        l2 = "inputs larger than L2 (K/V vs 129 MB), no flush" if units >= 2 * L2_BYTES else \
            "flushed between steps (256 MiB write, then 256 MiB read)"
        launches = 2 * args.steps
    else:
        unit = "TFLOP/s"
        roof = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"],
                "unit": unit, "frac": achieved / peaks["bf16_tflops"],
                "traffic": recorded_traffic(w.name, "prefill_kernel"),
                "peak_source": f"{peak_src} dense bf16 burst"}
        l2 = "flushed between steps (256 MiB write, then 256 MiB read)"
        launches = args.steps
    line = {
        "metric": METRIC,
        "value": value,
        "unit": unit,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": mean_ms_max,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": DTYPE_NAME[w.dtype],
        "data": "synthetic",
        "config": dict(workload_config(w), l2=l2, parallelism=f"replicas x{world}"),
        "roofline": roof,
        "e2e": {"value": e2e_value, "unit": unit, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": launches,
        "clocks": clk,
    }
    line.update(extras)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
