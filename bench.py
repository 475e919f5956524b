#!/usr/bin/env python3
"""Benchmark of the attention forward hot path on GB300.

One step = one attn_fwd call through the C ABI (the persistent forward kernel
plus, when the schedule splits key ranges, the combine kernel) over one batch
of synthetic inputs already resident in HBM.  The default workload is the
single-head L = 8192, d = 128 causal BF16 problem (page S23-J17 §3 table);
``--workload`` picks another of tiled_attention_attn_gb300.inputs.WORKLOADS.

Metric: attention forward TFLOP/s, causal-adjusted (4 * d * Hq * sum over
sequences of Lq * Lk, halved when causal), and its fraction of the measured
dense BF16 tensor peak.

Timing: W warm-up steps, then K timed steps bracketed by a barrier and a
device synchronisation.  The inputs (6 MiB for the default workload) fit in
L2, so a 256 MiB buffer is written before every step and each step is timed
with its own pair of CUDA events on the launching stream (the flush is
outside the events).  Clocks are sampled with nvidia-smi during the timed
steps.  Further legs: the main kernel's own duration (library profiling
events) for the roofline; an end-to-end leg through pinned host buffers
(host->device copies of q, k, v and device->host copies of O and lse inside
the timed region); and, on rank 0 at N = 1, the fp64 CPU oracle timed on a
bounded sample of the same workload.

``--impl reference`` times the oracle alone, as the reference arm.
N > 1 (torchrun): every rank runs an independent replica of the workload
(the forward pass has no exchange step); value = all ranks' FLOPs / the
slowest rank's time.
"""

from __future__ import annotations

import argparse
import glob
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from tiled_attention_attn_gb300.inputs import HEADLINE, WORKLOADS, generate  # noqa: E402

METRIC = "attn fwd TFLOP/s (causal-adjusted) and % of GB300 dense BF16 tensor peak"
UNIT = "TFLOP/s"
FLUSH_BYTES = 256 * 1024 * 1024          # > 129 MB L2
FALLBACK_PEAK = {"bf16_tflops": 1900.0, "hbm_gbs": 6800.0}
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "attn_fwd_kernel_l8192_d128_causal.ncu.txt")


# ---------------------------------------------------------------------------
# workload accounting
# ---------------------------------------------------------------------------

def workload_flops(wl, lengths=None) -> float:
    """Causal-adjusted FLOPs: 4 * d per (query, key) pair, pairs halved when causal."""
    if wl.varlen:
        pairs = sum(n * n for n in lengths)
    else:
        pairs = wl.B * wl.Lq * wl.Lk
    if wl.causal:
        pairs *= 0.5
    return 4.0 * wl.d * wl.Hq * pairs


def workload_bytes(wl, lengths=None) -> float:
    """Algorithmic HBM bytes: Q, K, V read once, O written once (input dtype), lse (fp32)."""
    rows_q = sum(lengths) if wl.varlen else wl.B * wl.Lq
    rows_k = sum(lengths) if wl.varlen else wl.B * wl.Lk
    return 2.0 * wl.d * (2 * rows_q * wl.Hq + 2 * rows_k * wl.Hkv) + 4.0 * rows_q * wl.Hq


def sample_flops(wl, rows) -> float:
    """Exact FLOPs of the oracle's work on sampled rows (4 * d per allowed key)."""
    tot = 0
    for (b, h, i) in rows:
        n = wl.Lk if not wl.causal else min(wl.Lk, i + (wl.Lk - wl.Lq) + 1)
        tot += max(n, 0)
    return 4.0 * wl.d * tot


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"bf16_tflops": float(d["bf16_tflops"]), "hbm_gbs": float(d["hbm_gbs"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAK, bf16_tflops_sustained=1700.0, source="fallback")


# the files the forward kernel and its launch are built from (the profile of
# the forward kernel under profiles/ records their hash)
FWD_SOURCES = ("attn_kernel.cuh", "attn_kernels.inc", "attn_kernels_d64.cu", "attn_kernels_d128.cu", "attn_params.h",
               "attn_launch.h", "attn_host.cu", "attn_plan.cpp", "attn_plan.h", "ptx.cuh", "tmem_regs.cuh",
               "attn_cache.h", "attn_pair_launch.h")


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for p in sorted(os.path.join(ROOT, "tiled_attention_attn_gb300", "csrc", f) for f in FWD_SOURCES):
        with open(p, "rb") as f:
            h.update(os.path.basename(p).encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic():
    """DRAM bytes per launch of the main kernel from the committed ncu summary,
    if it was taken on the current kernel sources (else None)."""
    try:
        kv = {}
        with open(PROFILE_SUMMARY) as f:
            for line in f:
                if ":" in line and not line.startswith("#"):
                    k, v = line.split(":", 1)
                    kv[k.strip()] = v.strip()
        if kv.get("kernel_source_sha256") != kernel_source_hash():
            return None
        return float(kv["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: str):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(1.0)   # nvidia-smi start-up
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, which):
        if which == "begin":
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sel = [l for (t, l) in self.lines if self.t0 is not None and self.t0 - 0.05 <= t <= self.t1 + 0.05]
        mhz, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in sel:
            parts = [p.strip() for p in l.split(",")]
            if len(parts) < 9:
                continue
            try:
                mhz.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(mhz) if mhz else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(mhz)}


def gpu_index_for(local_rank: int) -> str:
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        ids = [x.strip() for x in vis.split(",") if x.strip()]
        if local_rank < len(ids):
            return ids[local_rank]
    return str(local_rank)


def head_start(n_steps: int) -> float:
    """Keeps the device ahead of the host through a timed loop that does not
    synchronise per step: a device-side sleep enqueued just before the loop,
    outside every step's events.  Without it a host stall longer than the L2
    flush (an NVML query of the clock sampler holds the driver for tens of
    microseconds) lets the device reach a step's start event before the
    step's kernels are enqueued, and that idle time is counted in the step.
    Returns the sleep in milliseconds."""
    seconds = min(0.2, 1e-3 + n_steps * 1e-4)
    torch.cuda._sleep(int(seconds * 2.0e9))
    return seconds * 1e3


# ---------------------------------------------------------------------------
# distributed plumbing (replicas only)
# ---------------------------------------------------------------------------

def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
        return dist, world, rank, local
    return None, 1, 0, 0


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(dist, x: float, device) -> float:
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# the CPU oracle on a bounded sample
# ---------------------------------------------------------------------------

def oracle_sample(wl, inp, budget_s: float, max_rows: int = 400000, seed: int = 99):
    """Times the oracle on sampled rows of the workload for about budget_s
    seconds; returns (TFLOP/s, seconds, n_rows, threads)."""
    import oracle

    oracle.build()
    q = oracle.f64(inp.q)
    k = oracle.f64(inp.k)
    v = oracle.f64(inp.v)
    rng = np.random.default_rng(seed)

    def rows_of(n):
        b = rng.integers(0, wl.B, n)
        h = rng.integers(0, wl.Hq, n)
        i = rng.integers(0, wl.Lq, n)
        return [(int(x), int(y), int(z)) for x, y, z in zip(b, h, i)]

    threads = oracle.num_threads()
    # calibrate on 32 rows per thread (fewer leave the call overhead dominant)
    cal = rows_of(max(threads, 1) * 32)
    t0 = time.perf_counter()
    oracle.attention_rows(q, k, v, cal, causal=wl.causal, scale=wl.softmax_scale)
    t_cal = max(time.perf_counter() - t0, 1e-6)
    n = int(min(max_rows, max(threads, len(cal) * budget_s / t_cal)))
    rows = rows_of(n)
    t0 = time.perf_counter()
    oracle.attention_rows(q, k, v, rows, causal=wl.causal, scale=wl.softmax_scale)
    dt = time.perf_counter() - t0
    return sample_flops(wl, rows) / dt / 1e12, dt, n, threads


def workload_config(wl, lengths=None) -> dict:
    cfg = {"workload": wl.name, "B": wl.B, "Hq": wl.Hq, "Hkv": wl.Hkv, "d": wl.d,
           "causal": wl.causal, "scale": wl.softmax_scale}
    if wl.varlen:
        cfg.update({"varlen": True, "lengths": "U[%d,%d]" % (wl.len_lo, wl.len_hi), "total_tokens": sum(lengths)})
    else:
        cfg.update({"Lq": wl.Lq, "Lk": wl.Lk})
    return cfg


# ---------------------------------------------------------------------------
# arms
# ---------------------------------------------------------------------------

def run_reference(args, wl):
    dist, world, rank, local = dist_setup(args.gpus)
    if rank != 0:
        return 0
    import oracle

    inp = generate(wl)
    oracle.build()
    q, k, v = oracle.f64(inp.q), oracle.f64(inp.k), oracle.f64(inp.v)
    rng = np.random.default_rng(7)
    steps, warm = args.steps, args.warmup
    # size each step's sample so that the whole run stays within a few minutes
    budget_per_step = min(2.0, 150.0 / max(steps + warm, 1))
    cal = [(0, 0, wl.Lq - 1)]
    t0 = time.perf_counter()
    oracle.attention_rows(q, k, v, cal, causal=wl.causal, scale=wl.softmax_scale)
    t_row = max(time.perf_counter() - t0, 1e-6)
    rows_per_step = max(1, int(budget_per_step / t_row))

    def step():
        b = rng.integers(0, wl.B, rows_per_step)
        h = rng.integers(0, wl.Hq, rows_per_step)
        i = rng.integers(0, wl.Lq, rows_per_step)
        rows = [(int(x), int(y), int(z)) for x, y, z in zip(b, h, i)]
        oracle.attention_rows(q, k, v, rows, causal=wl.causal, scale=wl.softmax_scale)
        return sample_flops(wl, rows)

    for _ in range(warm):
        step()
    t0 = time.perf_counter()
    fl = 0.0
    for _ in range(steps):
        fl += step()
    dt = time.perf_counter() - t0
    value = fl / dt / 1e12
    threads = oracle.num_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": steps, "warmup": warm, "ms_per_step": dt / steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(wl),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": f"{rows_per_step} random query rows per step of {wl.name}, fp64, "
                                   f"S and P rows materialised"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


PAD_SHAPE = (64, 4096, 16, 128)   # B, L, H, d of the padded-batch leg: 1 GiB of bf16, larger than L2


def pad_leg(attn, device, stream, peaks, iters: int = 20):
    """The padded-batch kernels on a padded bf16 batch (B 64, L 4096, H 16,
    d 128; lengths uniform in [L/2, L] from a fixed seed): the unpad index,
    the gather of the kept rows into the packed layout and the scatter back.
    Bound: HBM.  Algorithmic bytes of a gather or scatter: each kept row read
    once and written once, plus its 4-byte index."""
    B, L, H, d = PAD_SHAPE
    g = torch.Generator().manual_seed(77)
    lengths = torch.randint(L // 2, L + 1, (B,), generator=g)
    mask = (torch.arange(L)[None, :] < lengths[:, None]).to(device)
    x = torch.randn(B * L, H, d, device=device, dtype=torch.bfloat16)
    cu, idx = attn.unpad_index(mask, stream)
    n_dev = cu[B:]
    packed = torch.empty_like(x)
    back = torch.zeros_like(x)
    kept = int(lengths.sum())
    row = H * d * 2
    moved = kept * (2 * row + 4)

    def timed(fn):
        fn()
        torch.cuda.synchronize(device)
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        for _ in range(iters):
            fn()
        e.record(stream)
        torch.cuda.synchronize(device)
        return s.elapsed_time(e) / iters

    t_idx = timed(lambda: attn.unpad_index(mask, stream))
    t_g = timed(lambda: attn.gather_rows(x, idx, n_dev, B * L, out=packed, stream=stream))
    t_s = timed(lambda: attn.scatter_rows(packed, idx, n_dev, back, stream=stream))
    gbs_g = moved / (t_g / 1e3) / 1e9
    gbs_s = moved / (t_s / 1e3) / 1e9
    return {"workload": f"padded bf16 B{B} L{L} H{H} d{d}, {kept} kept rows of {B * L}",
            "bound": "hbm", "unit": "GB/s", "peak": peaks["hbm_gbs"],
            "gather": {"achieved": gbs_g, "frac": gbs_g / peaks["hbm_gbs"], "ms": t_g},
            "scatter": {"achieved": gbs_s, "frac": gbs_s / peaks["hbm_gbs"], "ms": t_s},
            "unpad_index_ms": t_idx, "algorithmic_bytes_per_launch": moved}


CACHE_SHAPE = (16, 16, 4, 128)   # B, Hq, Hkv, d of the key/value-cache leg
ROTARY_SHAPE = (2, 8192, 32, 128)   # B, L, H, d of the rotary leg: 128 MiB of bf16


def rotary_leg(attn, device, stream, peaks, iters: int = 20):
    """attn_rotary in place on a (B 2, L 8192, H 32, d 128) bf16 tensor with
    full rotary dimension (GPT-NeoX pairing).  Bound: HBM; algorithmic bytes
    = the tensor read once and written once."""
    B, L, H, d = ROTARY_SHAPE
    x = torch.randn(B, L, H, d, device=device, dtype=torch.bfloat16)
    attn.rotary(x, out=x, stream=stream)
    torch.cuda.synchronize(device)
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(stream)
    for _ in range(iters):
        attn.rotary(x, out=x, stream=stream)
    e.record(stream)
    torch.cuda.synchronize(device)
    ms = s.elapsed_time(e) / iters
    moved = 2 * x.numel() * x.element_size()
    gbs = moved / (ms / 1e3) / 1e9
    return {"workload": f"rotary in place, bf16 B{B} L{L} H{H} d{d}", "bound": "hbm", "achieved": gbs,
            "unit": "GB/s", "peak": peaks["hbm_gbs"], "frac": gbs / peaks["hbm_gbs"], "ms": ms,
            "algorithmic_bytes_per_launch": moved}


def cache_leg(attn, device, stream, peaks, iters: int = 20):
    """Queries extending a key/value cache through attn_fwd_varlen: B 16
    sequences of Lq_b ~ U[64, 512] new tokens over Lk_b = Lq_b + cache_b keys
    (cache_b ~ U[0, 4096]), GQA 16/4, d 128, bf16, causal (bottom-right).
    FLOPs: 4 * d * Hq * (allowed query-key pairs, counted exactly).  Inputs
    (~21 MB) fit in L2, so each timed call follows a 256 MiB buffer write."""
    B, Hq, Hkv, d = CACHE_SHAPE
    g = torch.Generator().manual_seed(88)
    lq = torch.randint(64, 513, (B,), generator=g)
    cache = torch.randint(0, 4097, (B,), generator=g)
    lk = lq + cache
    q = torch.randn(int(lq.sum()), Hq, d, generator=g).to(torch.bfloat16).to(device)
    k = torch.randn(int(lk.sum()), Hkv, d, generator=g).to(torch.bfloat16).to(device)
    v = torch.randn(int(lk.sum()), Hkv, d, generator=g).to(torch.bfloat16).to(device)
    cu_q = torch.tensor([0] + torch.cumsum(lq, 0).tolist(), dtype=torch.int32, device=device)
    cu_k = torch.tensor([0] + torch.cumsum(lk, 0).tolist(), dtype=torch.int32, device=device)
    pairs = sum(int(a) * int(c) + int(a) * (int(a) + 1) // 2 for a, c in zip(lq, cache))
    flops = 4.0 * d * Hq * pairs
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=device)
    o, lse = attn.attn_fwd(q, k, v, causal=True, cu_seqlens=cu_q, cu_seqlens_k=cu_k, stream=stream)
    torch.cuda.synchronize(device)
    ms = []
    for _ in range(iters):
        flush.zero_()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        attn.attn_fwd(q, k, v, causal=True, cu_seqlens=cu_q, cu_seqlens_k=cu_k, out=o, lse=lse, stream=stream)
        e.record(stream)
        torch.cuda.synchronize(device)
        ms.append(s.elapsed_time(e))
    t = statistics.median(ms)
    tf = flops / (t / 1e3) / 1e12
    return {"workload": f"kv cache: B{B} Hq{Hq} Hkv{Hkv} d{d} bf16 causal, Lq~U[64,512], cache~U[0,4096]",
            "value": tf, "unit": "TFLOP/s", "frac": tf / peaks["bf16_tflops"], "ms": t,
            "flops_per_call": flops, "query_tokens": int(lq.sum()), "key_tokens": int(lk.sum())}


BWD_SHAPE = (2, 32, 8, 4096, 128)   # B, Hq, Hkv, L, d of the backward leg (causal, bf16)


def bwd_leg(attn, device, stream, peaks, iters: int = 10):
    """attn_bwd on B 2, Hq 32, Hkv 8, L 4096, d 128, bf16, causal (the
    grouped-query training shape), after attn_fwd on the same inputs.  FLOPs
    counted as the five algorithmic contractions of the backward (S, dP, dv,
    dk, dq: 2.5 x the forward's 4 d per allowed pair, causal half); the
    kernels execute seven (S and dP are formed once for dk/dv and again for
    dq), reported beside it.  L2 flushed before every timed call."""
    B, Hq, Hkv, L, d = BWD_SHAPE
    g = torch.Generator().manual_seed(77)
    q = torch.randn(B, L, Hq, d, generator=g).to(torch.bfloat16).to(device)
    k = torch.randn(B, L, Hkv, d, generator=g).to(torch.bfloat16).to(device)
    v = torch.randn(B, L, Hkv, d, generator=g).to(torch.bfloat16).to(device)
    do = torch.randn(B, L, Hq, d, generator=g).to(torch.bfloat16).to(device)
    o, lse = attn.attn_fwd(q, k, v, causal=True, stream=stream)
    dq, dk, dv = attn.attn_bwd(q, k, v, o, lse, do, causal=True, stream=stream)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=device)
    torch.cuda.synchronize(device)
    ms = []
    for _ in range(iters):
        flush.zero_()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        attn.attn_bwd(q, k, v, o, lse, do, causal=True, dq=dq, dk=dk, dv=dv, stream=stream)
        e.record(stream)
        torch.cuda.synchronize(device)
        ms.append(s.elapsed_time(e))
    if attn.get_error() != attn.ATTN_OK:
        raise RuntimeError(f"device error in the backward leg: {attn.last_device_error():#x}")
    t = statistics.median(ms)
    fwd_flops = 4.0 * d * Hq * B * L * L / 2
    flops = 2.5 * fwd_flops
    tf = flops / (t / 1e3) / 1e12
    out = {"workload": f"backward: B{B} Hq{Hq} Hkv{Hkv} L{L} d{d} bf16 causal", "value": tf, "unit": "TFLOP/s",
           "frac": tf / peaks["bf16_tflops"], "ms": t, "algorithmic_flops_per_call": flops,
           "executed_flops_per_call": 3.5 * fwd_flops,
           "executed_tflops": 3.5 * fwd_flops / (t / 1e3) / 1e12}
    del q, k, v, do, o, lse, dq, dk, dv
    # the packed (varlen) backward: 8 sequences of U[1024, 4096] tokens, same heads and d;
    # FLOPs 10 d Hq per allowed pair, counted exactly (causal: L_b (L_b + 1) / 2 pairs)
    lens = torch.randint(1024, 4097, (8,), generator=g)
    tot = int(lens.sum())
    qv = torch.randn(tot, Hq, d, generator=g).to(torch.bfloat16).to(device)
    kv = torch.randn(tot, Hkv, d, generator=g).to(torch.bfloat16).to(device)
    vv = torch.randn(tot, Hkv, d, generator=g).to(torch.bfloat16).to(device)
    dov = torch.randn(tot, Hq, d, generator=g).to(torch.bfloat16).to(device)
    cu = torch.tensor([0] + torch.cumsum(lens, 0).tolist(), dtype=torch.int32, device=device)
    ov, lsev = attn.attn_fwd(qv, kv, vv, causal=True, cu_seqlens=cu, stream=stream)
    grads = attn.attn_bwd(qv, kv, vv, ov, lsev, dov, causal=True, cu_seqlens=cu, stream=stream)
    torch.cuda.synchronize(device)
    msv = []
    for _ in range(iters):
        flush.zero_()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        attn.attn_bwd(qv, kv, vv, ov, lsev, dov, causal=True, cu_seqlens=cu, dq=grads[0], dk=grads[1], dv=grads[2],
                      stream=stream)
        e.record(stream)
        torch.cuda.synchronize(device)
        msv.append(s.elapsed_time(e))
    if attn.get_error() != attn.ATTN_OK:
        raise RuntimeError(f"device error in the varlen backward leg: {attn.last_device_error():#x}")
    tv = statistics.median(msv)
    pairs = sum(int(n) * (int(n) + 1) // 2 for n in lens)
    fv = 10.0 * d * Hq * pairs
    out["varlen"] = {"workload": f"varlen backward: 8 sequences of U[1024,4096] ({tot} tokens), Hq{Hq} Hkv{Hkv} "
                                 f"d{d} bf16 causal", "value": fv / (tv / 1e3) / 1e12, "unit": "TFLOP/s",
                     "frac": fv / (tv / 1e3) / 1e12 / peaks["bf16_tflops"], "ms": tv,
                     "algorithmic_flops_per_call": fv}
    return out


DECODE_SHAPE = (32, 32, 8, 128, 4096)      # B, Hq, Hkv, d, cache length of the decode leg
DECODE_LONG_SHAPE = (1, 32, 8, 128, 131072)   # one sequence with a long cache
DECODE_D64_SHAPES = ((32, 32, 8, 64, 4096), (1, 32, 8, 64, 131072))   # the same at head_dim 64


def decode_inputs(device, shape):
    """q (B, Hq, d), packed caches k, v (B (C + 1), Hkv, d) bf16 N(0, 1), and
    the query and key offsets of a decoding step of ``shape``."""
    B, Hq, Hkv, d, C = shape
    g = torch.Generator().manual_seed(66)
    q = torch.randn(B, Hq, d, generator=g).to(torch.bfloat16).to(device)
    k = torch.randn(B * (C + 1), Hkv, d, generator=g).to(torch.bfloat16).to(device)
    v = torch.randn(B * (C + 1), Hkv, d, generator=g).to(torch.bfloat16).to(device)
    cu_q = torch.arange(0, B + 1, dtype=torch.int32, device=device)
    cu_k = torch.arange(0, B + 1, dtype=torch.int32, device=device) * (C + 1)
    return q, k, v, cu_q, cu_k


def decode_step_times(attn, device, stream, shape, iters: int = 20, no_flush: bool = False):
    """Median CUDA-event times (ms) of one decoding step, one new token per
    sequence over a cache of C tokens (+ the new one), through attn_decode
    and through attn_fwd_varlen; L2 flushed before each call.  With
    ``no_flush`` also the time of attn_decode in back-to-back calls with no
    flush between them (the caches are larger than L2), as a fifth value: the
    flush leaves up to L2's size of dirty lines whose write-back the next
    kernel shares HBM with."""
    B, Hq, Hkv, d, C = shape
    q, k, v, cu_q, cu_k = decode_inputs(device, shape)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=device)

    def timed(call):
        call()
        torch.cuda.synchronize(device)
        ms = []
        for _ in range(iters):
            flush.zero_()
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record(stream)
            call()
            e.record(stream)
            torch.cuda.synchronize(device)
            ms.append(s.elapsed_time(e))
        if attn.get_error() != attn.ATTN_OK:
            raise RuntimeError(f"device error in the decode leg: {attn.last_device_error():#x}")
        return statistics.median(ms)

    o, lse = torch.empty_like(q), torch.empty(Hq, B, dtype=torch.float32, device=device)
    t_dec = timed(lambda: attn.attn_decode(q, k, v, cu_k, out=o, lse=lse, stream=stream))
    attn.set_decode_path(False)
    try:
        t_cc = timed(lambda: attn.attn_decode(q, k, v, cu_k, out=o, lse=lse, stream=stream))
    finally:
        attn.set_decode_path(True)
    t_fwd = timed(lambda: attn.attn_fwd(q, k, v, causal=True, cu_seqlens=cu_q, cu_seqlens_k=cu_k, out=o, lse=lse,
                                        stream=stream))
    if not no_flush:
        return t_dec, t_cc, t_fwd, 2 * k.numel() * k.element_size()
    runs = []
    for _ in range(5):
        torch.cuda.synchronize(device)
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        for _ in range(iters):
            attn.attn_decode(q, k, v, cu_k, out=o, lse=lse, stream=stream)
        e.record(stream)
        torch.cuda.synchronize(device)
        runs.append(s.elapsed_time(e) / iters)
    if attn.get_error() != attn.ATTN_OK:
        raise RuntimeError(f"device error in the decode leg: {attn.last_device_error():#x}")
    return t_dec, t_cc, t_fwd, 2 * k.numel() * k.element_size(), statistics.median(runs)


def decode_leg(attn, device, stream, peaks, iters: int = 20):
    """One new token per sequence over a key/value cache (the generation step
    of the training page §4.3), bf16, Hq 32, Hkv 8, d 128 and d 64.
    Memory-bound: the rate is the cache bytes read (K and V once) per second
    against the HBM copy peak.  Two shapes per head dim, B 32 sequences of
    4096 + 1 keys and one sequence of 131072 + 1 keys (``long``), each
    through attn_decode on its default route (the transposed tensor-core
    decode kernel, caches cut into pieces when the (sequence, head group)
    units are few), through attn_decode on its CUDA-core route, and through
    attn_fwd_varlen (the packed forward without pieces).  L2 is flushed (a
    256 MiB write) before each call; ``no_flush`` is attn_decode in
    back-to-back calls, the caches (268-537 MB) being larger than L2."""
    def entry(shape):
        B, Hq, Hkv, d, C = shape
        t_dec, t_cc, t_fwd, nbytes, t_nf = decode_step_times(attn, device, stream, shape, iters, no_flush=True)
        gbs = lambda t: nbytes / (t / 1e3) / 1e9
        return {"workload": f"decode: B{B} Hq{Hq} Hkv{Hkv} d{d} bf16, 1 new token over a {C}-token cache",
                "entry": "attn_decode (tensor cores)", "bound": "hbm", "achieved": gbs(t_dec), "unit": "GB/s",
                "peak": peaks["hbm_gbs"], "frac": gbs(t_dec) / peaks["hbm_gbs"], "ms": t_dec,
                "cache_bytes_per_call": nbytes,
                "no_flush": {"achieved": gbs(t_nf), "frac": gbs(t_nf) / peaks["hbm_gbs"], "ms": t_nf},
                "attn_decode_cuda_cores": {"achieved": gbs(t_cc), "frac": gbs(t_cc) / peaks["hbm_gbs"], "ms": t_cc},
                "attn_fwd_varlen": {"achieved": gbs(t_fwd), "frac": gbs(t_fwd) / peaks["hbm_gbs"], "ms": t_fwd}}
    out = entry(DECODE_SHAPE)
    out["long"] = entry(DECODE_LONG_SHAPE)
    out["d64"] = entry(DECODE_D64_SHAPES[0])
    out["d64"]["long"] = entry(DECODE_D64_SHAPES[1])
    return out


def cluster_merge_leg(attn, device, stream, peaks, iters: int = 30):
    """Split key ranges merged two ways (page S23-J17 §3.1's rescaling across
    pieces): the default combine pass (pieces of planned lengths, fp32
    partials in a workspace) against the in-cluster merge
    (attn_set_cluster_merge: equal pieces of every query block as one
    cluster, partials merged over distributed shared memory), median
    CUDA-event times with L2 flushed before each call, bf16, non-causal."""
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=device)

    def timed(call):
        call()
        torch.cuda.synchronize(device)
        ms = []
        for _ in range(iters):
            flush.zero_()
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record(stream)
            call()
            e.record(stream)
            torch.cuda.synchronize(device)
            ms.append(s.elapsed_time(e))
        if attn.get_error() != attn.ATTN_OK:
            raise RuntimeError(f"device error in the cluster-merge leg: {attn.last_device_error():#x}")
        return statistics.median(ms)

    out = {}
    try:
        for (B, H, L, d) in ((1, 1, 8192, 128), (1, 4, 4096, 64)):
            g = torch.Generator().manual_seed(21)
            q, k, v = (torch.randn(B, L, H, d, generator=g).to(torch.bfloat16).to(device) for _ in range(3))
            o, lse = attn.attn_fwd(q, k, v, causal=False)
            fl = 4.0 * d * B * H * L * L
            entry = {}
            for cs in (0, 2, 4, 8):
                attn.set_cluster_merge(cs)
                t = timed(lambda: attn.attn_fwd(q, k, v, causal=False, out=o, lse=lse, stream=stream))
                entry["combine_pass" if cs == 0 else f"cluster_{cs}"] = {"ms": t, "tflops": fl / (t / 1e3) / 1e12}
            out[f"B{B} H{H} L{L} d{d} non-causal"] = entry
    finally:
        attn.set_cluster_merge(0)
    return out


def rope_fused_leg(attn, device, stream, peaks, iters: int = 30):
    """The forward of rotary-embedded q and k (training page §4), three ways,
    median CUDA-event times with L2 flushed before each call: attn_fwd_rope
    (Q rotated inside the forward kernel, K by the rotary pass), the unfused
    route (attn_rotary on q and on k, then attn_fwd) and attn_fwd alone on
    the same tensors (no rotation: the floor).  GPT-NeoX pairing over the full
    head dimension, base 10000.  Two shapes: the headline workload and the
    GQA configuration."""
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=device)

    def timed(call):
        call()
        torch.cuda.synchronize(device)
        ms = []
        for _ in range(iters):
            flush.zero_()
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record(stream)
            call()
            e.record(stream)
            torch.cuda.synchronize(device)
            ms.append(s.elapsed_time(e))
        if attn.get_error() != attn.ATTN_OK:
            raise RuntimeError(f"device error in the rope leg: {attn.last_device_error():#x}")
        return statistics.median(ms)

    out = {}
    for name in ("single_head_l8192_d128_causal", "gqa_b2_hq32_hkv8_l4096_d128_causal"):
        wl = WORKLOADS[name]
        inp = generate(wl)
        q, k, v = inp.q.to(device), inp.k.to(device), inp.v.to(device)
        o, lse = attn.attn_fwd(q, k, v, causal=wl.causal, scale=wl.softmax_scale)
        qr, kr = torch.empty_like(q), torch.empty_like(k)

        def fused():
            attn.attn_fwd_rope(q, k, v, causal=wl.causal, scale=wl.softmax_scale, out=o, lse=lse, stream=stream)

        def unfused():
            attn.rotary(q, out=qr, stream=stream)
            attn.rotary(k, out=kr, stream=stream)
            attn.attn_fwd(qr, kr, v, causal=wl.causal, scale=wl.softmax_scale, out=o, lse=lse, stream=stream)

        def plain():
            attn.attn_fwd(q, k, v, causal=wl.causal, scale=wl.softmax_scale, out=o, lse=lse, stream=stream)

        t_f, t_u, t_p = timed(fused), timed(unfused), timed(plain)
        fl = workload_flops(wl, inp.lengths)
        out[name] = {"fused_ms": t_f, "unfused_ms": t_u, "attn_fwd_only_ms": t_p,
                     "fused_tflops": fl / (t_f / 1e3) / 1e12, "unfused_tflops": fl / (t_u / 1e3) / 1e12}
    return out


CONFIG_ORDER = ("mha_l256_d64", "single_head_l8192_d128_causal", "mha_b2_h16_l2048_d64_fp16_causal",
                "gqa_b2_hq32_hkv8_l4096_d128_causal", "varlen_b16_h12_d64")


def configs_leg(attn, device, stream, peaks, flush, iters: int = 40, rows: int = 48):
    """Every workload of the pages' five configurations through attn_fwd, in
    the launch configuration of the headline: per call L2 flushed, CUDA events
    on the launching stream, median of ``iters`` calls.  Reports TFLOP/s
    (causal-adjusted), its fraction of the measured bf16 peak and the main
    kernel's median duration (library profiling events).  Also returns, per
    configuration, the GPU's O and lse on ``rows`` sampled rows (varlen: every
    row), which the CPU-baseline leg checks against the oracle."""
    from tiled_attention_attn_gb300.inputs import sample_rows

    out, kept = {}, {}
    for name in CONFIG_ORDER:
        wl = WORKLOADS[name]
        inp = generate(wl)
        q, k, v = inp.q.to(device), inp.k.to(device), inp.v.to(device)
        cu = inp.cu_seqlens.to(device) if inp.cu_seqlens is not None else None
        o, lse = attn.attn_fwd(q, k, v, causal=wl.causal, scale=wl.softmax_scale, cu_seqlens=cu)
        for _ in range(5):
            flush.zero_()
            attn.attn_fwd(q, k, v, causal=wl.causal, scale=wl.softmax_scale, cu_seqlens=cu, out=o, lse=lse)
        ms = []
        for _ in range(iters):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            attn.attn_fwd(q, k, v, causal=wl.causal, scale=wl.softmax_scale, cu_seqlens=cu, out=o, lse=lse)
            b.record(stream)
            torch.cuda.synchronize(device)
            ms.append(a.elapsed_time(b))
        attn.profile_enable(iters)
        for _ in range(iters):
            flush.zero_()
            attn.attn_fwd(q, k, v, causal=wl.causal, scale=wl.softmax_scale, cu_seqlens=cu, out=o, lse=lse)
        main_ms, _ = attn.profile_read(iters)
        attn.profile_disable()
        if attn.get_error() != attn.ATTN_OK:
            raise RuntimeError(f"device error in the configs leg ({name}): {attn.last_device_error():#x}")
        t = statistics.median(ms)
        fl = workload_flops(wl, inp.lengths)
        on = o.float().cpu().double().numpy()
        ln = lse.cpu().double().numpy()
        if wl.varlen:
            kept[name] = (wl, inp, None, on, ln)
        else:
            rs = sample_rows(wl, rows)
            idx = np.array(rs)
            kept[name] = (wl, inp, rs, on[idx[:, 0], idx[:, 2], idx[:, 1]], ln[idx[:, 0], idx[:, 1], idx[:, 2]])
        tf = fl / (t / 1e3) / 1e12
        out[name] = {"ms_median": t, "ms_min": min(ms), "tflops": tf, "frac": tf / peaks["bf16_tflops"],
                     "kernel_ms": statistics.median(main_ms),
                     "kernel_tflops": fl / (statistics.median(main_ms) / 1e3) / 1e12,
                     "dtype": wl.dtype, "flops": fl}
        del q, k, v, o, lse
    return out, kept


def configs_oracle_check(cfgs, kept):
    """CPU-baseline leg for the five configurations: the fp64 oracle on the
    rows the configs leg kept (timed: its TFLOP/s on those rows is the
    configuration's CPU baseline), and the largest |O - O_ref|, |lse - lse_ref|
    of the GPU's outputs on them."""
    import oracle

    oracle.build()
    for name, (wl, inp, rs, o_gpu, lse_gpu) in kept.items():
        t0 = time.perf_counter()
        if rs is None:
            o_ref, lse_ref = oracle.varlen_attention(inp.q, inp.k, inp.v, inp.lengths, causal=wl.causal,
                                                     scale=wl.softmax_scale)
            fl = workload_flops(wl, inp.lengths)
            checked = "every row"
        else:
            o_ref, lse_ref = oracle.attention_rows(inp.q, inp.k, inp.v, rs, causal=wl.causal, scale=wl.softmax_scale)
            fl = sample_flops(wl, rs)
            checked = f"{len(rs)} sampled rows"
        dt = max(time.perf_counter() - t0, 1e-9)
        fin = np.isfinite(lse_ref)
        cfgs[name].update({"max_abs_err_o": float(np.max(np.abs(o_gpu - o_ref))),
                           "max_abs_err_lse": float(np.max(np.abs(lse_gpu[fin] - lse_ref[fin]))) if fin.any() else 0.0,
                           "checked": checked, "bar": {"o": 1e-2, "lse": 1e-3},
                           "cpu_baseline_tflops": fl / dt / 1e12})


def pair_headline(attn, wl, q, k, v, o, lse, stream, device, flush, iters: int = 40):
    """The headline workload on the CTA-pair kernel (attn_set_pair_forward),
    for comparison with the default single-CTA kernel: median call time."""
    attn.set_pair_forward(True)
    try:
        for _ in range(5):
            flush.zero_()
            attn.attn_fwd(q, k, v, causal=wl.causal, scale=wl.softmax_scale, out=o, lse=lse)
        ms = []
        for _ in range(iters):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            attn.attn_fwd(q, k, v, causal=wl.causal, scale=wl.softmax_scale, out=o, lse=lse)
            b.record(stream)
            torch.cuda.synchronize(device)
            ms.append(a.elapsed_time(b))
    finally:
        attn.set_pair_forward(False)
    if attn.get_error() != attn.ATTN_OK:
        raise RuntimeError(f"device error in the pair-kernel leg: {attn.last_device_error():#x}")
    return statistics.median(ms)


def run_ours(args, wl):
    from tiled_attention_attn_gb300 import attn, build

    dist, world, rank, local = dist_setup(args.gpus)
    build.build()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    inp = generate(wl)
    q, k, v = inp.q.to(device), inp.k.to(device), inp.v.to(device)
    cu = inp.cu_seqlens.to(device) if inp.cu_seqlens is not None else None
    o = torch.empty_like(q)
    lse_shape = (wl.Hq, q.shape[0]) if wl.varlen else (wl.B, wl.Hq, wl.Lq)
    lse = torch.empty(lse_shape, dtype=torch.float32, device=device)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=device)
    flops = workload_flops(wl, inp.lengths)
    stream = torch.cuda.current_stream(device)
    if args.bwd_only:
        # the backward leg alone (for profiling it)
        if rank == 0:
            print(json.dumps({"backward": bwd_leg(attn, device, stream, measured_peaks())}), flush=True)
        return 0
    if args.legs_only:
        # the padded-batch, kv-cache and rotary legs alone (for profiling them)
        peaks = measured_peaks()
        if rank == 0:
            print(json.dumps({"pad_unpad": pad_leg(attn, device, stream, peaks),
                              "kv_cache": cache_leg(attn, device, stream, peaks),
                              "rotary": rotary_leg(attn, device, stream, peaks),
                              "decode": decode_leg(attn, device, stream, peaks),
                              "rope_fused": rope_fused_leg(attn, device, stream, peaks),
                              "cluster_merge": cluster_merge_leg(attn, device, stream, peaks),
                              "backward": bwd_leg(attn, device, stream, peaks)}), flush=True)
        return 0

    def call():
        attn.attn_fwd(q, k, v, causal=wl.causal, scale=wl.softmax_scale, cu_seqlens=cu, out=o, lse=lse)

    if args.profile_decode > 0:
        # attn_decode calls of the decode leg's batch shape (for profiling)
        shape = DECODE_SHAPE if args.decode_d == 128 else DECODE_D64_SHAPES[0]
        dq, dk, dv, _, dcu = decode_inputs(device, shape)
        do = torch.empty_like(dq)
        dl = torch.empty(shape[1], shape[0], dtype=torch.float32, device=device)
        for _ in range(args.profile_decode):
            flush.zero_()
            attn.attn_decode(dq, dk, dv, dcu, out=do, lse=dl, stream=stream)
        torch.cuda.synchronize(device)
        if attn.get_error() != attn.ATTN_OK:
            raise RuntimeError(f"device error: {attn.last_device_error():#x}")
        print(f"{args.profile_decode} attn_decode calls of B{shape[0]} x {shape[4]}, d {shape[3]}")
        return 0
    if args.profile_calls > 0:
        attn.set_pair_forward(args.pair)
        for _ in range(args.profile_calls):
            flush.zero_()
            call()
        torch.cuda.synchronize(device)
        if attn.get_error() != attn.ATTN_OK:
            raise RuntimeError(f"device error: {attn.last_device_error():#x}")
        print(f"{args.profile_calls} calls of {wl.name}" + (" on the CTA-pair kernel" if args.pair else ""))
        return 0

    # warm-up
    for _ in range(args.warmup):
        flush.zero_()
        call()
    if attn.get_error() != attn.ATTN_OK:
        raise RuntimeError(f"device error during warm-up: {attn.last_device_error():#x}")

    # ---- headline: K steps, L2 flushed before each, per-step events
    K = args.steps
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    sampler = ClockSampler(gpu_index_for(local))
    sampler.start()
    barrier(dist)
    torch.cuda.synchronize(device)
    sampler.mark("begin")
    lc0 = attn.launch_count()
    head_ms = head_start(K)
    for i in range(K):
        flush.zero_()
        starts[i].record(stream)
        call()
        ends[i].record(stream)
    torch.cuda.synchronize(device)
    barrier(dist)
    sampler.mark("end")
    launches = attn.launch_count() - lc0
    clocks = sampler.stop()
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    total_ms = sum(step_ms)
    total_ms = max_over_ranks(dist, total_ms, device)
    if attn.get_error() != attn.ATTN_OK:
        raise RuntimeError(f"device error in the timed region: {attn.last_device_error():#x}")
    value = world * flops * K / (total_ms / 1e3) / 1e12

    # ---- roofline: the main kernel's own duration (library profiling events)
    KR = min(K, 2000)
    attn.profile_enable(KR)
    for _ in range(KR):
        flush.zero_()
        call()
    main_ms, call_ms = attn.profile_read(KR)
    attn.profile_disable()
    main_avg = statistics.mean(main_ms)
    peaks = measured_peaks()
    achieved = flops / (main_avg / 1e3) / 1e12
    traffic = profiled_traffic()
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": achieved / peaks["bf16_tflops"], "traffic": traffic,
                "kernel": "attn_fwd_kernel", "kernel_ms": main_avg,
                "peak_source": f"{peaks['source']} bf16 burst (MEASURED_PEAKS.json)"
                if peaks["source"] == "measured" else "fallback 1.9 PFLOP/s bf16",
                "algorithmic_flops_per_launch": flops,
                "algorithmic_bytes_per_launch": workload_bytes(wl, inp.lengths)}

    # ---- end to end through pinned host buffers: the step's inputs arrive in
    # one host-to-device copy (q, k, v, cu_seqlens packed in one pinned
    # buffer, used on the device through views) and O and lse leave in one
    # device-to-host copy (one device buffer holds both)
    KE = min(K, args.e2e_steps)

    def packed(ts):
        """One uint8 buffer holding the tensors back to back (16-byte aligned
        offsets) and the offsets."""
        offs, n = [], 0
        for t in ts:
            offs.append(n)
            n += (t.numel() * t.element_size() + 15) // 16 * 16
        return n, offs

    host_in = [inp.q, inp.k, inp.v] + ([inp.cu_seqlens] if inp.cu_seqlens is not None else [])
    n_in, off_in = packed(host_in)
    hin = torch.empty(n_in, dtype=torch.uint8).pin_memory()
    din = torch.empty(n_in, dtype=torch.uint8, device=device)

    def view(buf, off, like):
        nb = like.numel() * like.element_size()
        return buf[off:off + nb].view(like.dtype).view(like.shape)

    for t, o_ in zip(host_in, off_in):
        view(hin, o_, t).copy_(t)
    qe, ke, ve = (view(din, off_in[i], host_in[i]) for i in range(3))
    cue = view(din, off_in[3], host_in[3]) if inp.cu_seqlens is not None else None
    n_out, off_out = packed([o, lse])
    dout_buf = torch.empty(n_out, dtype=torch.uint8, device=device)
    hout = torch.empty(n_out, dtype=torch.uint8).pin_memory()
    oe, lsee = view(dout_buf, off_out[0], o), view(dout_buf, off_out[1], lse)
    e_s = [torch.cuda.Event(enable_timing=True) for _ in range(KE)]
    e_e = [torch.cuda.Event(enable_timing=True) for _ in range(KE)]
    barrier(dist)
    torch.cuda.synchronize(device)
    head_start(KE)
    for i in range(KE):
        flush.zero_()
        e_s[i].record(stream)
        din.copy_(hin, non_blocking=True)
        attn.attn_fwd(qe, ke, ve, causal=wl.causal, scale=wl.softmax_scale, cu_seqlens=cue, out=oe, lse=lsee)
        hout.copy_(dout_buf, non_blocking=True)
        e_e[i].record(stream)
    torch.cuda.synchronize(device)
    e2e_ms = max_over_ranks(dist, sum(s.elapsed_time(e) for s, e in zip(e_s, e_e)), device)
    e2e = {"value": world * flops * KE / (e2e_ms / 1e3) / 1e12, "unit": UNIT,
           "h2d_bytes_per_step": n_in, "d2h_bytes_per_step": n_out, "steps": KE,
           "copies_per_step": {"h2d": 1, "d2h": 1}}
    if not torch.equal(view(hout, off_out[0], o), o.cpu()):
        raise RuntimeError("e2e leg: the output read back differs from the device result")
    if attn.get_error() != attn.ATTN_OK:
        raise RuntimeError(f"device error in the e2e leg: {attn.last_device_error():#x}")

    # ---- padded batches: unpad index and row gather / scatter (HBM-bound)
    pad = cache = rot = bwd = dec = rope = cmerge = None
    if not args.no_pad_leg:
        pad = pad_leg(attn, device, stream, peaks)
        cache = cache_leg(attn, device, stream, peaks)
        dec = decode_leg(attn, device, stream, peaks)
        bwd = bwd_leg(attn, device, stream, peaks)
        rot = rotary_leg(attn, device, stream, peaks)
        rope = rope_fused_leg(attn, device, stream, peaks)
        cmerge = cluster_merge_leg(attn, device, stream, peaks)

    # ---- the five configurations, and the headline on the CTA-pair kernel
    cfgs = pair = kept = None
    if rank == 0 and not args.no_configs_leg:
        cfgs, kept = configs_leg(attn, device, stream, peaks, flush)
        if not wl.varlen and wl.d == 128:
            t_pair = pair_headline(attn, wl, q, k, v, o, lse, stream, device, flush)
            pair = {"kernel": "attn_pair_kernel (attn_set_pair_forward(1))", "ms_median": t_pair,
                    "tflops": flops / (t_pair / 1e3) / 1e12,
                    "frac": flops / (t_pair / 1e3) / 1e12 / peaks["bf16_tflops"]}

    # ---- CPU baseline: the oracle on a bounded sample (rank 0, N = 1)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tf, dt, n, threads = oracle_sample(wl, inp, args.cpu_budget_s)
        cpu = {"value": tf, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": f"{n} random query rows of {wl.name} ({dt:.1f} s), fp64, S and P rows materialised"}
        if cfgs is not None:
            configs_oracle_check(cfgs, kept)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
            "ms_per_step": total_ms / K, "ms_per_step_median": statistics.median(step_ms),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": wl.dtype, "data": "synthetic",
            "config": dict(workload_config(wl, inp.lengths), parallelism=f"replicas x{world}",
                           l2="256 MiB buffer written before every step, outside the per-step CUDA events",
                           head_start_ms=head_ms),
            "pct_of_peak": 100.0 * value / world / peaks["bf16_tflops"],
            "pct_of_sustained_peak": 100.0 * value / world / peaks["bf16_tflops_sustained"],
            "step_ms": {"median": statistics.median(step_ms), "min": min(step_ms), "max": max(step_ms), "mean": total_ms / K,
                        "per_rank_events": "one CUDA-event pair per step on the launching stream"},
            "clocks": clocks, "e2e": e2e, "gpu_launches": launches, "roofline": roofline,
            "cpu_baseline": cpu, "configs": cfgs, "pair_kernel_headline": pair,
            "pad_unpad": pad, "kv_cache": cache, "rotary": rot, "backward": bwd, "decode": dec, "rope_fused": rope, "cluster_merge": cmerge,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=HEADLINE, choices=sorted(WORKLOADS))
    ap.add_argument("--e2e-steps", type=int, default=500)
    ap.add_argument("--cpu-budget-s", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-pad-leg", action="store_true", help="skip the padded-batch, kv-cache, rotary and backward legs")
    ap.add_argument("--no-configs-leg", action="store_true", help="skip the five-configuration leg")
    ap.add_argument("--bwd-only", action="store_true", help="run only the backward leg")
    ap.add_argument("--legs-only", action="store_true", help="run only the padded-batch, kv-cache, rotary and backward legs")
    ap.add_argument("--profile-calls", type=int, default=0,
                    help="only make this many attn_fwd calls of --workload (L2 flushed before each) and exit: "
                         "the program the ncu summaries capture")
    ap.add_argument("--profile-decode", type=int, default=0,
                    help="only make this many attn_decode calls of the decode leg's batch shape "
                         "(L2 flushed before each) and exit")
    ap.add_argument("--decode-d", type=int, default=128, choices=[64, 128],
                    help="with --profile-decode: the head dim of the decode shape")
    ap.add_argument("--pair", action="store_true", help="with --profile-calls: run the CTA-pair kernel")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    wl = WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, wl)
    return run_ours(args, wl)


if __name__ == "__main__":
    sys.exit(main())
