"""Benchmark of the exact-attention hot path on GB300.

One step = forward + backward (fa_forward, then the three backward stages
fa_backward runs for dense d <= 128: preprocess, dK/dV, dQ) over one batch
of the workload, by default the causal N=8192, d=128, bf16, B=2, H=32
problem.  Prints ONE JSON line (rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload C4]
    python bench.py --impl reference ...   # the float64 CPU oracle as the baseline arm

Throughput convention: F = 4 B H N^2 d (halved under the causal mask);
value = 2.5 F / (t_fwd + t_bwd) in TFLOP/s, summed over all GPUs.
Multi-GPU (torchrun): every rank runs its own copy of the workload (its own
heads; no collective in the data path), so per-GPU work is fixed: weak scaling.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attention TFLOPS (fwd, fwd+bwd) & % of GB300 dense BF16 tensor peak, N=4K–32K"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# The ncu capture of the roofline kernel (one C4 launch): its summary under profiles/ records
# dram__bytes_read.sum + dram__bytes_write.sum per launch and a hash of the kernel's source
# files at capture time; the bench reports that traffic only while the sources still hash the
# same (a changed kernel reports null until it is captured again).
DKDV_PROFILE = os.path.join(ROOT, "profiles", "fa_bwd_dkdv_split_C4_causal_n8192_d128_bf16.md")
DKDV_SOURCES = ("fa_bwd_split.cu", "fa_bwd_kernel.cuh", "fa_ptx.cuh", "fa_internal.h", "fa_layout.cuh",
                "fa_philox.cuh")
# The same for the variant lines whose roofline object is the split dK/dV kernel.
VARIANT_PROFILES = {
    "blocksparse": os.path.join(ROOT, "profiles", "fa_bwd_dkdv_split_blocksparse_S1_n8192_d128_bf16.md"),
    "varlen": os.path.join(ROOT, "profiles", "fa_bwd_dkdv_split_varlen_V1_causal_d128_bf16.md"),
}


def kernel_source_hash(names=DKDV_SOURCES) -> str:
    """First 16 hex digits of the sha256 of the named csrc files, in order."""
    import hashlib
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "exact_io_aware_forward_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def captured_traffic(path=DKDV_PROFILE):
    """(bytes per launch, note) from a profile summary's `traffic_bytes_per_launch:` and
    `source_sha256_16:` lines; bytes is None when absent or taken on other sources."""
    try:
        text = open(path, encoding="utf-8").read()
    except OSError:
        return None, "no capture"
    vals = {}
    for line in text.splitlines():
        for key in ("traffic_bytes_per_launch", "source_sha256_16"):
            if line.strip().startswith(key + ":"):
                vals[key] = line.split(":", 1)[1].strip().strip("`")
    if "traffic_bytes_per_launch" not in vals or "source_sha256_16" not in vals:
        return None, "capture lacks traffic or hash"
    if vals["source_sha256_16"] != kernel_source_hash():
        return None, "kernel changed since the capture"
    return int(vals["traffic_bytes_per_launch"]), os.path.relpath(path, ROOT)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def max_over_ranks(value: float, dist, device) -> float:
    """The largest `value` over all ranks (every rank gets it); `value` itself
    when there is no process group.  The timing rule of the multi-GPU line: the
    slowest rank's time is the job's time."""
    if dist is None:
        return float(value)
    import torch
    t = torch.tensor([float(value)], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, work_per_rank: float, ms_slowest: float) -> float:
    """Whole-job throughput of a weak-scaling run: every rank processes
    `work_per_rank` units (its own heads), the job takes the slowest rank's time."""
    return world * work_per_rank / (ms_slowest * 1e-3)


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for name, flag in zip(names, parts[5:9]):
                if flag.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm_sorted = sorted(sm)
        return {"sm_mhz": sm_sorted[len(sm_sorted) // 2], "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(power)}


# ---------------------------------------------------------------- CPU oracle leg
def oracle_sample(w, budget_s: float, max_heads: int):
    """Time the float64 oracle (forward + explicit backward, S and P
    materialised) on whole heads of the workload until `budget_s` is spent.
    Returns (TFLOP/s in the metric's convention, heads timed, seconds, threads)."""
    import numpy as np
    from exact_io_aware_forward_gb300.synth import as_float64, attention_inputs
    from oracle import attention as A

    # One head at a time (B = H = 1, per-head seeds) keeps host memory bounded.
    heads, spent = 0, 0.0
    scale = 1.0 / math.sqrt(w.d)
    while heads < max_heads and (heads == 0 or spent < budget_s):
        q, k, v, do = as_float64(*attention_inputs(1, 1, w.N, w.d, w.dtype, seed=w.seed * 1000 + heads,
                                                   k_row_scale=w.k_row_scale))
        t0 = time.perf_counter()
        if w.N <= 16384:
            A.forward_head(q[0, 0], k[0, 0], v[0, 0], scale, w.causal)
            A.backward_head(q[0, 0], k[0, 0], v[0, 0], do[0, 0], scale, w.causal)
        else:  # bounded host memory: the same definition in 2048-row stripes
            for r0 in range(0, w.N, 2048):
                A.forward_head(q[0, 0], k[0, 0], v[0, 0], scale, w.causal, rows=np.arange(r0, min(w.N, r0 + 2048)))
            A.backward_head_sampled(q[0, 0], k[0, 0], v[0, 0], do[0, 0], scale, w.causal,
                                    np.arange(w.N), np.arange(w.N))
        spent += time.perf_counter() - t0
        heads += 1
    per_head = 2.5 * w.fwd_flops() / w.heads
    threads = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    return per_head * heads / spent / 1e12, heads, spent, threads


# ---------------------------------------------------------------- decode (split-KV)
def oracle_decode_sample(w, budget_s: float, max_heads: int):
    """float64 oracle on whole heads of a decode workload; GB/s of K/V covered."""
    from exact_io_aware_forward_gb300.synth import as_float64, attention_inputs
    from oracle import attention as A
    heads, spent = 0, 0.0
    scale = 1.0 / math.sqrt(w.d)
    wall0 = time.perf_counter()  # the budget also covers input generation
    while heads < min(max_heads, w.B * w.H) and (heads == 0 or time.perf_counter() - wall0 < budget_s):
        q, _, _, _ = attention_inputs(1, 1, w.Nq, w.d, w.dtype, seed=w.seed * 1000 + heads, with_do=False)
        _, k, v, _ = attention_inputs(1, 1, w.Nk, w.d, w.dtype, seed=w.seed * 1000 + heads + 1, with_do=False)
        q, k, v = as_float64(q, k, v)
        t0 = time.perf_counter()
        A.forward_head(q[0, 0], k[0, 0], v[0, 0], scale, w.causal)
        spent += time.perf_counter() - t0
        heads += 1
    per_head = w.kv_bytes() / (w.B * w.H)
    threads = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    return per_head * heads / spent / 1e9, heads, spent, threads


def measure_decode(dev, w, steps, warmup):
    """Device-resident timing of fa_forward_decode (split + combine kernels) on
    workload `w`; the L2 is flushed before every timed call."""
    import torch

    import exact_io_aware_forward_gb300 as fa
    from exact_io_aware_forward_gb300.synth import decode_inputs

    q, k, v = (x.to(dev) for x in decode_inputs(w))
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.Nq), device=dev, dtype=torch.float32)
    ws = torch.empty(fa.fa_decode_workspace_size(w.B, w.H, w.Nq, w.Nk, w.d, 0), device=dev, dtype=torch.uint8)
    flush = torch.empty(256 << 20, device=dev, dtype=torch.uint8)
    for _ in range(warmup):
        fa.fa_forward_decode(q, k, v, o, lse, ws, w.causal)
    fa.fa_device_status()
    total = 0.0
    for _ in range(steps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        fa.fa_forward_decode(q, k, v, o, lse, ws, w.causal)
        e1.record()
        torch.cuda.synchronize()
        total += e0.elapsed_time(e1)
    fa.fa_device_status()
    ms = total / steps
    byts = w.kv_bytes() + 2 * (w.B * w.H * w.Nq * w.d * 2)
    return ms, byts, (q, k, v, ws)


def run_decode(args, world, rank, local):
    import dataclasses

    import torch

    import exact_io_aware_forward_gb300 as fa
    from exact_io_aware_forward_gb300.synth import D1 as w
    if args.decode_d != w.d:  # the same keys at another head dimension (d = 256: half the heads)
        w = dataclasses.replace(w, d=args.decode_d, H=w.H if args.decode_d <= 128 else w.H // 2)
    if args.nq != w.Nq or args.decode_d != 128:
        w = dataclasses.replace(w, Nq=args.nq,
                                name=f"D1 decode causal Nq={args.nq} Nk={w.Nk} H={w.H} d={w.d} {w.dtype}")

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    peaks, peak_src = load_peaks()
    sampler = ClockSampler(local)
    sampler.start()
    ms, byts, (q, k, v, ws) = measure_decode(dev, w, args.steps, args.warmup)
    clocks = sampler.stop()
    gbs = byts / (ms * 1e-3) / 1e9
    hq, hk, hv = (x.cpu().pin_memory() for x in (q, k, v))
    ho = torch.empty_like(hq).pin_memory()
    hl = torch.empty((w.B, w.H, w.Nq), dtype=torch.float32).pin_memory()

    def e2e_step():
        gq, gk, gv = (x.to(dev, non_blocking=True) for x in (hq, hk, hv))
        go, gl = fa.forward_decode(gq, gk, gv, causal=w.causal, workspace=ws)
        ho.copy_(go, non_blocking=True)
        hl.copy_(gl, non_blocking=True)

    e2e_step()
    torch.cuda.synchronize()
    c0 = time.perf_counter()
    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    e2e_ms = (time.perf_counter() - c0) * 1e3 / 3
    cpu, heads, spent, threads = oracle_decode_sample(w, args.cpu_budget, 4096)
    peak = float(peaks["hbm_gbs"])
    return {
        "metric": "split-KV decode throughput (K/V bytes streamed per second)", "value": round(world * gbs, 1),
        "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic (seeded N(0,1) Q, K, V; no dataset)",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "Nq": w.Nq, "Nk": w.Nk, "d": w.d, "causal": w.causal,
                   "l2": "flushed (256 MB write) before every timed call"},
        "roofline": {"bound": "hbm", "kernel": "fa_decode_tc_kernel + fa_decode_combine_kernel",
                     "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s", "frac": round(gbs / peak, 4),
                     "traffic": None, "peak_source": f"{peak_src} hbm_gbs",
                     "algorithmic": "K + V + Q + O bytes per call"},
        "e2e": {"value": round(world * byts / (e2e_ms * 1e-3) / 1e9, 1), "unit": "GB/s",
                "h2d_bytes_per_step": int(hq.numel() * 2 + hk.numel() * 2 + hv.numel() * 2),
                "d2h_bytes_per_step": int(ho.numel() * 2 + hl.numel() * 4), "ms_per_step": round(e2e_ms, 3)},
        "gpu_launches": 2 * args.steps,
        "clocks": clocks,
        "cpu_baseline": {"value": cpu, "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": f"{heads} whole head(s) of {w.name}, float64 forward, {spent:.1f} s"},
    }


# ---------------------------------------------------------------- block-sparse
def block_mask_flops(w, bm) -> float:
    """Forward FLOPs over the kept blocks: 4 * d per (query, key) pair that a
    kept block covers (2 for Q K^T, 2 for P V), counting only rows and keys that
    exist in a ragged last tile and, under the causal mask, only key <= query."""
    import numpy as np
    T = w.tiles
    size = np.minimum(128, w.N - 128 * np.arange(T)).astype(np.float64)
    pairs = np.outer(size, size)
    if w.causal:
        pairs = np.tril(pairs)
        pairs[np.arange(T), np.arange(T)] = size * (size + 1) / 2
    per_mask = (bm * pairs).sum(axis=(1, 2))
    total = per_mask.sum() * (w.B * w.H if bm.shape[0] == 1 else 1)
    return 4.0 * w.d * float(total)


def varlen_pairs(lengths, causal) -> float:
    """(query, key) pairs computed over a packed batch with Nq = Nk per sequence."""
    return float(sum(n * (n + 1) // 2 if causal else n * n for n in lengths))


def oracle_varlen_sample(w, budget_s: float):
    """float64 oracle on whole (sequence, head) problems of a packed batch, in
    order, until `budget_s` is spent; TFLOP/s in the 2.5 F convention."""
    from exact_io_aware_forward_gb300.synth import as_float64, attention_inputs
    from oracle import attention as A
    scale = 1.0 / math.sqrt(w.d)
    done, spent, flops = 0, 0.0, 0.0
    for n in sorted(w.lengths):  # shortest first so that the sample covers several sequences
        if done and spent >= budget_s:
            break
        q, k, v, do = as_float64(*attention_inputs(1, 1, n, w.d, w.dtype, seed=w.seed * 1000 + done))
        t0 = time.perf_counter()
        A.forward_head(q[0, 0], k[0, 0], v[0, 0], scale, w.causal)
        A.backward_head(q[0, 0], k[0, 0], v[0, 0], do[0, 0], scale, w.causal)
        spent += time.perf_counter() - t0
        flops += 2.5 * 4.0 * w.d * varlen_pairs([n], w.causal)
        done += 1
    threads = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    return flops / spent / 1e12, done, spent, threads


def oracle_variant_sample(kind, w, bm, budget_s: float, max_heads: int):
    """float64 oracle (forward + explicit backward) on whole heads of a
    block-sparse or dropout workload until `budget_s` is spent; TFLOP/s in the
    2.5 F convention, F counted like the GPU line."""
    from exact_io_aware_forward_gb300.synth import as_float64, attention_inputs
    from oracle import attention as A
    from oracle import dropout as DR
    heads, spent, flops = 0, 0.0, 0.0
    scale = 1.0 / math.sqrt(w.d)
    per_head = (block_mask_flops(w, bm) if kind == "blocksparse" else w.fwd_flops()) / (w.B * w.H)
    while heads < max_heads and (heads == 0 or spent < budget_s):
        q, k, v, do = as_float64(*attention_inputs(1, 1, w.N, w.d, w.dtype, seed=w.seed * 1000 + heads))
        q, k, v, do = q[0, 0], k[0, 0], v[0, 0], do[0, 0]
        t0 = time.perf_counter()
        if kind == "blocksparse":
            m = bm[0 if bm.shape[0] == 1 else heads % bm.shape[0]]
            A.forward_head(q, k, v, scale, w.causal, block_mask=m)
            A.backward_head(q, k, v, do, scale, w.causal, block_mask=m)
        else:  # the keep mask is part of the method: drawn inside the timed region
            keep = DR.keep_mask(DROP_SEED, DROP_OFFSET, DROP_P, heads, w.N, w.N)
            c = DR.keep_scale(DROP_P)
            A.forward_head(q, k, v, scale, w.causal, keep=keep, keep_scale=c)
            A.backward_head(q, k, v, do, scale, w.causal, keep=keep, keep_scale=c)
        spent += time.perf_counter() - t0
        flops += 2.5 * per_head
        heads += 1
    threads = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    return flops / spent / 1e12, heads, spent, threads


# Dropout line: the long causal training workload with p = 0.1.
DROP_P, DROP_SEED, DROP_OFFSET = 0.1, 2024, 0


def measure_variant(dev, kind, w, steps, warmup, sampler=None):
    """Device-resident fwd+bwd of a block-sparse or dropout workload, each of
    the four kernels timed with CUDA events on the launching stream.
    Returns (ms per step, per-kernel ms, clocks, buffers)."""
    import torch

    import exact_io_aware_forward_gb300 as fa
    from exact_io_aware_forward_gb300.synth import blocksparse_inputs, varlen_workload_inputs, workload_inputs

    cu_q = cu_k = None
    if kind == "blocksparse":
        q, k, v, do, bm = blocksparse_inputs(w)
        md = torch.from_numpy(bm.astype("uint8")).to(dev)
    elif kind == "varlen":
        q, k, v, do, cu_q, cu_k = varlen_workload_inputs(w)
        cu_q, cu_k = cu_q.to(dev), cu_k.to(dev)
        bm = md = None
    else:
        q, k, v, do = workload_inputs(w)
        bm = md = None
    q, k, v, do = (x.to(dev) for x in (q, k, v, do))
    d = w.d
    if kind == "varlen":  # packed [T, H, d]; the flat [1, 1, T*H, d] view serves the row-wise stages
        T, H = q.shape[0], q.shape[1]
        rows = T * H
        lse = torch.empty((T, H), device=dev, dtype=torch.float32)
        ws = torch.empty(fa.fa_backward_varlen_workspace_size(T, H, d), device=dev, dtype=torch.uint8)
        shape_r = (T, H)
        maxlen = max(w.lengths)
    else:
        B, H, N = w.B, w.H, w.N
        rows = B * H * N
        lse = torch.empty((B, H, N), device=dev, dtype=torch.float32)
        ws = torch.empty(fa.fa_backward_workspace_size(B, H, N, d), device=dev, dtype=torch.uint8)
        shape_r = (B, H, N)
    o = torch.empty_like(q)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    delta = ws[: rows * 4].view(torch.float32).view(*shape_r)
    off = (rows * 4 + 255) // 256 * 256
    acc = ws[off: off + rows * d * 4].view(torch.float32).view(*q.shape)
    flat = (lambda x: x.view(1, 1, rows, -1)) if kind == "varlen" else (lambda x: x)
    stream = torch.cuda.current_stream()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(steps)]

    def fwd():
        if kind == "dense":
            fa.fa_forward(q, k, v, o, lse, w.causal)
        elif kind == "blocksparse":
            fa.fa_forward_blocksparse(q, k, v, o, lse, md, w.causal)
        elif kind == "varlen":
            fa.fa_forward_varlen(q, k, v, o, lse, cu_q, cu_k, maxlen, maxlen, w.causal)
        else:
            fa.fa_forward_dropout(q, k, v, o, lse, DROP_P, DROP_SEED, DROP_OFFSET, w.causal)

    split = kind in ("dense", "blocksparse", "varlen") and d != 256  # the strategy fa_backward takes

    def dkdv():
        if split and kind == "blocksparse":
            fa.fa_backward_dk_dv_blocksparse(q, k, v, do, lse, delta, dk, dv, md, w.causal)
        elif split and kind == "varlen":
            fa.fa_backward_dk_dv_varlen(q, k, v, do, lse, delta, dk, dv, cu_q, cu_k, maxlen, maxlen, w.causal)
        elif split:
            fa.fa_backward_dk_dv(q, k, v, do, lse, delta, dk, dv, w.causal)
        elif kind == "dense":
            fa.fa_backward_dkdv(q, k, v, do, lse, delta, acc, dk, dv, w.causal)
        elif kind == "blocksparse":
            fa.fa_backward_dkdv_blocksparse(q, k, v, do, lse, delta, acc, dk, dv, md, w.causal)
        elif kind == "varlen":
            fa.fa_backward_dkdv_varlen(q, k, v, do, lse, delta, acc, dk, dv, cu_q, cu_k, maxlen, maxlen, w.causal)
        else:
            fa.fa_backward_dkdv_dropout(q, k, v, do, lse, delta, acc, dk, dv, DROP_P, DROP_SEED, DROP_OFFSET,
                                        w.causal)

    def step(e=None):
        if e: e[0].record(stream)
        fwd()
        if e: e[1].record(stream)
        fa.fa_backward_preprocess(flat(o), flat(do), delta.view(1, 1, rows) if kind == "varlen" else delta,
                                  None if split else flat(acc))
        if e: e[2].record(stream)
        dkdv()
        if e: e[3].record(stream)
        if split and kind == "blocksparse":
            fa.fa_backward_dq_blocksparse(q, k, v, do, lse, delta, dq, md, w.causal)
        elif split and kind == "varlen":
            fa.fa_backward_dq_varlen(q, k, v, do, lse, delta, dq, cu_q, cu_k, maxlen, maxlen, w.causal)
        elif split:
            fa.fa_backward_dq(q, k, v, do, lse, delta, dq, w.causal)
        else:
            fa.fa_backward_dq_convert(flat(acc), flat(dq), scale=1.0 / math.sqrt(d))
        if e: e[4].record(stream)

    for _ in range(warmup):
        step()
    fa.fa_device_status()
    if sampler:
        sampler.start()
        time.sleep(0.3)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(steps):
        step(ev[i])
    t1.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop() if sampler else None
    fa.fa_device_status()
    parts = [sum(ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(steps)) / steps for j in range(4)]
    extra = (cu_q, cu_k) if kind == "varlen" else md
    return t0.elapsed_time(t1) / steps, parts, clocks, (q, k, v, do, extra, ws, bm)


def dkdv_factor(kind, w) -> float:
    """The dK/dV kernel's FLOPs in units of the forward's F: 2 (S^T, dP^T, dV, dK) where
    the backward takes the split strategy (d <= 128 without dropout: dense layouts with or without a
    block mask, and packed batches), 2.5 where that kernel also forms the dQ partials (d = 256,
    dropout)."""
    return 2.0 if kind in ("dense", "blocksparse", "varlen") and w.d != 256 else 2.5


def variant_flops(kind, w, bm):
    if kind == "blocksparse":
        return block_mask_flops(w, bm)
    if kind == "varlen":
        return 4.0 * w.d * w.H * varlen_pairs(w.lengths, w.causal)
    return w.fwd_flops()


def run_variant(args, world, rank, local, kind):
    """The JSON line of `--mode blocksparse` (S1), `--mode dropout` (C4 with p = 0.1)
    or `--mode varlen` (V1)."""
    import torch

    import exact_io_aware_forward_gb300 as fa
    from exact_io_aware_forward_gb300.synth import C4, S1, V1

    w = {"blocksparse": S1, "varlen": V1}.get(kind, C4)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    peaks, peak_src = load_peaks()
    ms, parts, clocks, (q, k, v, do, md, ws, bm) = measure_variant(dev, kind, w, args.steps, args.warmup,
                                                                   ClockSampler(local))
    F = variant_flops(kind, w, bm)
    value = 2.5 * F / (ms * 1e-3) / 1e12
    hq, hk, hv, hdo = (x.cpu().pin_memory() for x in (q, k, v, do))
    hm = None
    if kind == "blocksparse":
        hm = md.cpu().pin_memory()
    elif kind == "varlen":
        hm = tuple(x.cpu().pin_memory() for x in md)  # cu_seqlens_q, cu_seqlens_k
    ho, hdq, hdk, hdv = (torch.empty_like(x, device="cpu").pin_memory() for x in (q, q, q, q))
    hlse = torch.empty(q.shape[:2] if kind == "varlen" else (w.B, w.H, w.N), dtype=torch.float32).pin_memory()
    extra = {"block_mask": None} if kind == "blocksparse" else \
        {"dropout_p": DROP_P, "seed": DROP_SEED, "offset": DROP_OFFSET}

    def e2e_step():
        gq, gk, gv, gdo = (x.to(dev, non_blocking=True) for x in (hq, hk, hv, hdo))
        if kind == "varlen":
            cq, ck = (x.to(dev, non_blocking=True) for x in hm)
            L = max(w.lengths)
            go, glse = fa.forward_varlen(gq, gk, gv, cq, ck, L, L, causal=w.causal)
            gdq, gdk, gdv = fa.backward_varlen(gq, gk, gv, go, glse, gdo, cq, ck, L, L, causal=w.causal,
                                               workspace=ws)
        else:
            if kind == "blocksparse":
                extra["block_mask"] = hm.to(dev, non_blocking=True)
            go, glse = fa.forward(gq, gk, gv, causal=w.causal, **extra)
            gdq, gdk, gdv = fa.backward(gq, gk, gv, go, glse, gdo, causal=w.causal, workspace=ws, **extra)
        for h, g in ((ho, go), (hlse, glse), (hdq, gdq), (hdk, gdk), (hdv, gdv)):
            h.copy_(g, non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    n_e2e = max(3, min(args.steps, 10))
    c0 = time.perf_counter()
    for _ in range(n_e2e):
        e2e_step()
    torch.cuda.synchronize()
    e2e_ms = (time.perf_counter() - c0) * 1e3 / n_e2e
    fa.fa_device_status()
    elem = q.numel() * 2
    peak = float(peaks["bf16_tflops"])
    dkdv = dkdv_factor(kind, w) * F / (parts[2] * 1e-3) / 1e12
    fwd = F / (parts[0] * 1e-3) / 1e12
    if kind == "varlen":
        cpu, heads, spent, threads = oracle_varlen_sample(w, args.cpu_budget)
    else:
        cpu, heads, spent, threads = oracle_variant_sample(kind, w, bm, args.cpu_budget, 64)
    if kind == "varlen":
        metric = "variable-length attention TFLOPS over the packed batch (fwd+bwd = 2.5 F)"
        data = "synthetic (seeded N(0,1) packed Q, K, V, dO; seeded uniform sequence lengths; no dataset)"
        cfg = {"B": w.B, "lengths": list(w.lengths), "total_tokens": int(sum(w.lengths)),
               "flop_count": "F = 4*d*H per (query, key) pair of every sequence (causal: N(N+1)/2 pairs)"}
        kern = "fa_bwd_dkdv_split_kernel<128,causal,bf16,varlen>"
        alg = "8*d*H per (query, key) pair of every sequence (4 GEMMs: S^T, dP^T, dV, dK), per launch"
        h2d_extra = 2 * 4 * (w.B + 1)
        what = "(the shortest sequences first)"
    elif kind == "blocksparse":
        metric = "block-sparse attention TFLOPS over kept blocks (fwd+bwd = 2.5 F)"
        data = "synthetic (seeded N(0,1) Q, K, V, dO; seeded random block mask; no dataset)"
        cfg = {"density": w.density, "kept_blocks": int(bm.sum()), "mask_heads": int(bm.shape[0]),
               "flop_count": "F = 4*d per (query, key) pair inside kept blocks; fwd+bwd = 2.5 F"}
        kern = "fa_bwd_dkdv_split_kernel<128,non-causal,bf16,sparse>"
        alg = "8*d per (query, key) pair of the kept blocks (4 GEMMs: S^T, dP^T, dV, dK), per launch"
        h2d_extra = md.numel()
        what = "under the block mask"
    else:
        metric = "attention TFLOPS with dropout regenerated from (seed, offset) (fwd+bwd = 2.5 F)"
        data = "synthetic (seeded N(0,1) Q, K, V, dO; no dataset)"
        cfg = {"dropout_p": DROP_P, "seed": DROP_SEED, "offset": DROP_OFFSET,
               "flop_count": "fwd+bwd = 2.5 * 4*B*H*N^2*d (halved causal); generator work not counted"}
        kern = "fa_bwd_dkdv_kernel<128,causal,bf16,dropout>"
        alg = "10*N^2*d per head (5 GEMMs), halved causal, per launch"
        h2d_extra = 0
        what = "with the keep mask drawn by the oracle's generator"
    # DRAM traffic of the roofline kernel from the committed capture of this very workload, if any
    from exact_io_aware_forward_gb300.synth import S1, V1
    traffic, traffic_src = None, "no capture"
    if (kind, w.name) in (("blocksparse", S1.name), ("varlen", V1.name)):
        traffic, traffic_src = captured_traffic(VARIANT_PROFILES[kind])
    return {
        "metric": metric, "value": round(world * value, 2),
        "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": data,
        "config": dict({"workload": w.name, "B": w.B, "H": w.H, "N": getattr(w, "N", None), "d": w.d,
                        "causal": w.causal,
                        "l2": "inputs larger than L2 (each of Q, K, V, dO is %.0f MB > 129 MB)" % (elem / 1e6)},
                       **cfg),
        "fwd_tflops": round(fwd, 1), "fwd_frac_of_peak": round(fwd / peak, 4),
        "fwdbwd_frac_of_peak": round(value / peak, 4),
        "kernel_ms": ({"fa_fwd": round(parts[0], 4), "bwd_preprocess": round(parts[1], 4),
                       "bwd_dk_dv": round(parts[2], 4), "bwd_dq": round(parts[3], 4)} if kind != "dropout" else
                      {"fa_fwd": round(parts[0], 4), "bwd_preprocess": round(parts[1], 4),
                       "bwd_dkdv": round(parts[2], 4), "bwd_dq_convert": round(parts[3], 4)}),
        "roofline": {"bound": "tensor", "kernel": kern,
                     "achieved": round(dkdv, 1), "peak": peak, "unit": "TFLOP/s", "frac": round(dkdv / peak, 4),
                     "traffic": traffic, "traffic_source": traffic_src,
                     "peak_source": f"{peak_src} bf16_tflops (burst)", "algorithmic": alg},
        "e2e": {"value": round(world * 2.5 * F / (e2e_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": int(4 * elem + h2d_extra),
                "d2h_bytes_per_step": int(4 * elem + hlse.numel() * 4), "ms_per_step": round(e2e_ms, 3)},
        "gpu_launches": 4 * args.steps,
        "clocks": clocks,
        "cpu_baseline": {"value": cpu, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": f"{heads} whole head(s) of {w.name}, float64 forward + explicit backward "
                                   f"{what}, {spent:.1f} s"},
    }


# ---------------------------------------------------------------- GPU arm
def run_gpu(args, w, world, rank, local):
    import torch

    import exact_io_aware_forward_gb300 as fa
    from exact_io_aware_forward_gb300.synth import workload_inputs

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    peaks, peak_src = load_peaks()
    B, H, N, d = w.B, w.H, w.N, w.d
    q, k, v, do = (x.to(dev) for x in workload_inputs(w))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), device=dev, dtype=torch.float32)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    ws = torch.empty(fa.fa_backward_workspace_size(B, H, N, d), device=dev, dtype=torch.uint8)
    rows = B * H * N
    delta = ws[: rows * 4].view(torch.float32).view(B, H, N)
    off = (rows * 4 + 255) // 256 * 256
    acc = ws[off: off + rows * d * 4].view(torch.float32).view(B, H, N, d)
    stream = torch.cuda.current_stream()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]

    split = d != 256  # the dQ strategy fa_backward takes (decided by measurement; see bwd_strategies)

    def step(e=None):
        # The same launches fa_backward makes, split so that each kernel is timed.
        if e: e[0].record(stream)
        fa.fa_forward(q, k, v, o, lse, w.causal)
        if e: e[1].record(stream)
        fa.fa_backward_preprocess(o, do, delta, None if split else acc)
        if e: e[2].record(stream)
        if split:
            fa.fa_backward_dk_dv(q, k, v, do, lse, delta, dk, dv, w.causal)
        else:
            fa.fa_backward_dkdv(q, k, v, do, lse, delta, acc, dk, dv, w.causal)
        if e: e[3].record(stream)
        if split:
            fa.fa_backward_dq(q, k, v, do, lse, delta, dq, w.causal)
        else:
            fa.fa_backward_dq_convert(acc, dq)
        if e: e[4].record(stream)

    def backward_strategies(reps=10):
        """CUDA-event times of the two dQ strategies' backward stages on the
        resident inputs (the A/B that chose fa_backward's path)."""
        runs = {"split": [lambda: fa.fa_backward_preprocess(o, do, delta, None),
                          lambda: fa.fa_backward_dk_dv(q, k, v, do, lse, delta, dk, dv, w.causal),
                          lambda: fa.fa_backward_dq(q, k, v, do, lse, delta, dq, w.causal)],
                "accumulated": [lambda: fa.fa_backward_preprocess(o, do, delta, acc),
                                lambda: fa.fa_backward_dkdv(q, k, v, do, lse, delta, acc, dk, dv, w.causal),
                                lambda: fa.fa_backward_dq_convert(acc, dq)]}
        if not split:  # d = 256: the split stages do not exist
            runs.pop("split")
        out = {}
        for name, fns in runs.items():
            for _ in range(3):
                for f in fns:
                    f()
            tot = [0.0] * 3
            for _ in range(reps):
                ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
                ev[0].record(stream)
                for i, f in enumerate(fns):
                    f()
                    ev[i + 1].record(stream)
                torch.cuda.synchronize()
                for i in range(3):
                    tot[i] += ev[i].elapsed_time(ev[i + 1])
            ms = [t / reps for t in tot]
            out[name] = {"stage_ms": [round(x, 4) for x in ms], "bwd_ms": round(sum(ms), 4),
                         "bwd_tflops_2p5F": round(2.5 * w.fwd_flops() / (sum(ms) * 1e-3) / 1e12, 1)}
        fa.fa_device_status()
        return out

    torch.cuda.reset_peak_memory_stats(dev)
    mem_inputs = torch.cuda.memory_allocated(dev)
    for _ in range(args.warmup):
        step()
    fa.fa_device_status()
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(args.steps):
        step(ev[i])
    t1.record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clocks = sampler.stop()
    fa.fa_device_status()
    peak_mem = torch.cuda.max_memory_allocated(dev)
    total_ms = t0.elapsed_time(t1)
    parts = [sum(ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(args.steps)) / args.steps for j in range(4)]
    total_ms = max_over_ranks(total_ms, dist, dev)
    ms_step = total_ms / args.steps
    F = w.fwd_flops()
    value = job_throughput(world, 2.5 * F, ms_step) / 1e12

    # End to end through the public API: pinned host inputs in, results out.
    hq, hk, hv, hdo = (x.cpu().pin_memory() for x in (q, k, v, do))
    ho, hdq, hdk, hdv = (torch.empty_like(x, device="cpu").pin_memory() for x in (q, q, q, q))
    hlse = torch.empty((B, H, N), dtype=torch.float32).pin_memory()

    def e2e_step():
        gq, gk, gv, gdo = (x.to(dev, non_blocking=True) for x in (hq, hk, hv, hdo))
        go, glse = fa.forward(gq, gk, gv, causal=w.causal)
        gdq, gdk, gdv = fa.backward(gq, gk, gv, go, glse, gdo, causal=w.causal, workspace=ws)
        for h, g in ((ho, go), (hlse, glse), (hdq, gdq), (hdk, gdk), (hdv, gdv)):
            h.copy_(g, non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    e2e_steps = max(3, min(args.steps, 10))
    if dist:
        dist.barrier()
    c0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_step()
    torch.cuda.synchronize()
    e2e_serial_ms = (time.perf_counter() - c0) * 1e3 / e2e_steps
    e2e_serial_ms = max_over_ranks(e2e_serial_ms, dist, dev)
    fa.fa_device_status()

    # The same steps as a training loop runs them: the inputs of step i+1 are
    # copied in (side stream) while step i computes, and the results of step i
    # are copied out (another side stream) while step i+1 computes.  Every
    # step's copies are still inside the timed region.
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    compute = torch.cuda.current_stream(dev)
    bufs = [[torch.empty_like(x) for x in (q, k, v, do)] for _ in range(2)]
    ready = [torch.cuda.Event() for _ in range(2)]
    free = [torch.cuda.Event() for _ in range(2)]
    for e in free:
        e.record(compute)

    def e2e_pipelined(n_steps):
        for i in range(n_steps):
            b = i % 2
            with torch.cuda.stream(s_in):
                s_in.wait_event(free[b])
                for dst, src in zip(bufs[b], (hq, hk, hv, hdo)):
                    dst.copy_(src, non_blocking=True)
                ready[b].record(s_in)
            compute.wait_event(ready[b])
            gq, gk, gv, gdo = bufs[b]
            go, glse = fa.forward(gq, gk, gv, causal=w.causal)
            gdq, gdk, gdv = fa.backward(gq, gk, gv, go, glse, gdo, causal=w.causal, workspace=ws)
            free[b].record(compute)
            s_out.wait_event(free[b])
            with torch.cuda.stream(s_out):
                for h, g in ((ho, go), (hlse, glse), (hdq, gdq), (hdk, gdk), (hdv, gdv)):
                    g.record_stream(s_out)
                    h.copy_(g, non_blocking=True)

    e2e_pipelined(2)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    c0 = time.perf_counter()
    e2e_pipelined(e2e_steps)
    torch.cuda.synchronize()
    e2e_ms = (time.perf_counter() - c0) * 1e3 / e2e_steps
    e2e_ms = max_over_ranks(e2e_ms, dist, dev)
    fa.fa_device_status()
    elem = B * H * N * d * 2
    h2d = 4 * elem
    d2h = 4 * elem + B * H * N * 4

    result = None
    if rank == 0:
        peak = float(peaks["bf16_tflops"])
        # the dK/dV kernel's own work: 4 GEMMs (S^T, dP^T, dV, dK) = 2 F with the split
        # strategy, 5 (with the dQ partials) = 2.5 F with the accumulated one
        dkdv_flops = (2.0 if split else 2.5) * F
        dkdv_tflops = dkdv_flops / (parts[2] * 1e-3) / 1e12
        fwd_tflops = F / (parts[0] * 1e-3) / 1e12
        bwd_ms = parts[1] + parts[2] + parts[3]
        naive_sp = 2 * N * N * 2 * B * H
        traffic, traffic_src = captured_traffic() if (split and w.name.startswith("C4")) else (None, "no capture")
        result = {
            "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
            "data": "synthetic (seeded N(0,1) Q, K, V, dO; no dataset)",
            "config": {"workload": w.name, "B": B, "H": H, "N": N, "d": d, "causal": w.causal,
                       "global_batch": B * world, "seq_len": N, "parallelism": f"independent heads x{world}",
                       "flop_count": "fwd+bwd = 2.5 * 4*B*H*N^2*d (halved causal)",
                       "l2": "inputs larger than L2 (each of Q, K, V, dO is %.0f MB > 129 MB)" % (elem / 1e6)},
            "fwd_tflops": round(fwd_tflops, 1), "fwd_frac_of_peak": round(fwd_tflops / peak, 4),
            "fwdbwd_frac_of_peak": round(value / world / peak, 4),
            "fwdbwd_tflops_3p5F": round(3.5 * F / (ms_step * 1e-3) / 1e12, 1),
            "bwd_tflops_2p5F": round(2.5 * F / (bwd_ms * 1e-3) / 1e12, 1),
            "kernel_ms": ({"fa_fwd": round(parts[0], 4), "bwd_preprocess": round(parts[1], 4),
                           "bwd_dk_dv": round(parts[2], 4), "bwd_dq": round(parts[3], 4)} if split else
                          {"fa_fwd": round(parts[0], 4), "bwd_preprocess": round(parts[1], 4),
                           "bwd_dkdv": round(parts[2], 4), "bwd_dq_convert": round(parts[3], 4)}),
            "roofline": {"bound": "tensor",
                         "kernel": f"{'fa_bwd_dkdv_split_kernel' if split else 'fa_bwd_dkdv_kernel'}"
                                   f"<{128 if d == 96 else d},{'causal' if w.causal else 'non-causal'},{w.dtype}>",
                         "achieved": round(dkdv_tflops, 1), "peak": peak, "unit": "TFLOP/s",
                         "frac": round(dkdv_tflops / peak, 4),
                         "traffic": traffic, "traffic_source": traffic_src,
                         "peak_source": f"{peak_src} bf16_tflops (burst)",
                         "algorithmic": ("8*N^2*d per head (4 GEMMs: S^T, dP^T, dV, dK), halved causal, per launch"
                                         if split else
                                         "10*N^2*d per head (5 GEMMs), halved causal, per launch")},
            "peak_memory_bytes": int(peak_mem), "inputs_bytes": int(mem_inputs),
            "naive_sp_bytes": int(naive_sp),
            "e2e": {"value": round(world * 2.5 * F / (e2e_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                    "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                    "ms_per_step": round(e2e_ms, 3),
                    "overlap": "step i+1's inputs copied in and step i's results copied out on two side "
                               "streams while step i+1 computes",
                    "serial_ms_per_step": round(e2e_serial_ms, 3),
                    "serial_value": round(world * 2.5 * F / (e2e_serial_ms * 1e-3) / 1e12, 2)},
            "gpu_launches": 4 * args.steps,
            "clocks": clocks,
        }
    if rank == 0:
        result["bwd_strategies"] = backward_strategies()
        result["bwd_strategies"]["note"] = ("dQ by its own kernel (split: preprocess without accumulator, dK/dV, dQ) "
                                            "vs fp32 dQ partials reduced into an accumulator by the dK/dV kernel "
                                            "(accumulated: preprocess, dK/dV, convert); the step uses "
                                            + ("split" if split else "accumulated"))
        from exact_io_aware_forward_gb300.synth import D1
        import dataclasses
        for key, dw in (("decode", D1), ("decode_nq16", dataclasses.replace(D1, Nq=16, name="D1 Nq=16")),
                        ("decode_nq64", dataclasses.replace(D1, Nq=64, name="D1 Nq=64")),
                        ("decode_d256_nq16", dataclasses.replace(D1, H=16, d=256, Nq=16,
                                                                 name="D1 shape at d=256 H=16 Nq=16"))):
            dms, dbytes, _ = measure_decode(dev, dw, 10, 3)
            dgbs = dbytes / (dms * 1e-3) / 1e9
            result[key] = {"workload": dw.name, "ms": round(dms, 4), "GB_per_s": round(dgbs, 1),
                           "frac_of_hbm_peak": round(dgbs / float(peaks["hbm_gbs"]), 4)}
        from exact_io_aware_forward_gb300.synth import S1
        from exact_io_aware_forward_gb300.synth import V1
        from exact_io_aware_forward_gb300.synth import W96, W256
        result["long"] = measure_long(dev, peak)
        for key, kind, vw in (("blocksparse", "blocksparse", S1), ("dropout", "dropout", w), ("varlen", "varlen", V1),
                              ("d96", "dense", W96), ("d256", "dense", W256)):
            sms, sparts, _, sbufs = measure_variant(dev, kind, vw, 10, 3)
            sF = variant_flops(kind, vw, sbufs[-1])
            result[key] = {"workload": vw.name + (f" p={DROP_P}" if kind == "dropout" else ""),
                            "ms": round(sms, 4), "fwdbwd_tflops": round(2.5 * sF / (sms * 1e-3) / 1e12, 1),
                            "fwd_tflops": round(sF / (sparts[0] * 1e-3) / 1e12, 1),
                            "dkdv_frac_of_peak": round(dkdv_factor(kind, vw) * sF / (sparts[2] * 1e-3) / 1e12 / peak,
                                                       4)}
    if dist:
        dist.destroy_process_group()
    return result


def measure_long(dev, peak):
    """The long-sequence workload (C5: causal, B=1, H=8, N=32768, d=128): fwd,
    dK/dV and fwd+bwd throughput, and the peak device memory of its fwd+bwd
    steps (inputs, outputs and the O(N) workspace) against the 2*N^2*2 bytes
    per head that a naive path would spend on S and P."""
    import torch

    from exact_io_aware_forward_gb300.synth import C5 as w
    torch.cuda.synchronize(dev)
    base = torch.cuda.memory_allocated(dev)
    torch.cuda.reset_peak_memory_stats(dev)
    ms, parts, _, bufs = measure_variant(dev, "dense", w, 10, 3)
    torch.cuda.synchronize(dev)
    used = torch.cuda.max_memory_allocated(dev) - base
    F = w.fwd_flops()
    elem = w.B * w.H * w.N * w.d * 2
    return {"workload": w.name, "ms": round(ms, 4), "fwdbwd_tflops": round(2.5 * F / (ms * 1e-3) / 1e12, 1),
            "fwdbwd_frac_of_peak": round(2.5 * F / (ms * 1e-3) / 1e12 / peak, 4),
            "fwd_tflops": round(F / (parts[0] * 1e-3) / 1e12, 1),
            "fwd_frac_of_peak": round(F / (parts[0] * 1e-3) / 1e12 / peak, 4),
            "dkdv_frac_of_peak": round(dkdv_factor("dense", w) * F / (parts[2] * 1e-3) / 1e12 / peak, 4),
            "peak_memory_bytes": int(used), "inputs_bytes": int(4 * elem),
            "naive_sp_bytes": int(2 * w.N * w.N * 2 * w.B * w.H),
            "memory": "peak torch allocation of the fwd+bwd steps above the allocations before them: Q, K, V, dO, "
                      "O, LSE, dQ, dK, dV and the backward workspace"}


def run_reference(args, w, world, rank):
    """The float64 CPU oracle as the baseline arm: each step is a bounded
    sample (whole heads of the same workload) on the host cores."""
    if rank != 0:
        return None
    for _ in range(args.warmup):
        oracle_sample(w, 0.0, 1)
    vals, heads_total, spent_total, threads = [], 0, 0.0, 1
    for _ in range(args.steps):
        v, heads, spent, threads = oracle_sample(w, 0.0, 1)
        vals.append(v)
        heads_total += heads
        spent_total += spent
    value = heads_total * 2.5 * w.fwd_flops() / w.heads / spent_total / 1e12
    sample = f"{heads_total} whole head(s) of {w.name} over {args.steps} steps, float64 NumPy oracle"
    return {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(spent_total * 1e3 / args.steps, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": w.causal},
        "impl": "reference",
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="C4", help="C2, C3N, C3C, C4, C5, W96 (d=96) or W256 (d=256)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--mode", default="train", choices=["train", "decode", "blocksparse", "dropout", "varlen"],
                    help="train: fwd+bwd step (the headline); decode: split-KV decoding line; "
                         "blocksparse: fwd+bwd under a 128x128 block mask; dropout: fwd+bwd of the "
                         "training workload with dropout p=0.1; varlen: fwd+bwd of a packed batch of "
                         "16 causal sequences")
    ap.add_argument("--cpu-budget", type=float, default=10.0, help="seconds of oracle timing (rank 0, N=1)")
    ap.add_argument("--nq", type=int, default=1, help="--mode decode: queries per head (1: the D1 workload)")
    ap.add_argument("--decode-d", type=int, default=128, choices=[64, 128, 256],
                    help="--mode decode: head dimension (256 runs the D1 keys with H = 16)")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    from exact_io_aware_forward_gb300.synth import WORKLOADS
    w = WORKLOADS[args.workload]
    world, rank, local = dist_env()
    if args.impl == "ours" and args.mode in ("decode", "blocksparse", "dropout", "varlen"):
        from exact_io_aware_forward_gb300 import build as fa_build
        fa_build.build()
        if args.mode == "decode":
            out = run_decode(args, world, rank, local)
        else:
            out = run_variant(args, world, rank, local, args.mode)
        if rank == 0:
            print(json.dumps(out), flush=True)
        return
    if args.impl == "reference":
        out = run_reference(args, w, world, rank)
    else:
        from exact_io_aware_forward_gb300 import build as fa_build
        fa_build.build()
        out = run_gpu(args, w, world, rank, local)
        if out is not None and world == 1:
            v, heads, spent, threads = oracle_sample(w, args.cpu_budget, 64)
            out["cpu_baseline"] = {"value": v, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                                   "sample": f"{heads} whole head(s) of {w.name} (N={w.N}, d={w.d}), "
                                             f"float64 forward + explicit backward, {spent:.1f} s"}
    if out is not None:
        print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
