#!/usr/bin/env python3
"""Benchmark of the USP-Attention forward hot path on GB300 (one JSON line on stdout, rank 0).

A step is one pass of the whole hot path over one batch of the workload: for every head group, the
zigzag split of Q, K, V (a1) composed with AllToAll4D (a2) in one launch, ring attention with the LSE
merge (a3 + a4) and the inverse AllToAll4D of out and lse (a5). ``value`` is the causal-adjusted attention FLOPs of the step
(2 * bs * hq * L^2 * hd) divided by the step time, in TFLOP/s, aggregated over all ranks (each rank
runs an independent replica: the virtual-rank grid lives inside one device, nothing is exchanged).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload I] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from seeded_inputs import WORKLOADS, default_seed, make_rows, make_workload_qkv  # noqa: E402

# the largest single-GPU workload: GQA 32/8, L = 262144, u2 x r4, head groups of 8 query heads
DEFAULT_WORKLOAD = 4
L2_BYTES = 129 * 10 ** 6
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
# DRAM bytes per attention launch from ncu captures, keyed by workload and kernel source hash
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "attn_tc_traffic.json")
# GB300 dense bf16 tensor peak (nominal, without 2:4 sparsity): the metric's "% of dense peak"
DENSE_BF16_NOMINAL_TFLOPS = 2250.0
# a timed region at least this long runs under the power cap: the sustained peak applies
SUSTAINED_REGION_S = 1.0
# the forward attention kernel's sources: the traffic figure is valid only for this exact code
ATTN_SRCS = [os.path.join(ROOT, "sequence_long_context_zigzag_gb300", "csrc", f)
             for f in ("attn_tc.cu", "tc_ptx.cuh", "tc_common.cuh")]
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: about half a second of steps, at least 20)")
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", type=int, default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="target CPU work of the oracle baseline")
    return ap.parse_args()


# ------------------------------------------------------------------------------------------------
# distributed plumbing (barrier and max over ranks only; no data-path collective)
# ------------------------------------------------------------------------------------------------
class Dist:
    def __init__(self, backend=None):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            dist.init_process_group(backend=backend or ("nccl" if torch.cuda.is_available() else "gloo"))
            self.pg = dist

    def barrier(self):
        if self.pg:
            if torch.cuda.is_available() and self.pg.get_backend() == "nccl":
                self.pg.barrier(device_ids=[torch.cuda.current_device()])
            else:
                self.pg.barrier()

    def max(self, x: float) -> float:
        if not self.pg:
            return x
        dev = "cuda" if self.pg.get_backend() == "nccl" else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


def load_peaks():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return FALLBACK, "fallback"


def pick_peak(peaks, src, region_s):
    """The bf16 roofline denominator for a kernel timed over ``region_s`` seconds: the burst cuBLAS
    rate for a region shorter than SUSTAINED_REGION_S, the sustained (power-capped) rate otherwise.
    Returns (TFLOP/s, a sentence saying which and why)."""
    if region_s >= SUSTAINED_REGION_S:
        key, why = "bf16_tflops_sustained", f"timed region {region_s:.2f} s >= {SUSTAINED_REGION_S:.0f} s"
    else:
        key, why = "bf16_tflops", f"timed region {region_s:.3f} s < {SUSTAINED_REGION_S:.0f} s (burst)"
    val = peaks.get(key, FALLBACK[key])
    return val, f"{src} {key} = {val} TFLOP/s ({why})"


# ------------------------------------------------------------------------------------------------
# clocks during the timed region
# ------------------------------------------------------------------------------------------------
class ClockSampler:
    """nvidia-smi samples every 50 ms from start() to stop(); stop(t0, t1) keeps the samples whose
    timestamps fall inside the timed region [t0, t1] (host wall clock), or all of them if none do."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        self.path = None
        self.idx = gpu_index

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50",
                 "-i", str(self.idx)], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self, t0=None, t1=None):
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    rows.append((ts, float(parts[2]), float(parts[3]), parts[6:10]))
                except ValueError:
                    continue
        os.unlink(self.path)
        inside = [r for r in rows if t0 is not None and t0 <= r[0] <= t1]
        window = "timed region" if inside else "sampler run (no sample fell inside the timed region)"
        use = inside or rows
        if not use:
            return None
        reasons = sorted({nm for r in use for nm, val in zip(names, r[3]) if val.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in use), "sm_max_mhz": max(r[2] for r in use),
                "reasons": reasons, "samples": len(use), "window": window}


def gpu_index(local_rank):
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        ids = [x for x in vis.split(",") if x.strip()]
        if local_rank < len(ids):
            return ids[local_rank]
    return str(local_rank)


# ------------------------------------------------------------------------------------------------
# the step
# ------------------------------------------------------------------------------------------------
class Step:
    """Preallocated buffers and the ABI calls of one step (no allocation inside the timed loop)."""

    def __init__(self, usp, w, q, k, v):
        self.usp, self.w = usp, w
        self.q, self.k, self.v = q, k, v
        rd, ud, bs, L, hd = w.rd, w.ud, w.bs, w.L, w.hd
        hc = w.head_chunk or w.hq
        G = w.hq // w.hkv
        hkc = hc // G
        Lu, Lr = L // (rd * ud), L // rd
        dev, dt = q.device, q.dtype
        self.groups = [(g0, g0 // G) for g0 in range(0, w.hq, hc)]
        self.hc, self.hkc = hc, hkc
        hks = usp.heads_per_rank(hkc, ud) * ud  # head-sharded K/V heads (replicas when hkc < ud)
        self.qh = torch.empty(rd, ud, hc // ud, bs, Lr, hd, device=dev, dtype=dt)
        self.kh = torch.empty(rd, ud, hks // ud, bs, Lr, hd, device=dev, dtype=dt)
        self.vh = torch.empty_like(self.kh)
        self.oh = torch.empty_like(self.qh)
        self.lh = torch.empty(rd, ud, hc // ud, bs, Lr, device=dev, dtype=torch.float32)
        self.o_loc = torch.empty(rd, ud, bs, Lu, w.hq, hd, device=dev, dtype=dt)
        self.l_loc = torch.empty(rd, ud, bs, Lu, w.hq, device=dev, dtype=torch.float32)
        es = q.element_size()
        # algorithmic permute bytes per step: one read + one write of every moved tensor (the composed
        # split + all-to-all reads and writes each of Q, K, V once; replicated K/V heads are read once
        # and written once per replica)
        tok = bs * L
        self.permute_bytes = (tok * (2 * hc + 2 * (hkc + hks)) * hd * es
                              + 2 * tok * hc * (hd * es + 4)) * len(self.groups)
        self.launches_per_step = 3 * len(self.groups)
        self.attn_events = []
        self.perm_events = []

    def run(self, record=False):
        usp, w = self.usp, self.w
        rd, ud = w.rd, w.ud
        st = torch.cuda.current_stream()
        for g0, gk in self.groups:
            if record:
                e0 = torch.cuda.Event(enable_timing=True)
                e0.record(st)
            usp.usp_extract_a2a([self.q, self.k, self.v], [self.qh, self.kh, self.vh], rd, ud,
                                h0s=[g0, gk, gk], Hs=[self.hc, self.hkc, self.hkc])
            if record:
                e1 = torch.cuda.Event(enable_timing=True)
                e1.record(st)
            usp.usp_attn_fwd(self.qh, self.kh, self.vh, self.oh, self.lh, causal=w.causal, hkv=self.hkc)
            if record:
                e2 = torch.cuda.Event(enable_timing=True)
                e2.record(st)
            # AllToAll4D's inverse of out and lse, one launch
            usp.usp_a2a4d_multi([self.oh, self.lh], [self.o_loc, self.l_loc], rd, ud, -1, h0s=[g0, g0],
                                Hs=[self.hc, self.hc])
            if record:
                e3 = torch.cuda.Event(enable_timing=True)
                e3.record(st)
                self.attn_events.append((e1, e2))
                self.perm_events.append((e0, e1, e2, e3))


def time_backward(usp, w, step, reps=5):
    """The ring attention backward (usp_attn_bwd: the dk/dv and dq kernels) of the last head group,
    on the step's head-sharded buffers and a seeded upstream gradient, median of ``reps`` launches.
    Algorithmic FLOPs: 2.5x the forward's (five matrix products per causal pair instead of two)."""
    if w.dtype != "bf16":
        return None
    g = torch.Generator(device="cuda").manual_seed(7)
    dout = torch.randn(step.oh.shape, device="cuda", generator=g).to(step.oh.dtype)
    delta = torch.empty_like(step.lh)
    dq, dk, dv = torch.empty_like(step.qh), torch.empty_like(step.kh), torch.empty_like(step.vh)
    usp.usp_attn_fwd(step.qh, step.kh, step.vh, step.oh, step.lh, causal=w.causal, hkv=step.hkc)
    usp.usp_attn_bwd_delta(step.oh, dout, delta)

    def once():
        usp.usp_attn_bwd(step.qh, step.kh, step.vh, dout, step.lh, delta, dq, dk, dv, causal=w.causal, hkv=step.hkc)

    once()
    ts = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        once()
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1) / 1e3)
    usp.usp_check()
    t = statistics.median(ts)
    flops = 2.5 * w.causal_flops / len(step.groups)
    peaks, src = load_peaks()
    peak, peak_src = pick_peak(peaks, src, sum(ts))
    return {"kernel": "usp_attn_bwd (dk/dv and dq tensor-core kernels)", "ms": t * 1e3,
            "tflops": flops / t / 1e12, "frac_of_peak": flops / t / 1e12 / peak, "peak_source": peak_src,
            "frac_of_dense_nominal": flops / t / 1e12 / DENSE_BF16_NOMINAL_TFLOPS,
            "algorithmic_flops": flops, "note": f"one head group ({step.hc} query heads), median of {reps}"}


def packing(usp, w, step, reps=5):
    """The pages' packing case (ByteScale): the same total length packed as 1, 2 and L/1024 samples,
    each sample attending only within itself. The ring attention of the last head group is timed for
    each packing (median of ``reps``); FLOPs count each sample's causal pairs, 4 hq hd len^2 / 2."""
    if w.dtype != "bf16" or not w.causal:
        return None
    res = {}
    for n in (1, 2, max(2, w.L // 1024)):
        if w.L % n:
            continue
        cu = torch.arange(0, w.L + 1, w.L // n, dtype=torch.int32, device="cuda")
        kw = {} if n == 1 else {"cu_seqlens": cu}
        ts = []
        for r in range(reps + 1):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            usp.usp_attn_fwd(step.qh, step.kh, step.vh, step.oh, step.lh, causal=True, hkv=step.hkc, **kw)
            e1.record()
            torch.cuda.synchronize()
            if r:
                ts.append(e0.elapsed_time(e1) / 1e3)
        t = statistics.median(ts)
        fl = 4.0 * step.hc * w.hd * n * (w.L // n) ** 2 / 2 * w.bs
        res[f"{n}x{w.L // n}"] = {"ms": round(t * 1e3, 4), "tflops": round(fl / t / 1e12, 1)}
    usp.usp_check()
    return res


def rank_balance(usp, w, q, k, v, reps=5):
    """Per-ring-rank attention time under each sequence split (each rank's query rows computed alone,
    median of ``reps`` launches): the load imbalance a multi-GPU ring would see, measured on the device.
    The pages' claim: a contiguous split leaves the last of 4 ranks with 1.75x the mean work, zigzag
    balances it exactly."""
    hc = w.head_chunk or w.hq
    G = w.hq // w.hkv
    hkc = hc // G
    rd, ud, bs, L, hd = w.rd, w.ud, w.bs, w.L, w.hd
    dev, dt = q.device, q.dtype
    qh = torch.empty(rd, ud, hc // ud, bs, L // rd, hd, device=dev, dtype=dt)
    kh = torch.empty(rd, ud, usp.heads_per_rank(hkc, ud), bs, L // rd, hd, device=dev, dtype=dt)
    vh = torch.empty_like(kh)
    oh = torch.empty_like(qh)
    lh = torch.empty(qh.shape[:5], device=dev, dtype=torch.float32)
    res = {}
    for split in ("zigzag", "basic", "stripe"):
        usp.usp_extract_a2a([q, k, v], [qh, kh, vh], rd, ud, h0s=[0, 0, 0], Hs=[hc, hkc, hkc], split=split)
        ms = []
        for r in range(rd):
            ts = []
            for _ in range(reps):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                usp.usp_attn_fwd(qh, kh, vh, oh, lh, causal=w.causal, split=split, ring_rank=r, hkv=hkc)
                e1.record()
                torch.cuda.synchronize()
                ts.append(e0.elapsed_time(e1))
            ms.append(statistics.median(ts))
        res[split] = {"rank_ms": [round(x, 4) for x in ms], "max_over_mean": max(ms) / (sum(ms) / len(ms))}
    usp.usp_check()
    res["note"] = f"first head group ({hc} query heads), each ring rank's rows alone; median of {reps}"
    return res


def secondary_workloads(usp, main_wi, steps=5, warmup=2):
    """The other bf16 workloads, each timed briefly after the main timed region (not clock-sampled):
    the same step (split + AllToAll4D, ring attention, inverse, per head group) on seeded N(0,1)
    inputs drawn on the device. Reported as extra keys beside the main workload's line."""
    res = []
    for wi, w in enumerate(WORKLOADS):
        if wi == main_wi or w.dtype != "bf16":
            continue
        g = torch.Generator(device="cuda").manual_seed(default_seed(wi))
        q = torch.randn(w.bs, w.L, w.hq, w.hd, device="cuda", generator=g).to(torch.bfloat16)
        k = torch.randn(w.bs, w.L, w.hkv, w.hd, device="cuda", generator=g).to(torch.bfloat16)
        v = torch.randn(w.bs, w.L, w.hkv, w.hd, device="cuda", generator=g).to(torch.bfloat16)
        step = Step(usp, w, q, k, v)
        for _ in range(warmup):
            step.run()
        torch.cuda.synchronize()
        st = torch.cuda.current_stream()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        for _ in range(steps):
            step.run(record=True)
        e1.record(st)
        torch.cuda.synchronize()
        usp.usp_check()
        t = e0.elapsed_time(e1) / 1e3 / steps
        attn = sum(a.elapsed_time(b) for a, b in step.attn_events) / 1e3 / len(step.attn_events)
        perm = sum(a.elapsed_time(b) + c.elapsed_time(d) for a, b, c, d in step.perm_events) / 1e3 / steps
        res.append({"workload": w.name, "ms_per_step": round(t * 1e3, 3),
                    "step_tflops": round(w.causal_flops / t / 1e12, 1),
                    "attn_kernel_tflops": round(w.causal_flops / len(step.groups) / attn / 1e12, 1),
                    "permute_gbs": round(step.permute_bytes / perm / 1e9, 1), "steps": steps})
        del q, k, v, step
        torch.cuda.empty_cache()
    return res


def attn_src_hash():
    """First 16 hex digits of the SHA-256 of the forward kernel's sources, concatenated in order."""
    hs = hashlib.sha256()
    for fn in ATTN_SRCS:
        with open(fn, "rb") as f:
            hs.update(f.read())
    return hs.hexdigest()[:16]


def traffic_for_current_kernel(w):
    """DRAM bytes per attention launch (read + write) of workload ``w`` from the committed ncu record,
    if one was taken on this workload and on the attention kernel's source as it is now (else None)."""
    try:
        with open(TRAFFIC_FILE) as f:
            recs = json.load(f)["records"]
        h = attn_src_hash()
    except (OSError, ValueError, KeyError):
        return None
    for r in recs:
        if r.get("workload") == w.name and r.get("attn_src_sha256_16") == h:
            return int(r["dram_bytes_per_launch"])
    return None


# ------------------------------------------------------------------------------------------------
# the oracle on the host cores (the CPU baseline, and the reference arm)
# ------------------------------------------------------------------------------------------------
def oracle_rows_flops(w, rows):
    """Causal FLOPs of the selected query rows for every head: 4 hd (i + 1) per (row, head)."""
    n = sum((int(i) + 1) if w.causal else w.L for i in rows)
    return 4.0 * w.hd * n * w.hq * w.bs


def time_oracle(w, q, k, v, target_s, seed):
    import oracle
    oracle.build()
    n = 8
    rows = make_rows(w.L, w.c, n, seed)[:n]
    while True:
        t0 = time.perf_counter()
        oracle.attn_direct(q, k, v, causal=w.causal, rows=rows)
        dt = time.perf_counter() - t0
        if dt >= target_s or len(rows) >= w.L:
            break
        grow = max(2.0, min(16.0, target_s / max(dt, 1e-3)))
        n = min(w.L, int(n * grow) + 1)
        rows = list(range(0, w.L, max(1, w.L // n)))[:n]
    flops = oracle_rows_flops(w, rows)
    res = {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": oracle.num_threads(), "kind": "oracle",
           "sample": f"{len(rows)} query rows x {w.hq} heads of {w.name} (fp64 direct attention, "
                     f"{flops / 1e9:.1f} GFLOP causal-adjusted, {dt:.1f} s)"}
    res.update(time_oracle_permutes(w, q, k, v, seed))
    return res


def time_oracle_permutes(w, q, k, v, seed):
    """The oracle's index maps on the host (numpy gathers, one thread): the outputs of one step's
    permutes for the first head group -- split + AllToAll4D of Q, K, V and the inverse AllToAll4D of
    an out-shaped and an lse-shaped tensor -- over the full tensors of that group. GB/s counts the
    same algorithmic bytes as the GPU's permutes of one group (one read and one write of each
    tensor), so the two rates compare like for like."""
    import numpy as np

    import oracle
    hc = w.head_chunk or w.hq
    G = w.hq // w.hkv
    hkc = hc // G

    def raw(t):
        return t.view(torch.int16).numpy() if t.dtype == torch.bfloat16 else t.numpy()

    t0 = time.perf_counter()
    qh = oracle.a2a_fwd(oracle.extract_local(raw(q), w.rd, w.ud, 0, hc), w.ud)
    kh = oracle.a2a_fwd(oracle.extract_local(raw(k), w.rd, w.ud, 0, hkc), w.ud)
    vh = oracle.a2a_fwd(oracle.extract_local(raw(v), w.rd, w.ud, 0, hkc), w.ud)
    o_loc = oracle.a2a_inv(qh, w.ud)
    l_loc = oracle.a2a_inv(np.zeros(qh.shape[:5], dtype=np.float32), w.ud)
    dt = time.perf_counter() - t0
    es = 2 if w.dtype == "bf16" else 4
    tok = w.bs * w.L
    hks = kh.shape[2] * w.ud
    moved = tok * (2 * hc + 2 * (hkc + hks)) * w.hd * es + 2 * tok * hc * (w.hd * es + 4)
    del vh, o_loc, l_loc
    return {"permute_gbs": moved / dt / 1e9, "permute_cores": 1,
            "permute_sample": f"first head group ({hc} query heads, {hkc} KV heads) of {w.name}: split + "
                              f"AllToAll4D of Q, K, V and the inverse AllToAll4D of out and lse as numpy index "
                              f"gathers, {moved / 1e9:.2f} GB algorithmic in {dt:.2f} s"}


def run_reference(args, dist):
    """The reference arm: the oracle as it stands, timed on this host's cores."""
    if dist.rank != 0:
        return
    import oracle
    oracle.build()
    wi = args.workload
    w = WORKLOADS[wi]
    q, k, v = make_workload_qkv(w, default_seed(wi))
    if args.steps is None:
        args.steps = 5
    # a fixed bounded sample per step, sized so that the whole run takes about a minute and a half on
    # this host (2 s per step at most)
    per_step = min(2.0, max(0.05, 90.0 / (args.steps + args.warmup)))
    probe = list(range(w.L // 8, w.L, w.L // 4))[:4]
    t0 = time.perf_counter()
    oracle.attn_direct(q, k, v, causal=w.causal, rows=probe)
    per_row = max((time.perf_counter() - t0) / len(probe), 1e-6)
    n = max(1, min(w.L, int(per_step / per_row)))
    rows = list(range(0, w.L, max(1, w.L // n)))[:n]
    for _ in range(args.warmup):
        oracle.attn_direct(q, k, v, causal=w.causal, rows=rows)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.attn_direct(q, k, v, causal=w.causal, rows=rows)
    dt = (time.perf_counter() - t0) / args.steps
    flops = oracle_rows_flops(w, rows)
    value = flops / dt / 1e12
    cb = {"value": value, "unit": "TFLOP/s", "cores": oracle.num_threads(), "kind": "oracle",
          "sample": f"{len(rows)} query rows x {w.hq} heads of {w.name} per step (fp64 direct attention)"}
    line = {"impl": "reference", "metric": METRIC, "value": value,
            "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic", "config": workload_config(w),
            "cpu_baseline": cb, "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                                        "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def e2e_head_chunk(w):
    """Head groups for the host-buffer pipeline: the workload's own chunking, else about four groups
    (each a multiple of hq/hkv whose KV heads divide by ud or divide ud), so copies overlap kernels."""
    if w.head_chunk:
        return w.head_chunk
    G = w.hq // w.hkv
    for n in (4, 2):
        hc = w.hq // n
        if w.hq % n == 0 and hc % G == 0 and hc % w.ud == 0 and ((hc // G) % w.ud == 0 or w.ud % (hc // G) == 0):
            return hc
    return None


METRIC = "fwd causal-adjusted attention TFLOP/s (bf16) and % of GB300 dense peak; permute GB/s"


def step_working_set_bytes(w):
    """Device bytes one step touches: natural Q, K, V; the head-sharded Q, K, V and out of one head
    group (K/V replicated on every Ulysses rank when a group has fewer KV heads than ranks); the
    sequence-sharded out."""
    es = 2 if w.dtype == "bf16" else 4
    tok = w.bs * w.L
    hc = w.head_chunk or w.hq
    hkc = hc // (w.hq // w.hkv)
    hks = hkc if hkc % w.ud == 0 else w.ud
    heads = w.hq + 2 * w.hkv + hc + 2 * hks + hc + w.hq
    return tok * heads * w.hd * es


def workload_config(w):
    """The config both arms report: the workload, and how L2 is kept out of the timing (the step's
    working set is larger than L2, so nothing is flushed)."""
    return {"workload": w.name, "bs": w.bs, "seq_len": w.L, "hq": w.hq, "hkv": w.hkv, "head_dim": w.hd,
            "ulysses_degree": w.ud, "ring_degree": w.rd, "head_chunk": w.head_chunk, "causal": w.causal,
            "parallelism": f"virtual u{w.ud}xr{w.rd} grid on one GPU; replicas across GPUs",
            "l2": l2_statement(step_working_set_bytes(w))}


def l2_statement(ws):
    mib = ws / 2**20
    if ws > 129e6:
        return "step working set %.0f MiB > L2 (129 MB); no flush" % mib
    return "step working set %.0f MiB fits in L2 (129 MB): warm-cache timing of a small parity workload" % mib


# ------------------------------------------------------------------------------------------------
def main():
    args = parse()
    dist = Dist()
    if args.impl == "reference":
        run_reference(args, dist)
        dist.close()
        return
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(dist.local_rank)
    import sequence_long_context_zigzag_gb300 as usp

    wi = args.workload
    w = WORKLOADS[wi]
    seed = default_seed(wi)
    q_h, k_h, v_h = make_workload_qkv(w, seed)
    q, k, v = q_h.cuda(), k_h.cuda(), v_h.cuda()
    step = Step(usp, w, q, k, v)
    flops = w.causal_flops
    peaks, peak_src = load_peaks()

    for _ in range(args.warmup):
        step.run()
    usp.usp_check()
    if args.steps is None:
        # about half a second of timed steps (at least 20), the same count on every rank
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        step.run()
        torch.cuda.synchronize()
        args.steps = int(dist.max(min(2000.0, max(20.0, 0.5 / max(time.perf_counter() - t0, 1e-6)))))

    # ---- device-timed region ----------------------------------------------------------------
    sampler = ClockSampler(gpu_index(dist.local_rank))
    dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.3)  # nvidia-smi's start-up, so that its samples cover the timed region
    st = torch.cuda.current_stream()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_wall0 = time.time()
    ev0.record(st)
    for _ in range(args.steps):
        step.run(record=True)
    ev1.record(st)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    dist.barrier()
    clocks = sampler.stop(t_wall0, t_wall1)
    usp.usp_check()
    t_step = ev0.elapsed_time(ev1) / 1e3 / args.steps
    t_step_max = dist.max(t_step)
    attn_t = [a.elapsed_time(b) / 1e3 for a, b in step.attn_events]
    perm_t = [(a.elapsed_time(b) + c.elapsed_time(d)) / 1e3 for a, b, c, d in step.perm_events]
    per_group_flops = flops / len(step.groups)
    attn_avg = sum(attn_t) / len(attn_t)
    attn_tflops = per_group_flops / attn_avg / 1e12
    perm_gbs = step.permute_bytes / (sum(perm_t) / args.steps) / 1e9

    # ---- end to end through the public API, host buffers ------------------------------------
    # usp_forward_host: pinned host Q/K/V in, pinned host out/lse back, every step (the library moves
    # the bytes over the CPU-GPU link with its permute kernels and the copy engines); the
    # caller-owned workspace is allocated once, outside the timed loop
    qp, kp, vp = (x.pin_memory() for x in (q_h, k_h, v_h))
    out_h = torch.empty(w.bs, w.L, w.hq, w.hd, dtype=q_h.dtype).pin_memory()
    lse_h = torch.empty(w.bs, w.L, w.hq, dtype=torch.float32).pin_memory()
    h2d = sum(x.numel() * x.element_size() for x in (qp, kp, vp))
    d2h = out_h.numel() * out_h.element_size() + lse_h.numel() * 4
    chunk = e2e_head_chunk(w)
    ws = torch.empty(usp.usp_forward_workspace_size(qp, kp, w.ud, w.rd, chunk, host=True, causal=w.causal),
                     dtype=torch.uint8, device="cuda")

    def e2e_step():
        usp.usp_forward_host(qp, kp, vp, out_h, lse_h, w.ud, w.rd, causal=w.causal, head_chunk=chunk, workspace=ws)

    for _ in range(max(1, args.warmup)):
        e2e_step()
    torch.cuda.synchronize()
    dist.barrier()
    n_e2e = max(1, args.steps // 2)
    t0 = time.perf_counter()
    for _ in range(n_e2e):
        e2e_step()
    torch.cuda.synchronize()
    t_e2e = dist.max((time.perf_counter() - t0) / n_e2e)
    dist.barrier()
    usp.usp_check()

    # ---- per-ring-rank work under the three splits (outside the timed region) ----------------
    balance = rank_balance(usp, w, q, k, v) if w.rd > 1 else None

    # ---- the backward of one head group's ring attention (outside the timed region) ----------
    backward = time_backward(usp, w, step, reps=min(20, max(3, args.steps // 2)))
    packed = packing(usp, w, step)

    # ---- the other bf16 workloads, briefly (outside the timed region) ------------------------
    others = secondary_workloads(usp, wi) if dist.world == 1 else None

    # ---- CPU baseline (the oracle on the host cores), rank 0 at N = 1 -----------------------
    cpu = None
    if dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline:
        cpu = time_oracle(w, q_h, k_h, v_h, args.cpu_seconds, seed)

    if dist.rank == 0:
        # the timed region is the whole step loop: its length decides burst or sustained peak
        peak, peak_note = pick_peak(peaks, peak_src, t_step * args.steps)
        hbm = peaks.get("hbm_gbs", FALLBACK["hbm_gbs"])
        # exponentials of the causal softmax, bs * hq * L^2 / 2 per step (one per visible pair)
        exps = w.bs * w.hq * float(w.L) ** 2 / (2 if w.causal else 1)
        line = {
            "metric": METRIC,
            "value": dist.world * flops / t_step_max / 1e12,
            "unit": "TFLOP/s",
            "n_gpus": dist.world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": t_step_max * 1e3,
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "bf16" if w.dtype == "bf16" else "f32",
            "data": "synthetic: seeded N(0,1) Q/K/V rounded to bf16",
            "config": workload_config(w),
            "attn_kernel_tflops": attn_tflops,
            "attn_frac_of_dense_peak": attn_tflops / DENSE_BF16_NOMINAL_TFLOPS,
            "attn_frac_of_dense_peak_note": f"of GB300's nominal dense bf16 peak, {DENSE_BF16_NOMINAL_TFLOPS:.0f} "
                                            "TFLOP/s (roofline.frac is against the measured cuBLAS rate)",
            "attn_exp_per_s": exps / len(step.groups) / attn_avg,
            "permute_gbs": perm_gbs,
            "permute_frac_of_hbm": perm_gbs / hbm,
            "roofline": {"bound": "tensor", "achieved": attn_tflops, "peak": peak, "unit": "TFLOP/s",
                         "frac": attn_tflops / peak, "traffic": traffic_for_current_kernel(w),
                         "peak_source": peak_note,
                         "kernel": "usp_attn_fwd (bf16 ring attention)",
                         "algorithmic_flops_per_launch": per_group_flops},
            "e2e": {"value": dist.world * flops / t_e2e / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h,
                    "api": f"usp_forward_host (pinned host buffers, read and written by the permute kernels "
                           f"over the CPU-GPU link; head_chunk={chunk}; wall clock)"},
            "gpu_launches": step.launches_per_step * args.steps,
            "rank_balance": balance,
            "backward": backward,
            "packing": packed,
            "other_workloads": others,
            "other_workloads_note": "each timed for 5 steps after the main timed region, inputs drawn on the "
                                    "device, not clock-sampled",
            "clocks": clocks,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line))
    dist.close()


if __name__ == "__main__":
    main()
