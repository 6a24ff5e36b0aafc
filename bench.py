#!/usr/bin/env python3
"""Benchmark: HSTU attention forward + backward throughput on one GB300.

A step is one forward and one backward pass (all hot-path kernels: tile
scheduler, forward, dQ, dK/dV) over one batch of the recommender-training
workload: B = 32 sequences with lengths uniform in [256, 1024], H = 4,
D = 128, bf16 q/k/v/dO ~ N(0, 1), alpha = 1/sqrt(128), L_scale = max_seqlen,
causal.  Inputs are synthetic (seed 0) and resident in HBM before timing.

The metric counts algorithmic tensor FLOPs only, causal-aware:
N = H * sum_b L_b (L_b + 1) / 2 attended pairs; forward 4 D N, backward
10 D N (S recompute, dO V^T, dV, dK in the dK/dV units, dQ = dS K in the dQ
units, one backward launch).

Prints one JSON line.  ``--impl reference`` times the fp64 CPU oracle
instead, on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import tempfile
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "HSTU attn fwd+bwd TFLOP/s (varlen causal bf16) and % of GB300 dense BF16 peak"
WORKLOAD = "recsys"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d["bf16_tflops_sustained"]), "source": "measured"}
    except Exception:
        return dict(FALLBACK_PEAKS, source="fallback")


def pairs(lengths, H, causal):
    """Attended (query, key) pairs times heads; ``causal`` is a bool, a
    (left, right) token window (-1: unbounded side), or ("targets", n): causal
    plus the last n keys of the sequence; Lq = Lk per sequence."""
    if isinstance(causal, tuple) and causal[0] == "targets":
        n = 0
        for L in lengths:
            i = np.arange(L, dtype=np.int64)
            extra = np.maximum(0, L - np.maximum(i + 1, L - causal[1]))  # target keys past i
            n += int((i + 1).sum() + extra.sum())
        return H * n
    if isinstance(causal, tuple):
        left, right = causal
        n = 0
        for L in lengths:
            i = np.arange(L, dtype=np.int64)
            lo = np.zeros(L, dtype=np.int64) if left < 0 else np.maximum(0, i - left)
            hi = np.full(L, L - 1, dtype=np.int64) if right < 0 else np.minimum(L - 1, i + right)
            n += int(np.maximum(0, hi - lo + 1).sum())
        return H * n
    if causal:
        return H * sum(L * (L + 1) // 2 for L in lengths)
    return H * sum(L * L for L in lengths)


def replica_throughput(ms_total, steps, flops_step, world, dist=None, device=None):
    """Whole-job throughput of `world` independent replicas: the slowest
    rank's time (MAX over ranks) for the units all ranks processed.  Returns
    (ms per step, TFLOP/s)."""
    if dist is not None and world > 1:
        import torch
        t = torch.tensor([float(ms_total)], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms_total = float(t.item())
    ms_step = ms_total / steps
    return ms_step, world * flops_step / (ms_step * 1e-3) / 1e12


def workload_config(w, lengths, mask=None):
    d = w.describe()
    d["T"] = int(sum(lengths))
    d["max_seqlen"] = int(max(lengths))
    if mask is not None and isinstance(mask, tuple) and mask[0] == "targets":
        d["mask"] = f"func_tensor: causal plus the last {mask[1]} keys of each sequence"
    elif mask is not None and isinstance(mask, tuple):
        d["mask"] = f"window {mask}"
    d["N_pairs"] = int(pairs(lengths, w.heads, w.causal if mask is None else mask))
    return d


# ---------------------------------------------------------------- clocks
_NVML_REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                 0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}


class NvmlClockSampler:
    """SM clock and throttle reasons read through NVML (the driver's
    management library, read-only queries) from a background thread every
    `period_s`, so that even a timed region of a few milliseconds gets
    samples.  The device is found by its UUID, so the index seen by CUDA need
    not match NVML's."""

    def __init__(self, device_index: int, period_s: float = 2e-4):
        import ctypes
        import threading
        import torch
        self.samples, self.times, self.reasons, self.max_mhz = [], [], set(), None
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        self.dev = ctypes.c_void_p()
        uuid = "GPU-" + str(torch.cuda.get_device_properties(device_index).uuid)
        if self.lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.dev)) != 0:
            raise RuntimeError("NVML device not found")
        mx = ctypes.c_uint()
        if self.lib.nvmlDeviceGetMaxClockInfo(self.dev, 1, ctypes.byref(mx)) == 0:  # 1: SM clock
            self.max_mhz = float(mx.value)
        reasons_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        self.stop_flag = threading.Event()

        def loop():
            clk, rs = ctypes.c_uint(), ctypes.c_ulonglong()
            while not self.stop_flag.is_set():
                if self.lib.nvmlDeviceGetClockInfo(self.dev, 1, ctypes.byref(clk)) == 0:
                    self.samples.append(float(clk.value))
                    self.times.append(time.perf_counter())
                if reasons_fn(self.dev, ctypes.byref(rs)) == 0:
                    for bit, name in _NVML_REASONS.items():
                        if rs.value & bit:
                            self.reasons.add(name)
                self.stop_flag.wait(period_s)

        # the timed loop holds the interpreter lock between its (quick) calls:
        # switch threads often while sampling, and start only once the
        # sampler runs
        self.switch = sys.getswitchinterval()
        sys.setswitchinterval(1e-5)
        self.thread = threading.Thread(target=loop, daemon=True)
        self.thread.start()
        t0 = time.perf_counter()
        while not self.samples and time.perf_counter() - t0 < 1.0:
            time.sleep(1e-4)

    def stop(self):
        self.stop_flag.set()
        self.thread.join(timeout=5)
        sys.setswitchinterval(self.switch)
        try:
            self.lib.nvmlShutdown()
        except Exception:
            pass
        if not self.samples:
            return None
        return {"sm_mhz": statistics.median(self.samples),
                "sm_max_mhz": self.max_mhz if self.max_mhz else max(self.samples),
                "samples": len(self.samples), "reasons": sorted(self.reasons), "source": "nvml"}


class ClockSampler:
    """nvidia-smi sampling during the timed region (used when NVML cannot be
    loaded)."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, path: str):
        self.path = path
        self.proc = None
        try:
            self.f = open(path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={index}", f"--query-gpu={self.Q}", "--format=csv,noheader",
                 "-lms", "50"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1].split()[0]))
                mx.append(float(parts[2].split()[0]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons), "source": "nvidia-smi",
                "nvml_error": getattr(self, "nvml_error", None)}


def start_clock_sampler(local: int, rank: int):
    try:
        return NvmlClockSampler(local)
    except Exception as exc:
        c = ClockSampler(local, os.path.join(os.environ.get("HSTU_CLOCKS_DIR",
                                                            tempfile.gettempdir()),
                                             f"hstu_clocks_rank{rank}.csv"))
        c.nvml_error = f"{type(exc).__name__}: {exc}"
        return c


def kernel_sources_sha() -> str:
    """sha256 (first 16 hex digits) over the CUDA sources of the library, in
    name order: a committed ncu summary whose "sources" line differs was
    taken on other kernels, and its DRAM figures are not reported."""
    import hashlib
    d = os.path.join(ROOT, "generative_recommender_attention_gb300", "csrc")
    h = hashlib.sha256()
    for name in sorted(os.listdir(d)):
        if name.endswith((".cu", ".cuh", ".h")):
            h.update(name.encode())
            h.update(open(os.path.join(d, name), "rb").read())
    return h.hexdigest()[:16]


def summary_traffic(path: str, kernel: str):
    """DRAM bytes per launch of `kernel` from a committed ncu summary (lines
    "traffic <kernel> <bytes>"), if the summary's "sources <sha>" line matches
    the current kernel sources; else None."""
    if not os.path.exists(path):
        return None
    lines = [ln.split() for ln in open(path)]
    if not any(len(p) == 2 and p[0] == "sources" and p[1] == kernel_sources_sha() for p in lines):
        return None
    for p in lines:
        if len(p) == 3 and p[0] == "traffic" and p[1] == kernel:
            return int(p[2])
    return None


# ---------------------------------------------------------------- CPU oracle timing
def oracle_sample(x, w, budget_s: float, start: int = 0, threads: int = 0, mask=None):
    """Times the fp64 oracle fwd+bwd on whole sequences (all heads) of the
    workload, one after another from `start`, until `budget_s` is spent, on
    `threads` host threads (0: all cores).  Returns (flops, seconds,
    n_sequences, threads)."""
    import numpy as np
    import oracle
    threads = oracle.threads(threads if threads > 0 else (os.cpu_count() or 1))
    cu = x["cu_seqlens_q"].tolist()
    B = len(cu) - 1
    L_scale = oracle.resolve_scaling(w.scaling_seqlen, x["max_seqlen_q"])
    D = w.head_dim
    mask = w.causal if mask is None else mask
    flops, secs, n = 0.0, 0.0, 0
    b = start
    while n < B and (n == 0 or secs < budget_s):
        s0, s1 = cu[b], cu[b + 1]
        sub = {k: x[k][s0:s1].double().numpy() for k in ("q", "k", "v", "do")}
        c1 = np.array([0, s1 - s0], dtype=np.int32)
        t0 = time.perf_counter()
        om = mask
        if isinstance(mask, tuple) and mask[0] == "targets":  # the sequence's endpoint rows
            i = np.arange(s1 - s0)
            om = {"func": np.stack([i + 1, np.full_like(i, s1 - s0 - mask[1]),
                                    np.full_like(i, s1 - s0)]).astype(np.int32)}
        oracle.fwd(sub["q"], sub["k"], sub["v"], c1, c1, w.alpha, L_scale, om, threads)
        oracle.bwd(sub["do"], sub["q"], sub["k"], sub["v"], c1, c1, w.alpha, L_scale, om,
                   threads)
        secs += time.perf_counter() - t0
        flops += 14.0 * D * pairs([s1 - s0], w.heads, mask)
        n += 1
        b = (b + 1) % B
    return flops, secs, n, threads


def replayable(fn):
    """fn captured once in a CUDA graph (after one direct call on a side
    stream) and returned as the graph's replay, so that a timed call runs the
    same kernels with the same arguments without the binding's host work
    (tensor allocation, argument marshalling) in the device's critical path.
    Falls back to fn itself when capture fails; the second value says which."""
    import torch
    try:
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            fn()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            fn()
        torch.cuda.synchronize()
        return graph.replay, "CUDA graph of the call, replayed"
    except Exception as exc:
        torch.cuda.synchronize()
        return fn, f"direct calls (graph capture failed: {type(exc).__name__})"


def run_lmsd(args, dev):
    """--lmsd N,D: HBM throughput of the LMSD forward and backward (the op is
    bandwidth-bound), with the bytes each call must move counted from the
    tensors: forward reads x, u (and weight, bias) and writes y (3 segments),
    mask, mean, rstd; backward reads dy, x, u, mask, mean, rstd and writes dx,
    du (the column partials add 2 D floats per block)."""
    import torch
    from generative_recommender_attention_gb300 import lmsd
    n, d = (int(v) for v in args.lmsd.split(","))
    g = torch.Generator(device="cpu").manual_seed(0)
    x = torch.randn(n, d, generator=g).to(torch.bfloat16).to(dev)
    u = torch.randn(n, d, generator=g).to(torch.bfloat16).to(dev)
    wt = torch.randn(d, generator=g).to(torch.bfloat16).to(dev)
    bs = torch.randn(d, generator=g).to(torch.bfloat16).to(dev)
    p = 0.1
    out = lmsd.hstu_lmsd_forward(x, u, wt, bs, dropout_ratio=p, seed=1)
    dy = torch.randn(out["y_tensor"].shape, generator=g).to(torch.bfloat16).to(dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def fwd():
        lmsd.hstu_lmsd_forward(x, u, wt, bs, dropout_ratio=p, seed=1)

    def bwd():
        lmsd.hstu_lmsd_backward(dy, x, u, wt, bs, out["mean_tensor"], out["rstd_tensor"],
                                out["mask_tensor"], dropout_ratio=p)

    def timed(fn):
        run, timed.note = replayable(fn)
        for _ in range(args.warmup):
            flush.zero_()
            run()
        ts = []
        for _ in range(args.steps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            run()
            e1.record()
            ts.append((e0, e1))
        torch.cuda.synchronize()
        return statistics.mean(a.elapsed_time(b) for a, b in ts)

    ms_f, ms_b = timed(fwd), timed(bwd)
    # DRAM bytes of one forward and one backward launch, from the committed
    # ncu summary of this size, if it was taken on the current kernel sources
    tfile = os.path.join(ROOT, "profiles", f"kernels_lmsd_{n}x{d}.md")
    traffic = {k: summary_traffic(tfile, k) for k in ("hstu_lmsd_fwd_kernel", "hstu_lmsd_bwd_kernel")}
    traffic = {k: v for k, v in traffic.items() if v is not None}
    bytes_f = n * d * 2 * 2 + n * 3 * d * 2 + n * d + n * 8
    bytes_b = n * 3 * d * 2 + n * d * 2 * 2 + n * d + n * 8 + n * d * 2 * 2
    pk = peaks()
    gf, gb = bytes_f / (ms_f * 1e-3) / 1e9, bytes_b / (ms_b * 1e-3) / 1e9
    print(json.dumps({
        "metric": "HSTU LMSD fwd and bwd HBM throughput (GB/s)",
        "value": (bytes_f + bytes_b) / ((ms_f + ms_b) * 1e-3) / 1e9, "unit": "GB/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_f + ms_b, "higher_is_better": True, "dtype": "bf16",
        "data": "synthetic",
        "fwd": {"ms": ms_f, "gbs": gf, "bytes": bytes_f},
        "bwd": {"ms": ms_b, "gbs": gb, "bytes": bytes_b},
        "roofline": {"bound": "hbm", "achieved": (bytes_f + bytes_b) / ((ms_f + ms_b) * 1e-3) / 1e9,
                     "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": (bytes_f + bytes_b) / ((ms_f + ms_b) * 1e-3) / 1e9 / pk["hbm_gbs"],
                     "traffic": (sum(traffic.values()) if len(traffic) == 2 else None),
                     "traffic_note": "ncu DRAM bytes of one forward plus one backward launch"},
        "config": {"workload": f"LMSD N={n} D={d}", "dropout_ratio": p, "apply_u_silu": True,
                   "concat_u": True, "concat_x": True,
                   "l2": "flushed between calls (256 MiB write)", "launch": timed.note},
    }))
    return 0


def run_paged(args, w, hstu, dev):
    """--paged: forward-only throughput over a paged K/V cache (the page's
    paged path is a causal forward), the contiguous forward timed beside it."""
    import torch
    from generative_recommender_attention_gb300 import workloads
    x = workloads.make_inputs(w, seed=0)
    lengths = x["lengths"]
    H, D = w.heads, w.head_dim
    ck = x["cu_seqlens_k"].tolist()
    n_pages = [-(-L // 128) for L in lengths]
    rng = np.random.default_rng(0)
    perm = rng.permutation(sum(n_pages))
    kv = torch.zeros(sum(n_pages), 2, 128, H, D, dtype=x["k"].dtype)
    ids, ptr, used = [], [0], 0
    for b, L in enumerate(lengths):
        for p in range(n_pages[b]):
            page = int(perm[used])
            used += 1
            ids.append(page)
            lo, hi = ck[b] + 128 * p, ck[b] + min(L, 128 * p + 128)
            kv[page, 0, :hi - lo] = x["k"][lo:hi]
            kv[page, 1, :hi - lo] = x["v"][lo:hi]
        ptr.append(len(ids))
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    kv, ids, ptr = kv.to(dev), torch.tensor(ids, dtype=torch.int32, device=dev), \
        torch.tensor(ptr, dtype=torch.int32, device=dev)
    mq, mk = x["max_seqlen_q"], x["max_seqlen_k"]
    o = torch.empty_like(d["q"])
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    flops = 4.0 * D * pairs(lengths, H, True)

    def paged():
        hstu.hstu_attn_fwd_paged(d["q"], kv, ids, ptr, d["cu_seqlens_q"], d["cu_seqlens_k"], mq,
                                 mk, scaling_seqlen=w.scaling_seqlen, alpha=w.alpha, out=o)

    def contiguous():
        hstu.hstu_attn_fwd(d["q"], d["k"], d["v"], d["cu_seqlens_q"], d["cu_seqlens_k"], mq, mk,
                           scaling_seqlen=w.scaling_seqlen, alpha=w.alpha, causal=True, out=o)

    def timed(fn):
        run, timed.note = replayable(fn)
        for _ in range(args.warmup):
            flush.zero_()
            run()
        ts = []
        for _ in range(args.steps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            run()
            e1.record()
            ts.append((e0, e1))
        torch.cuda.synchronize()
        return statistics.mean(a.elapsed_time(b) for a, b in ts)

    ms_p, ms_c = timed(paged), timed(contiguous)
    print(json.dumps({
        "metric": "HSTU paged-KV attn fwd TFLOP/s (causal, 128-row pages)",
        "value": flops / (ms_p * 1e-3) / 1e12, "unit": "TFLOP/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_p,
        "higher_is_better": True, "dtype": "bf16" if w.dtype == torch.bfloat16 else "f16",
        "data": "synthetic",
        "contiguous_fwd": {"value": flops / (ms_c * 1e-3) / 1e12, "ms_per_step": ms_c},
        "config": dict(workload_config(w, lengths), pages=int(kv.shape[0]),
                       page_order="shuffled", l2="flushed between steps (256 MiB write)",
                       launch=timed.note + ", CUDA events around each forward"),
    }))
    return 0


def run_reference(args, w):
    """--impl reference: the oracle, as it stands, on the host cores."""
    import torch
    from generative_recommender_attention_gb300 import workloads
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    x = workloads.make_inputs(w, seed=0)
    per_step = []
    flops_tot = 0.0
    n_seq = 0
    threads = 1
    for i in range(args.warmup + args.steps):
        f, s, n, threads = oracle_sample(x, w, 0.0, start=i % w.batch,  # one sequence per step
                                         mask=args.mask)
        if i >= args.warmup:
            per_step.append(s)
            flops_tot += f
            n_seq += n
    secs = sum(per_step)
    value = flops_tot / secs / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * secs / max(1, args.steps), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(w, x["lengths"], args.mask),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                             "sample": f"{n_seq} whole sequences (all heads, fwd+bwd), one per step"},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# ---------------------------------------------------------------- GPU arm
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--window", default=None,
                    help="token window 'left,right' (-1: no bound) instead of the workload's "
                         "causal / full mask")
    ap.add_argument("--no-flush", action="store_true", help="do not flush L2 between steps")
    ap.add_argument("--no-graph", action="store_true",
                    help="launch every step through the Python binding instead of replaying a "
                         "CUDA graph of it")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle timing")
    ap.add_argument("--func-targets", type=int, default=None,
                    help="arbitrary (func_tensor) mask: causal plus the last N keys of every "
                         "sequence as targets")
    ap.add_argument("--lmsd", default=None,
                    help="time the LMSD forward and backward on an 'N,D' bf16 problem (dropout "
                         "0.1, SiLU, both extra segments); one JSON line in GB/s")
    ap.add_argument("--paged", action="store_true",
                    help="time the causal forward over a paged K/V cache (the workload's keys "
                         "in shuffled 128-row pages) beside the contiguous forward; one JSON line")
    ap.add_argument("--head-dim", type=int, default=None,
                    help="run the workload with another head dimension (32, 64, 128 or 256), "
                         "alpha = 1/sqrt(D); the name gets a _d<D> suffix")
    ap.add_argument("--batch", type=int, default=None,
                    help="draw only this many sequences of the workload (same length "
                         "distribution; the name gets a _b<B> suffix): smaller captures for ncu")
    ap.add_argument("--plan", action="store_true",
                    help="one hstu_attn_plan launch per step shared by the planned forward and "
                         "backward, instead of hstu_attn_fwd + hstu_attn_bwd scheduling each call")
    ap.add_argument("--kernels-only", action="store_true",
                    help="run warm-up and timed steps only (no second pass, end-to-end, clocks or "
                         "CPU baseline) and print no JSON line: for wrapping in a profiler")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    args.mask = None
    if args.window:
        left, right = (int(v) for v in args.window.split(","))
        args.mask = (left, right)
    if args.func_targets is not None:
        args.mask = ("targets", int(args.func_targets))

    import torch
    from generative_recommender_attention_gb300 import workloads
    w = workloads.WORKLOADS[args.workload]
    if args.head_dim is not None and args.head_dim != w.head_dim:
        import dataclasses as _dc
        w = _dc.replace(w, name=f"{w.name}_d{args.head_dim}", head_dim=args.head_dim,
                        alpha=1.0 / math.sqrt(args.head_dim))
    if args.batch is not None and args.batch != w.batch:
        import dataclasses as _dc
        w = _dc.replace(w, name=f"{w.name}_b{args.batch}", batch=args.batch)
    if args.impl == "reference":
        return run_reference(args, w)

    import __graft_entry__
    __graft_entry__.build()
    import generative_recommender_attention_gb300 as hstu

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if args.paged:
        return run_paged(args, w, hstu, dev)
    if args.lmsd:
        return run_lmsd(args, dev)

    x = workloads.make_inputs(w, seed=0)
    lengths = x["lengths"]
    B, T, H, D = w.batch, sum(lengths), w.heads, w.head_dim
    mask = w.causal if args.mask is None else args.mask
    N = pairs(lengths, H, mask)
    flops_step = 14.0 * D * N
    bytes_step = 11.0 * T * H * D * 2  # fwd 4 T H D and bwd 7 T H D elements of 2 bytes
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    o = torch.empty_like(d["q"])
    dq, dk, dv = torch.empty_like(d["q"]), torch.empty_like(d["k"]), torch.empty_like(d["v"])
    mq, mk = x["max_seqlen_q"], x["max_seqlen_k"]
    wsz = hstu.workspace_size_func if (args.mask and args.mask[0] == "targets") \
        else hstu.workspace_size
    ws_f = torch.empty(wsz(B, T, T, H, D, mq, mk, False), dtype=torch.uint8, device=dev)
    ws_b = torch.empty(wsz(B, T, T, H, D, mq, mk, True), dtype=torch.uint8, device=dev)
    kw = dict(scaling_seqlen=w.scaling_seqlen, alpha=w.alpha)
    if args.mask is None:
        kw["causal"] = w.causal
    elif args.mask[0] == "targets":
        i = np.concatenate([np.arange(L) for L in lengths])
        lk = np.concatenate([np.full(L, L) for L in lengths])
        kw["func"] = torch.from_numpy(
            np.stack([i + 1, lk - args.mask[1], lk]).astype(np.int32))[None].contiguous().to(dev)
    else:
        kw["window_size"] = args.mask
    flush = None if args.no_flush else torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    func_mode = "func" in kw
    # One plan per step (the scheduling launch shared by the forward and the
    # backward); the arbitrary-mask calls are not planned.
    use_plan = args.plan and not func_mode
    ws_p = torch.empty(hstu.plan_workspace_size(B, T, T, H, D, mq, mk), dtype=torch.uint8,
                       device=dev) if use_plan else None
    win_kw = {k: kw[k] for k in ("causal", "window_size") if k in kw}

    def planned_step(g, o_, dq_, dk_, dv_):
        p = hstu.hstu_attn_plan(g["cu_seqlens_q"], g["cu_seqlens_k"], T, T, H, D, mq, mk,
                                workspace=ws_p, **win_kw)
        hstu.hstu_attn_fwd(g["q"], g["k"], g["v"], g["cu_seqlens_q"], g["cu_seqlens_k"], mq, mk,
                           out=o_, plan=p, **kw)
        hstu.hstu_attn_bwd(g["do"], g["q"], g["k"], g["v"], g["cu_seqlens_q"], g["cu_seqlens_k"],
                           mq, mk, dq=dq_, dk=dk_, dv=dv_, plan=p, **kw)

    status_ws = [ws_p] if use_plan else [ws_f, ws_b]

    def step(evs=None):
        if evs is None and use_plan:
            planned_step(d, o, dq, dk, dv)
            return
        if evs is not None and func_mode:
            # the arbitrary-mask calls have no profiled variant: events go
            # around whole calls (the second event of each call is its start)
            evs[0].record(); evs[1].record()
            hstu.hstu_attn_fwd(d["q"], d["k"], d["v"], d["cu_seqlens_q"], d["cu_seqlens_k"], mq,
                               mk, out=o, workspace=ws_f, **kw)
            evs[2].record(); evs[3].record(); evs[4].record()
            hstu.hstu_attn_bwd(d["do"], d["q"], d["k"], d["v"], d["cu_seqlens_q"],
                               d["cu_seqlens_k"], mq, mk, dq=dq, dk=dk, dv=dv, workspace=ws_b,
                               **kw)
            evs[5].record(); evs[6].record()
            return
        hstu.hstu_attn_fwd(d["q"], d["k"], d["v"], d["cu_seqlens_q"], d["cu_seqlens_k"], mq, mk,
                           out=o, workspace=ws_f, events=None if evs is None else evs[0:3], **kw)
        hstu.hstu_attn_bwd(d["do"], d["q"], d["k"], d["v"], d["cu_seqlens_q"], d["cu_seqlens_k"],
                           mq, mk, dq=dq, dk=dk, dv=dv, workspace=ws_b,
                           events=None if evs is None else evs[3:7], **kw)

    # Timed region: whole steps between two events each; no events between the
    # kernels, so each grid may launch while its predecessor drains.
    e_beg = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    e_end = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    for i in range(args.warmup):
        if flush is not None:
            flush.zero_()
        step()
    torch.cuda.synchronize()
    # The step (both library calls, five kernels chained by programmatic
    # dependent launch) is captured once in a CUDA graph and replayed, so the
    # host's per-call work (argument checks, tensor-map encoding, launches)
    # is not in the device's critical path; the replayed kernels and their
    # arguments are exactly those of the direct calls.
    run, graph_note = step, "direct calls (no graph)"
    if not args.no_graph:
        try:
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side):
                step()
            torch.cuda.current_stream().wait_stream(side)
            torch.cuda.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                step()
            torch.cuda.synchronize()
            run, graph_note = graph.replay, "CUDA graph of one fwd+bwd step, replayed"
            for i in range(args.warmup):
                if flush is not None:
                    flush.zero_()
                run()
            torch.cuda.synchronize()
        except Exception as exc:  # capture unsupported: time the direct calls
            run, graph_note = step, f"direct calls (graph capture failed: {type(exc).__name__})"
            torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    if args.kernels_only:
        for i in range(args.steps):
            if flush is not None:
                flush.zero_()
            run()
        torch.cuda.synchronize()
        assert all(hstu.last_device_status(ws) == 0 for ws in status_ws)
        return 0
    # SM clocks sampled through NVML while the timed steps run (nvidia-smi
    # when NVML cannot be loaded; its raw samples go to $HSTU_CLOCKS_DIR)
    clocks = start_clock_sampler(local, rank)
    wall0 = time.perf_counter()
    for i in range(args.steps):
        if flush is not None:
            flush.zero_()
        e_beg[i].record()
        run()
        e_end[i].record()
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    if dist is not None:
        dist.barrier()
    clk = clocks.stop()
    if clk is None and getattr(clocks, "nvml_error", None):
        clk = {"error": "no samples; NVML: " + clocks.nvml_error}
    assert all(hstu.last_device_status(ws) == 0 for ws in status_ws)
    t_step = [b.elapsed_time(e) for b, e in zip(e_beg, e_end)]

    # Per-kernel pass: events between the kernels (one launch each, in
    # sequence), for the roofline of the dominant kernel.
    n_prof = max(3, min(args.steps, 200))
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(7)] for _ in range(n_prof + 1)]
    for row in ev:
        for e in row:
            e.record()   # creates the events before they are handed to the library
    torch.cuda.synchronize()
    for row in ev:
        if flush is not None:
            flush.zero_()
        step(row)
    torch.cuda.synchronize()
    timed = ev[1:]
    # Informational: the same steps back to back without the L2 flush (as in
    # consecutive training steps); not the headline value.
    n_warm = max(3, min(args.steps, 200))
    w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    run()
    w0.record()
    for _ in range(n_warm):
        run()
    w1.record()
    torch.cuda.synchronize()
    ms_warm = w0.elapsed_time(w1) / n_warm
    t_plan = []
    if use_plan:  # the plan launch alone, as it runs at the head of each planned step
        for _ in range(n_prof):
            if flush is not None:
                flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            hstu.hstu_attn_plan(d["cu_seqlens_q"], d["cu_seqlens_k"], T, T, H, D, mq, mk,
                                workspace=ws_p, **win_kw)
            e1.record()
            t_plan.append((e0, e1))
        torch.cuda.synchronize()
        t_plan = [a.elapsed_time(b) for a, b in t_plan]
    t_sched_f = [r[0].elapsed_time(r[1]) for r in timed]
    t_fwd = [r[1].elapsed_time(r[2]) for r in timed]
    t_sched_b = [r[3].elapsed_time(r[4]) for r in timed]
    # one backward launch (dK/dV units, then dQ units) between marks 4 and 5;
    # marks 5 and 6 are recorded back to back
    t_bwd = [r[4].elapsed_time(r[6]) for r in timed]
    ms_step, value = replica_throughput(sum(t_step), args.steps, flops_step, world, dist, dev)
    pk = peaks()

    # per-kernel live timings and algorithmic FLOPs per launch
    mean = lambda a: sum(a) / len(a)  # noqa: E731
    kernels = {
        "hstu_fwd_kernel": (4.0 * D * N, mean(t_fwd)),
        "hstu_bwd_kernel": (10.0 * D * N, mean(t_bwd)),
    }
    if func_mode:  # whole calls (see step)
        kernels = {"hstu_attn_fwd (whole call)": (4.0 * D * N, mean(t_fwd)),
                   "hstu_attn_bwd (whole call)": (10.0 * D * N, mean(t_bwd))}
    dom = max(kernels, key=lambda k: kernels[k][1])
    f_dom, ms_dom = kernels[dom]
    achieved = f_dom / (ms_dom * 1e-3) / 1e12
    # DRAM bytes of one launch of the dominant kernel, from the committed ncu
    # summary of this workload, if it was taken on the current kernel sources
    traffic = None
    if args.mask is None:  # the summary covers the default mask
        traffic = summary_traffic(os.path.join(ROOT, "profiles", f"kernels_{w.name}_full.md"), dom)

    # End to end through the public API: every step copies its inputs in from
    # pinned host memory and its results (O, dQ, dK, dV) back out.  Copy-in,
    # compute and copy-out run on three streams with two buffer sets, so step
    # i's compute overlaps step i+1's copy-in and step i-1's copy-out; the
    # timed region spans the first copy-in to the last copy-out.
    names = ("q", "k", "v", "do", "cu_seqlens_q", "cu_seqlens_k")
    pin = {k: x[k].pin_memory() for k in names}
    h2d = sum(t.numel() * t.element_size() for t in pin.values())
    dev_in = [{k: torch.empty_like(d[k]) for k in names} for _ in range(2)]
    dev_out = [[torch.empty_like(d["q"]), torch.empty_like(d["q"]), torch.empty_like(d["k"]),
                torch.empty_like(d["v"])] for _ in range(2)]
    host_out = [[torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in dev_out[0]]
                for _ in range(2)]
    d2h = sum(t.numel() * t.element_size() for t in host_out[0])
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    s_comp = torch.cuda.current_stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    n_e2e = max(3, min(args.steps, 50))

    def e2e_run(n):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(s_in)
        for i in range(n):
            b = i % 2
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_comp[b])  # step i-2 has finished reading this set
                for k in names:
                    dev_in[b][k].copy_(pin[k], non_blocking=True)
                ev_in[b].record(s_in)
            s_comp.wait_event(ev_in[b])
            if i >= 2:
                s_comp.wait_event(ev_out[b])  # step i-2's results have left this set
            g = dev_in[b]
            o_, dq_, dk_, dv_ = dev_out[b]
            if use_plan:
                planned_step(g, o_, dq_, dk_, dv_)
            else:
                hstu.hstu_attn_fwd(g["q"], g["k"], g["v"], g["cu_seqlens_q"], g["cu_seqlens_k"],
                                   mq, mk, out=o_, workspace=ws_f, **kw)
                hstu.hstu_attn_bwd(g["do"], g["q"], g["k"], g["v"], g["cu_seqlens_q"],
                                   g["cu_seqlens_k"], mq, mk, dq=dq_, dk=dk_, dv=dv_,
                                   workspace=ws_b, **kw)
            ev_comp[b].record(s_comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_comp[b])
                for src, dst in zip(dev_out[b], host_out[b]):
                    dst.copy_(src, non_blocking=True)
                ev_out[b].record(s_out)
        e1.record(s_out)  # the last copy-out follows every earlier copy and compute
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n

    e2e_run(3)  # warm-up
    e2e_ms_step = e2e_run(n_e2e)
    e2e_ms_step, e2e_value = replica_throughput(e2e_ms_step * n_e2e, n_e2e, flops_step, world,
                                                dist, dev)

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "pct_of_dense_bf16_peak": 100.0 * value / world / pk["bf16_tflops"],
        "pct_of_sustained_bf16_peak": 100.0 * value / world / pk["bf16_tflops_sustained"],
        "ms_per_step_median": statistics.median(t_step),
        "achieved_gbs": world * bytes_step / (ms_step * 1e-3) / 1e9,
        "achieved_gbs_note": "algorithmic bytes (fwd reads q,k,v and writes o; bwd reads q,k,v,dO and "
                             "writes dq,dk,dv) per step time, against %.1f GB/s measured HBM" % pk["hbm_gbs"],
        "value_l2_warm": world * flops_step / (ms_warm * 1e-3) / 1e12,
        "ms_per_step_l2_warm": ms_warm,
        "config": dict(workload_config(w, lengths, args.mask),
                       l2="flushed between steps (256 MiB write)" if flush is not None else "not flushed",
                       launch=graph_note,
                       schedule=("one hstu_attn_plan launch per step, shared by the planned "
                                 "forward and backward" if use_plan else
                                 "each call schedules its own work"),
                       parallelism="replicas" if world > 1 else "single GPU",
                       flops_per_step=flops_step, peaks_source=pk["source"]),
        "per_kernel_ms": {"plan": mean(t_plan) if t_plan else None,
                          "sched_fwd": mean(t_sched_f), "fwd": mean(t_fwd),
                          "sched_bwd": mean(t_sched_b), "bwd": mean(t_bwd),
                          "sum": mean([a + b + c + e for a, b, c, e in
                                       zip(t_sched_f, t_fwd, t_sched_b, t_bwd)]),
                          "steps": len(timed),
                          "note": "second pass with events between kernels (no launch overlap), "
                                  "each call scheduling its own work"},
        "roofline": {"kernel": dom, "bound": "tensor", "achieved": achieved,
                     "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": achieved / pk["bf16_tflops"], "traffic": traffic,
                     "peak_kind": "bf16 burst, of measured (the kernel's launches are timed "
                                  "one by one between events, %d of them)" % len(timed),
                     "frac_of_sustained": achieved / pk["bf16_tflops_sustained"]},
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": n_e2e, "ms_per_step": e2e_ms_step,
                "note": "copy-in, compute and copy-out of consecutive steps overlap on three "
                        "streams; L2 not flushed (each step's inputs arrive fresh from the host)"},
        "gpu_launches": (3 if use_plan else 6 if func_mode else 4) * args.steps,
        "clocks": clk,
        "wall_s_timed_loop": wall,
    }

    if rank == 0:
        f, s, n, threads = oracle_sample(x, w, args.cpu_budget, mask=args.mask)
        line["cpu_baseline"] = {"value": f / s / 1e12, "unit": "TFLOP/s", "cores": threads,
                                "kind": "oracle",
                                "sample": f"first {n} of {B} sequences, all heads, fwd+bwd (fp64)"}
        f1, s1, n1, _ = oracle_sample(x, w, min(2.0, args.cpu_budget), threads=1, mask=args.mask)
        line["cpu_baseline_one_core"] = {"value": f1 / s1 / 1e12, "unit": "TFLOP/s", "cores": 1,
                                         "sample": f"first {n1} sequences, all heads, fwd+bwd (fp64)"}
        print(json.dumps(line))
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
