#!/usr/bin/env python3
"""Benchmark of the block-scaled cast path on one GB300 (or N replicas).

Headline (value, ms_per_step, kernels, roofline): one step = every cast of
the path over one batch of the MoE-dispatch activations workload (BF16
16384 x 7168, N(0,1) rows times a per-row log-normal(0,1) magnitude, seed 0;
the tokens are split over 32 experts with Zipf(1.1) counts for the
transposed ragged conversion):

  1. mxfp4_quantize_rows   BF16 -> MXFP4 (packed E2M1 + UE8M0)
  2. fp4_to_fp8_rows       MXFP4 -> E4M3, 128-element blocks, k = 0
  3. fp4_to_fp8_cols       MXFP4 -> E4M3 transposed, 32 ragged expert groups
  4. nvfp4_amax            per-tensor amax
  5. nvfp4_quantize        NVFP4 1x16, stochastic rounding (seed = pass)
  6. nvfp4_quantize_2d     NVFP4 16x16 on the same tensor

The metric is effective bandwidth: algorithmic bytes read + written by the
kernels over their device time (CUDA events on the launching stream), as GB/s
and as a fraction of the measured HBM copy bandwidth.  The timed region is
--steps K steps, each step's pass repeated R times (R sized so that the
region lasts about a second and a half, so that the clock sampler sees it);
L2 is flushed (256 MB written, then read back) before every pass, outside
the events, which sit at the two ends of every pass.

`configs`: every configuration of the workload definition -- the 256 x 512
outlier tensor, the MoE-dispatch tensor, the 65536 x 2048 ragged experts, the
NVFP4 activations (16384 x 14336 Student-t(4)) and weights (14336 x 4096
N(0, 0.02)), the 1K-262144 row bandwidth sweep at 7168, a hidden size
that is a multiple of 128 but not of 512 (the transposed conversion's
exponent rows by four-row groups), and the same with a token count that is
not a multiple of 16 -- each call timed inside its configuration's chain (an
event between every two calls) and alone (L2 flushed before the call).

`error_stats`: the oracle's numbers about the formats on each
configuration's input (dequantization error per block; exact, rounded and
flushed elements of the FP4 -> FP8 conversion at k = 0 and 6).

--impl reference times the CPU oracle (the plain C implementation the tests
compare against) on a bounded sample of the headline workload.
"""
from __future__ import annotations

import argparse
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
sys.path.insert(0, ROOT)

METRIC = "effective GB/s (bytes read+written) per quantize/convert kernel; % of HBM peak"
M_ROWS, K_COLS, EXPERTS = 16384, 7168, 32
WORKLOAD = ("moe_dispatch bf16 16384x7168 (N(0,1) x row lognormal(0,1), seed 0), "
            "32 experts Zipf(1.1): mxfp4_quantize_rows -> fp4_to_fp8_rows(k=0) -> "
            "fp4_to_fp8_cols(ragged) ; nvfp4_amax -> nvfp4_quantize(SR) ; nvfp4_quantize_2d")
KERNELS = ["mxfp4_quantize_rows", "fp4_to_fp8_rows", "fp4_to_fp8_cols", "nvfp4_amax",
           "nvfp4_quantize", "nvfp4_quantize_2d"]
# source file of each entry point's kernels (for the ncu traffic record's
# staleness check)
KERNEL_SRC = {
    "mxfp4_quantize_rows": "fq_mxfp4.cu", "fp4_to_fp8_rows": "fq_mxfp4.cu",
    "fp4_to_fp8_cols": "fq_cols.cu", "nvfp4_amax": "fq_nvfp4.cu",
    "nvfp4_quantize": "fq_nvfp4.cu", "nvfp4_quantize_2d": "fq_nvfp4.cu",
    "bf16_to_mxfp4_fp8": "fq_fused.cu", "bf16_to_mxfp4_fp8_single_pass": "fq_fused.cu",
    "nvfp4_amax_rht": "fq_nvfp4.cu",
    "nvfp4_quantize_rht": "fq_nvfp4.cu", "nvfp4_quantize_rht_rne": "fq_nvfp4.cu",
    "fp8_quantize_1x128": "fq_fp8.cu",
    "fp8_quantize_128x128": "fq_fp8.cu", "mxfp4_dequantize_rows": "fq_fp8.cu",
    "nvfp4_quantize_delayed": "fq_nvfp4.cu", "nvfp4_quantize_2d_t": "fq_nvfp4.cu",
    "mxfp4_scales_mma_layout": "fq_mxfp4.cu",
}
FALLBACK_HBM_GBS = 6800.0
TIMED_REGION_S = 1.5
SWEEP_ROWS = [1024 << i for i in range(9)]
TWO_LAUNCH_K = 7040   # a multiple of 128, not of 512


# ------------------------------------------------------------------ algorithmic bytes

def b_mxfp4(M, K):
    E = M * K
    return 2 * E + E // 2 + E // 32


def b_rows(M, K):
    E = M * K
    return E // 2 + E // 32 + E + 4 * (E // 128)


def b_cols(M, K, nb, G):
    E = M * K
    return E // 2 + E // 32 + E + 4 * K * nb + 8 * (G + 1)


def b_amax(M, K):
    return 2 * M * K + 4


def b_nvfp4(M, K):
    E = M * K
    return 2 * E + E // 2 + E // 16 + 8


def b_2d(M, K):
    E = M * K
    return 2 * E + E // 2 + E // 256 + 8


def b_2d_t(M, K):
    E = M * K
    return 2 * E + E + 2 * (E // 256) + 8


def b_fused(M, K, nb, G):
    E = M * K
    return 2 * E + E // 2 + E // 32 + E + 4 * (E // 128) + E + 4 * K * nb + 8 * (G + 1)


def algorithmic_bytes(M: int, K: int, nblocks_cols: int, G: int) -> dict:
    """Bytes each kernel of the headline step must read + write."""
    return {"mxfp4_quantize_rows": b_mxfp4(M, K), "fp4_to_fp8_rows": b_rows(M, K),
            "fp4_to_fp8_cols": b_cols(M, K, nblocks_cols, G), "nvfp4_amax": b_amax(M, K),
            "nvfp4_quantize": b_nvfp4(M, K), "nvfp4_quantize_2d": b_2d(M, K)}


def col_blocks(offs) -> int:
    import numpy as np
    return int(((np.diff(np.asarray(offs)) + 127) // 128).sum())


def hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def file_sha(name: str) -> str:
    """sha256[:16] of a kernel's source file followed by the headers it uses."""
    h = hashlib.sha256()
    parts = [name, "fq_common.cuh"]
    if name in ("fq_cols.cu", "fq_fused.cu"):
        parts.append("fq_cols_common.cuh")
    for part in parts:
        with open(os.path.join(ROOT, "fp8_quantization_gb300", "csrc", part), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, or None if the
    kernel's source changed since it was captured."""
    p = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        for line in f:
            parts = line.split("#", 1)[0].split()
            if len(parts) >= 3 and parts[0] == kernel:
                if parts[2] != file_sha(KERNEL_SRC[kernel]):
                    return None
                return float(parts[1])
    return None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", str(self.gpu)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self, t0: float, t1: float):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.t.join(timeout=2)
        rows = [l for (ts, l) in self.lines if t0 - 0.06 <= ts <= t1 + 0.06]
        window = "timed"
        if not rows:
            rows = [l for _, l in self.lines]
            window = "around timed region (none inside)"
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            f = [x.strip() for x in r.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
                power.append(float(f[3]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "sm_mhz_min": min(sm) if sm else None,
                "power_w_max": max(power) if power else None,
                "reasons": sorted(reasons), "samples": len(sm), "window": window}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(value: float, backend_device=None) -> float:
    """Max of a float over all ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=backend_device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ CPU oracle

def oracle_sample_pass(bits, offs_rows, K):
    """One pass of every cast through the CPU oracle on a row sample; returns
    (seconds, algorithmic bytes)."""
    import oracle
    M = bits.shape[0]
    G = offs_rows.size - 1
    t0 = time.perf_counter()
    q, s = oracle.mxfp4_quantize_rows(bits)
    oracle.fp4_to_fp8_rows(q, s, 0)
    oracle.fp4_to_fp8_cols(q, s, offs_rows, 0)
    A = oracle.nvfp4_amax(bits)
    oracle.nvfp4_quantize(bits, A, use_sr=True, seed=1)
    oracle.nvfp4_quantize_2d(bits, A)
    dt = time.perf_counter() - t0
    return dt, sum(algorithmic_bytes(M, K, col_blocks(offs_rows), G).values())


def oracle_sample_inputs(rows: int):
    from fp8_quantization_gb300 import workloads
    bits = workloads.moe_dispatch(rows, K_COLS, seed=0)
    offs = workloads.zipf_group_offsets(rows, EXPERTS, 1.1, 0)
    return bits, offs


def cpu_baseline(target_s: float = 12.0) -> dict:
    import oracle
    rows = 64
    bits, offs = oracle_sample_inputs(rows)
    dt, nbytes = oracle_sample_pass(bits, offs, K_COLS)
    rows = int(min(M_ROWS, max(16, rows * target_s / max(dt, 1e-3))))
    rows = max(16, rows // 16 * 16)
    bits, offs = oracle_sample_inputs(rows)
    dt, nbytes = oracle_sample_pass(bits, offs, K_COLS)
    cores = oracle.num_threads()
    # the same pass on one core, over a smaller sample (about a third of the time)
    rows1 = max(16, int(rows * (target_s / 3) / max(dt * cores, 1e-3)) // 16 * 16)
    b1, o1 = oracle_sample_inputs(rows1)
    oracle.set_num_threads(1)
    try:
        dt1, nbytes1 = oracle_sample_pass(b1, o1, K_COLS)
    finally:
        oracle.set_num_threads(cores)
    return {"value": round(nbytes / dt / 1e9, 4), "unit": "GB/s", "cores": cores,
            "kind": "oracle",
            "sample": f"first {rows} of {M_ROWS} rows of the workload (same recipe), all six casts "
                      f"once, {dt:.1f} s",
            "one_core": {"value": round(nbytes1 / dt1 / 1e9, 4), "unit": "GB/s",
                         "sample": f"first {rows1} rows, {dt1:.1f} s"}}


def _r(d: dict, nd: int = 6) -> dict:
    return {k: (round(v, nd) if isinstance(v, float) else v) for k, v in d.items()}


def oracle_error_stats(host: dict) -> dict:
    """The oracle's dequantization error per block and FP4 -> FP8 exactness
    counts on every configuration's input (host BF16 bits)."""
    import oracle
    out = {}
    t0 = time.perf_counter()

    def mx_chain(bits, offs=None, rows=True):
        q, s = oracle.mxfp4_quantize_rows(bits)
        st = {"mxfp4 max|x-xhat|/amax_blk": _r(oracle.mxfp4_error_stats(bits, q, s))}
        for k in (0, 6):
            if rows:
                st[f"fp4_to_fp8_rows k={k}"] = oracle.fp4_to_fp8_counts(q, s, k)
            if offs is not None:
                st[f"fp4_to_fp8_cols k={k}"] = oracle.fp4_to_fp8_counts(q, s, k, offs)
        return st

    out["pr1 256x512"] = mx_chain(host["pr1"])
    x, offs = host["moe_dispatch"]
    st = mx_chain(x, offs)
    A = oracle.nvfp4_amax(x)
    q, sb, g = oracle.nvfp4_quantize(x, A, use_sr=True, seed=1000)
    st["nvfp4 1x16 SR (seed 1000) max|x-xhat|/amax_blk"] = _r(oracle.nvfp4_error_stats(x, q, sb, g))
    q, sb, g = oracle.nvfp4_quantize_2d(x, A)
    st["nvfp4 16x16 max|x-xhat|/amax_blk"] = _r(oracle.nvfp4_error_stats(x, q, sb, g, 16))
    out["moe_dispatch 16384x7168"] = st
    x, offs = host["ragged_experts"]
    out["ragged_experts 65536x2048"] = mx_chain(x, offs, rows=False)
    x = host["nvfp4_act"]
    A = oracle.nvfp4_amax(x)
    st = {}
    for sr in (False, True):
        q, sb, g = oracle.nvfp4_quantize(x, A, use_sr=sr, seed=1234)
        st[f"nvfp4 1x16 {'SR (seed 1234)' if sr else 'RNE'} max|x-xhat|/amax_blk"] = \
            _r(oracle.nvfp4_error_stats(x, q, sb, g))
    out["nvfp4 activations 16384x14336"] = st
    w = host["nvfp4_weight"]
    q, sb, g = oracle.nvfp4_quantize_2d(w, oracle.nvfp4_amax(w))
    out["nvfp4 weights 14336x4096"] = {
        "nvfp4 16x16 max|x-xhat|/amax_blk": _r(oracle.nvfp4_error_stats(w, q, sb, g, 16))}
    xs = host["sweep_sample"]
    import numpy as np
    out[f"sweep Student-t(3) x 7168, first {xs.shape[0]} rows (every size is a prefix)"] = \
        mx_chain(xs, np.array([0, xs.shape[0]], dtype=np.int64))
    out["seconds"] = round(time.perf_counter() - t0, 1)
    return out


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    # size the per-step sample so that warmup + steps take about two minutes
    probe_rows = 64
    bits, offs = oracle_sample_inputs(probe_rows)
    dt, _ = oracle_sample_pass(bits, offs, K_COLS)
    per_step = 120.0 / max(1, args.steps + args.warmup)
    rows = int(min(M_ROWS, max(16, probe_rows * per_step / max(dt, 1e-3))))
    rows = max(16, rows // 16 * 16)
    bits, offs = oracle_sample_inputs(rows)
    for _ in range(args.warmup):
        oracle_sample_pass(bits, offs, K_COLS)
    tot_t, tot_b = 0.0, 0
    for _ in range(args.steps):
        dt, nb = oracle_sample_pass(bits, offs, K_COLS)
        tot_t += dt
        tot_b += nb
    value = tot_b / tot_t / 1e9
    sample = f"first {rows} of {M_ROWS} rows of the workload per step, all six casts"
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(tot_t / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "M": M_ROWS, "K": K_COLS, "experts": EXPERTS,
                   "sample_rows": rows},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ GPU timing helpers

class Timer:
    """CUDA-event timing on one stream, with an L2 flush (a 256 MB buffer
    written, then read back, so that its dirty lines are written out before
    the timed work) ahead of every timed call or pass, outside the events."""

    def __init__(self, dev, warmup):
        import torch
        self.torch = torch
        self.dev = dev
        self.warmup = warmup
        self.stream = torch.cuda.current_stream(dev)
        self.flush_buf = torch.empty((256 << 20,), dtype=torch.uint8, device=dev)

    def flush(self):
        self.flush_buf.fill_(1)
        self.flush_buf.sum(dtype=self.torch.int64)

    def event(self):
        return self.torch.cuda.Event(enable_timing=True)

    def alone_us(self, fn, reps):
        """Mean device time of fn() with L2 flushed before every call."""
        for _ in range(self.warmup):
            self.flush()
            fn()
        ev = [(self.event(), self.event()) for _ in range(reps)]
        for a, b in ev:
            self.flush()
            a.record(self.stream)
            fn()
            b.record(self.stream)
        self.torch.cuda.synchronize(self.dev)
        return sum(a.elapsed_time(b) for a, b in ev) / reps * 1e3

    def chain_us(self, fns, reps):
        """Per-call device times inside the chain (an event between every two
        calls) and the chain's time with events at its two ends only."""
        n = len(fns)
        for _ in range(self.warmup):
            self.flush()
            for fn in fns:
                fn()
        ev = [[self.event() for _ in range(n + 1)] for _ in range(reps)]
        for e in ev:
            self.flush()
            for j, fn in enumerate(fns):
                e[j].record(self.stream)
                fn()
            e[n].record(self.stream)
        ends = [(self.event(), self.event()) for _ in range(reps)]
        for a, b in ends:
            self.flush()
            a.record(self.stream)
            for fn in fns:
                fn()
            b.record(self.stream)
        self.torch.cuda.synchronize(self.dev)
        per = [sum(e[j].elapsed_time(e[j + 1]) for e in ev) / reps * 1e3 for j in range(n)]
        total = sum(a.elapsed_time(b) for a, b in ends) / reps * 1e3
        return per, total


def link_rates(dev, nbytes=256 << 20, reps=5):
    """Pinned host <-> device copy rates (GB/s): each direction alone and both
    directions at once on two streams."""
    import torch
    h_in = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    h_out = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    d_in = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    d_out = torch.ones(nbytes, dtype=torch.uint8, device=dev)
    s1, s2 = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def one(stream, fn):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            fn()
            a.record(stream)
            for _ in range(reps):
                fn()
            b.record(stream)
        torch.cuda.synchronize(dev)
        return nbytes * reps / (a.elapsed_time(b) * 1e-3) / 1e9

    h2d = one(s1, lambda: d_in.copy_(h_in, non_blocking=True))
    d2h = one(s2, lambda: h_out.copy_(d_out, non_blocking=True))
    torch.cuda.synchronize(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(s1)
    s2.wait_event(a)
    with torch.cuda.stream(s1):
        for _ in range(reps):
            d_in.copy_(h_in, non_blocking=True)
    with torch.cuda.stream(s2):
        for _ in range(reps):
            h_out.copy_(d_out, non_blocking=True)
    e2 = torch.cuda.Event()
    e2.record(s2)
    s1.wait_event(e2)
    b.record(s1)
    torch.cuda.synchronize(dev)
    both = 2 * nbytes * reps / (a.elapsed_time(b) * 1e-3) / 1e9
    return {"h2d": round(h2d, 1), "d2h": round(d2h, 1), "both_directions_total": round(both, 1),
            "copy_bytes": nbytes}


# ------------------------------------------------------------------ GPU arm

def run_gpu(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    import fp8_quantization_gb300 as fq
    from fp8_quantization_gb300 import workloads

    ws, rank, local = dist_env()
    if ws > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if ws > 1 else 0)
    torch.cuda.set_device(dev)
    fq.abi()  # fail loudly if the library is missing
    peak, peak_kind = hbm_peak()
    l2_bytes = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 126 << 20))
    T = Timer(dev, args.warmup)
    stream = T.stream
    u8 = dict(dtype=torch.uint8, device=dev)
    f32 = dict(dtype=torch.float32, device=dev)
    wall0 = time.time()

    def to_dev(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(
            torch.bfloat16)

    def frac(nbytes, us):
        gbs = nbytes / (us * 1e-6) / 1e9
        return round(gbs, 1), round(gbs / peak, 4)

    # ---------------------------------------------------------------- headline
    M, K, G = M_ROWS, K_COLS, EXPERTS
    bits = workloads.moe_dispatch(M, K, seed=0)
    offs_np = workloads.zipf_group_offsets(M, G, 1.1, 0)
    nb_cols = col_blocks(offs_np)
    nbytes = algorithmic_bytes(M, K, nb_cols, G)
    launches_per_pass = (1 + 1 + fq.fp4_to_fp8_cols_launch_count(K) + 2 + 1 + 1)
    step_bytes = sum(nbytes.values())
    x = to_dev(bits)
    offs = torch.from_numpy(offs_np).to(dev)
    cap = fq.fp4_to_fp8_cols_scale_capacity(M, G)
    out = {
        "q": torch.empty((M, K // 2), **u8), "s": torch.empty((M, K // 32), **u8),
        "y": torch.empty((M, K), **u8), "ys": torch.empty((M, K // 128), **f32),
        "yT": torch.empty((K, M), **u8), "yTs": torch.empty((cap, K), **f32),
        "amax": torch.empty((1,), **f32),
        "q4": torch.empty((M, K // 2), **u8), "sb4": torch.empty((M, K // 16), **u8),
        "g4": torch.empty((1,), **f32),
        "q2": torch.empty((M, K // 2), **u8), "sb2": torch.empty((M // 16, K // 16), **u8),
        "g2": torch.empty((1,), **f32),
    }

    def step_calls(i, xin, o=None, offs_d=None):
        o = out if o is None else o
        offs_d = offs if offs_d is None else offs_d
        return [
            lambda: fq.mxfp4_quantize_rows(xin, o["q"], o["s"]),
            lambda: fq.fp4_to_fp8_rows(o["q"], o["s"], 0, o["y"], o["ys"]),
            lambda: fq.fp4_to_fp8_cols(o["q"], o["s"], offs_d, 0, o["yT"], o["yTs"]),
            lambda: fq.nvfp4_amax(xin, o["amax"]),
            lambda: fq.nvfp4_quantize(xin, o["amax"], use_sr=True, seed=1000 + i, offset=0,
                                      q=o["q4"], sb=o["sb4"], g=o["g4"]),
            lambda: fq.nvfp4_quantize_2d(xin, o["amax"], o["q2"], o["sb2"], o["g2"]),
        ]

    def step(i, xin, o=None, offs_d=None):
        for fn in step_calls(i, xin, o, offs_d):
            fn()

    # warm-up passes, which also size the repetition count R of the timed steps
    wev = [(T.event(), T.event(), T.event()) for _ in range(args.warmup)]
    for i, (a, b, c) in enumerate(wev):
        a.record(stream)
        T.flush()
        b.record(stream)
        step(i, x)
        c.record(stream)
    torch.cuda.synchronize(dev)
    pass_ms = min(b.elapsed_time(c) for a, b, c in wev)
    flush_ms = min(a.elapsed_time(b) for a, b, c in wev)
    reps = max(1, math.ceil(TIMED_REGION_S * 1e3 / (args.steps * (pass_ms + flush_ms + 0.01))))
    if ws > 1:
        reps = int(max_over_ranks(float(reps), dev))

    # The timed region: K steps x R passes, CUDA events at the two ends of
    # every pass only.  An event recorded between two kernels holds the next
    # launch until it is processed (about 2 us per kernel boundary), so the
    # split of the step over its kernels is measured in a second pass below.
    npass = args.steps * reps
    sevs = [(T.event(), T.event()) for _ in range(npass)]
    sampler = ClockSampler(dev.index)
    sampler.start()
    time.sleep(0.3)  # let the sampler start before the timed region
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    t0 = time.time()
    for i, (a, b) in enumerate(sevs):
        T.flush()
        a.record(stream)
        step(i, x)
        b.record(stream)
    torch.cuda.synchronize(dev)
    t1 = time.time()
    if ws > 1:
        dist.barrier()
    clocks = sampler.stop(t0, t1)
    pass_total_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in sevs), dev)
    ms_per_step = pass_total_ms / npass
    value = ws * step_bytes * npass / (pass_total_ms * 1e-3) / 1e9

    # the split: the same passes with an event between every two kernels,
    # and each cast alone with L2 flushed before it
    split_reps = max(3, min(args.steps, 200))
    per_us, _ = T.chain_us(step_calls(0, x), split_reps)
    kernels = {}
    for k, us in zip(KERNELS, per_us):
        us = max_over_ranks(us, dev)
        gbs, fr = frac(nbytes[k], us)
        kernels[k] = {"us": round(us, 2), "bytes": nbytes[k], "GB/s": gbs, "frac": fr}
    for k, fn in zip(KERNELS, step_calls(7, x)):
        us = max_over_ranks(T.alone_us(fn, split_reps), dev)
        gbs, fr = frac(nbytes[k], us)
        kernels[k]["alone"] = {"us": round(us, 2), "GB/s": gbs, "frac": fr}
    # the dominant kernel: the longest on its own (L2 flushed before the
    # call).  In the chain the amax's events also carry the write-back of
    # the transposed cast's output still dirty in L2 (about 60 MB), which
    # puts the amax and the 1x16 quantizer within a few tenths of a
    # microsecond of each other there, in either order from run to run.
    dom = max(KERNELS, key=lambda k: kernels[k]["alone"]["us"])
    roofline = {"bound": "hbm", "kernel": dom, "achieved": kernels[dom]["GB/s"],
                "peak": peak, "unit": "GB/s", "frac": kernels[dom]["frac"],
                "traffic": ncu_traffic(dom), "peak_source": f"hbm_gbs of {peak_kind}",
                "algorithmic_bytes": nbytes[dom],
                "timing": "CUDA events around the kernel inside the step (split pass)",
                "dominant": "longest alone (L2 flushed); the longest in the chain is "
                            + max(KERNELS, key=lambda k: kernels[k]["us"])}

    # ---------------------------------------------------------------- calls
    # beyond the six casts, on the same tensor, each timed alone
    extra_reps = max(3, min(args.steps, 200))
    E = M * K

    def entry(call, us, nb, launches, traffic_key=None, **kw):
        gbs, fr = frac(nb, us)
        return {"call": call, "us": round(us, 2), "bytes": nb, "GB/s": gbs, "frac": fr,
                "launches_per_call": launches, "traffic": ncu_traffic(traffic_key or call), **kw}

    def alone(fn):
        return max_over_ranks(T.alone_us(fn, extra_reps), dev)

    fo = {k: torch.empty_like(out[k]) for k in ("q", "s", "y", "ys", "yT", "yTs")}
    fused_us = alone(lambda: fq.bf16_to_mxfp4_fp8(x, offs, 0, fo["q"], fo["s"], fo["y"], fo["ys"],
                                                  fo["yT"], fo["yTs"]))
    single_us = alone(lambda: fq.bf16_to_mxfp4_fp8_single_pass(x, offs, 0, fo["q"], fo["s"], fo["y"],
                                                               fo["ys"], fo["yT"], fo["yTs"]))
    sep_us = sum(kernels[k]["alone"]["us"] for k in KERNELS[:3])
    rht_mask = 0x9E37
    ar = torch.empty((1,), **f32)
    amax_rht_us = alone(lambda: fq.nvfp4_amax_rht(x, rht_mask, ar))
    rht_us = alone(lambda: fq.nvfp4_quantize_rht(x, ar, rht_mask, True, 4242, 0, out["q4"],
                                                 out["sb4"], out["g4"]))
    rht_rne_us = alone(lambda: fq.nvfp4_quantize_rht(x, ar, rht_mask, False, 0, 0, out["q4"],
                                                     out["sb4"], out["g4"]))
    fy = torch.empty((M, K), **u8)
    fs1 = torch.empty((M, K // 128), **f32)
    fs2 = torch.empty((M // 128, K // 128), **f32)
    fp8_1x128_us = alone(lambda: fq.fp8_quantize_1x128(x, fy, fs1))
    fp8_128_us = alone(lambda: fq.fp8_quantize_128x128(x, fy, fs2))
    deq = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
    deq_us = alone(lambda: fq.mxfp4_dequantize_rows(out["q"], out["s"], deq))
    hist = fq.amax_history(64, device=dev)
    dstep = [0]

    def delayed_call():
        fq.nvfp4_quantize_delayed(x, hist, dstep[0], True, 99, 0, out["q4"], out["sb4"], out["g4"])
        dstep[0] += 1

    delayed_us = alone(delayed_call)
    qT = torch.empty((K, M // 2), **u8)
    sbT = torch.empty((K // 16, M // 16), **u8)
    w2t_us = alone(lambda: fq.nvfp4_quantize_2d_t(x, out["amax"], out["q2"], out["sb2"], qT, sbT,
                                                  out["g2"]))
    mma_n = fq.mxfp4_scales_mma_bytes(M, K)
    s_mma = torch.empty((mma_n,), **u8)
    mma_us = alone(lambda: fq.mxfp4_scales_mma_layout(out["s"], s_mma))
    next_rows = {
        "bf16_to_mxfp4_fp8": entry("bf16_to_mxfp4_fp8", fused_us, b_fused(M, K, nb_cols, G),
                                   1 + fq.fp4_to_fp8_cols_launch_count(K),
                                   separate_calls_alone_us=round(sep_us, 2)),
        "bf16_to_mxfp4_fp8_single_pass": entry("bf16_to_mxfp4_fp8_single_pass", single_us,
                                               b_fused(M, K, nb_cols, G), 1),
        "nvfp4_amax_rht": entry("nvfp4_amax_rht", amax_rht_us, 2 * E + 4, 2),
        "nvfp4_quantize_rht_sr": entry("nvfp4_quantize_rht", rht_us, b_nvfp4(M, K), 1,
                                       sign_mask=rht_mask),
        "nvfp4_quantize_rht_rne": entry("nvfp4_quantize_rht", rht_rne_us, b_nvfp4(M, K), 1,
                                        traffic_key="nvfp4_quantize_rht_rne", sign_mask=rht_mask),
        "fp8_quantize_1x128": entry("fp8_quantize_1x128", fp8_1x128_us, 3 * E + 4 * (E // 128), 1),
        "fp8_quantize_128x128": entry("fp8_quantize_128x128", fp8_128_us,
                                      3 * E + 4 * (E // 16384), 1),
        "mxfp4_dequantize_rows": entry("mxfp4_dequantize_rows", deq_us,
                                       E // 2 + E // 32 + 2 * E, 1),
        "nvfp4_quantize_delayed_sr": entry(
            "nvfp4_quantize_delayed", delayed_us, b_nvfp4(M, K) + 16 * 65, 1, window=64,
            amax_then_quantize_alone_us=round(kernels["nvfp4_amax"]["alone"]["us"] +
                                              kernels["nvfp4_quantize"]["alone"]["us"], 2)),
        "nvfp4_quantize_2d_t": entry("nvfp4_quantize_2d_t", w2t_us, b_2d_t(M, K), 1,
                                     without_transpose_alone_us=kernels["nvfp4_quantize_2d"][
                                         "alone"]["us"]),
        "mxfp4_scales_mma_layout": entry("mxfp4_scales_mma_layout", mma_us, E // 32 + mma_n, 1,
                                         l2_resident=E // 32 + mma_n <= l2_bytes),
        "reps": extra_reps, "timing": "alone, L2 flushed before every call",
    }
    del fo, fy, fs1, fs2, deq, qT, sbT, s_mma

    # ---------------------------------------------------------------- configs
    cfg_reps = max(3, min(args.steps, 50))
    host = {"pr1": workloads.pr1(256, 512, seed=0), "moe_dispatch": (bits, offs_np)}
    configs = {}

    def run_config(name, workload, calls):
        """calls: (label, fn, bytes) in chain order."""
        fns = [c[1] for c in calls]
        per, total = T.chain_us(fns, cfg_reps)
        res = {"workload": workload, "calls": {}}
        tot_bytes = 0
        for (label, fn, nbb), us_c in zip(calls, per):
            us_c = max_over_ranks(us_c, dev)
            us_a = max_over_ranks(T.alone_us(fn, cfg_reps), dev)
            gc, fc = frac(nbb, us_c)
            ga, fa = frac(nbb, us_a)
            res["calls"][label] = {"bytes": nbb, "chained_us": round(us_c, 2), "chained_frac": fc,
                                   "alone_us": round(us_a, 2), "alone_GB/s": ga, "alone_frac": fa,
                                   "l2_resident": nbb <= l2_bytes}
            tot_bytes += nbb
        total = max_over_ranks(total, dev)
        g, f = frac(tot_bytes, total)
        res["chain"] = {"us": round(total, 2), "GB/s": g, "frac": f,
                        "events": "at the chain's two ends"}
        configs[name] = res

    def mx_outputs(Mc, Kc, Gc):
        capc = fq.fp4_to_fp8_cols_scale_capacity(Mc, Gc)
        return {"q": torch.empty((Mc, Kc // 2), **u8), "s": torch.empty((Mc, Kc // 32), **u8),
                "y": torch.empty((Mc, Kc), **u8), "ys": torch.empty((Mc, Kc // 128), **f32),
                "yT": torch.empty((Kc, Mc), **u8), "yTs": torch.empty((capc, Kc), **f32)}

    # PR1: 256 x 512 (L2-resident), MXFP4 then FP8 rows at k = 0 and 6
    xp = to_dev(host["pr1"])
    op = mx_outputs(256, 512, 1)
    run_config("pr1 256x512", "N(0,1), 0.1% x100 (seed 0)", [
        ("mxfp4_quantize_rows", lambda: fq.mxfp4_quantize_rows(xp, op["q"], op["s"]),
         b_mxfp4(256, 512)),
        ("fp4_to_fp8_rows k=0", lambda: fq.fp4_to_fp8_rows(op["q"], op["s"], 0, op["y"], op["ys"]),
         b_rows(256, 512)),
        ("fp4_to_fp8_rows k=6", lambda: fq.fp4_to_fp8_rows(op["q"], op["s"], 6, op["y"], op["ys"]),
         b_rows(256, 512))])
    del xp, op

    # MoE dispatch: the headline chain (its figures are in `kernels` as well)
    run_config("moe_dispatch 16384x7168", "N(0,1) x row lognormal(0,1), 32 Zipf(1.1) experts",
               list(zip(KERNELS, step_calls(3, x), [nbytes[k] for k in KERNELS])))

    # ragged experts: 65536 x 2048, 32 Zipf(1.1) groups: MXFP4, then the
    # transposed conversion
    Mr, Kr = 65536, 2048
    bits_r, offs_r = workloads.ragged_experts(Mr, Kr, 32, seed=0)
    host["ragged_experts"] = (bits_r, offs_r)
    xr = to_dev(bits_r)
    offr = torch.from_numpy(offs_r).to(dev)
    orr = mx_outputs(Mr, Kr, 32)
    run_config("ragged_experts 65536x2048", "N(0,1), 32 experts Zipf(1.1), no padding", [
        ("mxfp4_quantize_rows", lambda: fq.mxfp4_quantize_rows(xr, orr["q"], orr["s"]),
         b_mxfp4(Mr, Kr)),
        ("fp4_to_fp8_cols", lambda: fq.fp4_to_fp8_cols(orr["q"], orr["s"], offr, 0, orr["yT"],
                                                       orr["yTs"]),
         b_cols(Mr, Kr, col_blocks(offs_r), 32))])
    del xr, offr, orr

    # NVFP4: activations 16384 x 14336 Student-t(4) (amax, SR, RNE) and
    # weights 14336 x 4096 N(0, 0.02) (amax, 2D, 2D with the DGRAD operand)
    Ma, Ka = 16384, 14336
    host["nvfp4_act"] = workloads.nvfp4_act(Ma, Ka, seed=0)
    xa = to_dev(host["nvfp4_act"])
    aa = torch.empty((1,), **f32)
    qa, sba, ga = (torch.empty((Ma, Ka // 2), **u8), torch.empty((Ma, Ka // 16), **u8),
                   torch.empty((1,), **f32))
    run_config("nvfp4 activations 16384x14336", "Student-t(4), seed 0", [
        ("nvfp4_amax", lambda: fq.nvfp4_amax(xa, aa), b_amax(Ma, Ka)),
        ("nvfp4_quantize SR", lambda: fq.nvfp4_quantize(xa, aa, True, 1234, 0, qa, sba, ga),
         b_nvfp4(Ma, Ka)),
        ("nvfp4_quantize RNE", lambda: fq.nvfp4_quantize(xa, aa, False, 0, 0, qa, sba, ga),
         b_nvfp4(Ma, Ka))])
    del xa, qa, sba
    Nw, Kw = 14336, 4096
    host["nvfp4_weight"] = workloads.nvfp4_weight(Nw, Kw, seed=0)
    xw = to_dev(host["nvfp4_weight"])
    aw = torch.empty((1,), **f32)
    qw, sbw, gw = (torch.empty((Nw, Kw // 2), **u8), torch.empty((Nw // 16, Kw // 16), **u8),
                   torch.empty((1,), **f32))
    qwT, sbwT = torch.empty((Kw, Nw // 2), **u8), torch.empty((Kw // 16, Nw // 16), **u8)
    run_config("nvfp4 weights 14336x4096", "N(0, 0.02), seed 0", [
        ("nvfp4_amax", lambda: fq.nvfp4_amax(xw, aw), b_amax(Nw, Kw)),
        ("nvfp4_quantize_2d", lambda: fq.nvfp4_quantize_2d(xw, aw, qw, sbw, gw), b_2d(Nw, Kw)),
        ("nvfp4_quantize_2d_t", lambda: fq.nvfp4_quantize_2d_t(xw, aw, qw, sbw, qwT, sbwT, gw),
         b_2d_t(Nw, Kw))])
    del xw, qw, sbw, qwT, sbwT

    # bandwidth sweep: M = 1K .. 256K rows x 7168 Student-t(3): MXFP4, FP8
    # rows, FP8 columns (one group); every size is a prefix of the largest
    Ks, Mmax = 7168, SWEEP_ROWS[-1]
    bits_s = workloads.sweep(Mmax, Ks, seed=0)
    host["sweep_sample"] = np.ascontiguousarray(bits_s[:16384])
    xs = to_dev(bits_s)
    del bits_s
    qs, ss = torch.empty((Mmax, Ks // 2), **u8), torch.empty((Mmax, Ks // 32), **u8)
    ys_, yss = torch.empty((Mmax, Ks), **u8), torch.empty((Mmax, Ks // 128), **f32)
    yTflat = torch.empty((Mmax * Ks,), **u8)
    yTsflat = torch.empty(((Mmax // 128 + 1) * Ks,), **f32)
    for m in SWEEP_ROWS:
        xm, qm, sm, ym, ysm = xs[:m], qs[:m], ss[:m], ys_[:m], yss[:m]
        yTm = yTflat[: m * Ks].view(Ks, m)
        capm = fq.fp4_to_fp8_cols_scale_capacity(m, 1)
        yTsm = yTsflat[: capm * Ks].view(capm, Ks)
        om = torch.tensor([0, m], dtype=torch.int64, device=dev)
        run_config(f"sweep {m}x7168", "Student-t(3), seed 0 (prefix rows), one group", [
            ("mxfp4_quantize_rows", lambda: fq.mxfp4_quantize_rows(xm, qm, sm), b_mxfp4(m, Ks)),
            ("fp4_to_fp8_rows", lambda: fq.fp4_to_fp8_rows(qm, sm, 0, ym, ysm), b_rows(m, Ks)),
            ("fp4_to_fp8_cols", lambda: fq.fp4_to_fp8_cols(qm, sm, om, 0, yTm, yTsm),
             b_cols(m, Ks, (m + 127) // 128, 1))])
    del xs, qs, ss, ys_, yss, yTflat, yTsflat

    # a hidden size that is a multiple of 128 but not of 512 (the transposed
    # conversion's exponent rows by four-row groups), MoE-dispatch recipe, 32
    # Zipf experts; then the same with a token count that is not a multiple
    # of 16 (output rows of yT not 16-byte aligned, the last M % 4 exponent
    # rows patched)
    Mt, Kt = 16384, TWO_LAUNCH_K
    xt = to_dev(workloads.moe_dispatch(Mt, Kt, seed=0))
    offt = torch.from_numpy(offs_np).to(dev)
    ot = mx_outputs(Mt, Kt, 32)
    run_config(f"moe_dispatch {Mt}x{Kt} (K % 512 != 0)",
               f"N(0,1) x row lognormal(0,1), 32 Zipf(1.1) experts; the transposed conversion "
               f"launches {fq.fp4_to_fp8_cols_launch_count(Kt)} kernels", [
                   ("mxfp4_quantize_rows", lambda: fq.mxfp4_quantize_rows(xt, ot["q"], ot["s"]),
                    b_mxfp4(Mt, Kt)),
                   ("fp4_to_fp8_cols", lambda: fq.fp4_to_fp8_cols(ot["q"], ot["s"], offt, 0,
                                                                  ot["yT"], ot["yTs"]),
                    b_cols(Mt, Kt, nb_cols, 32))])
    del xt, offt, ot
    Mu = 16389
    offs_u = workloads.zipf_group_offsets(Mu, EXPERTS, 1.1, 0)
    xu = to_dev(workloads.moe_dispatch(Mu, Kt, seed=0))
    offu = torch.from_numpy(offs_u).to(dev)
    ou = mx_outputs(Mu, Kt, 32)
    run_config(f"moe_dispatch {Mu}x{Kt} (M % 16 != 0, K % 512 != 0)",
               "N(0,1) x row lognormal(0,1), 32 Zipf(1.1) experts", [
                   ("mxfp4_quantize_rows", lambda: fq.mxfp4_quantize_rows(xu, ou["q"], ou["s"]),
                    b_mxfp4(Mu, Kt)),
                   ("fp4_to_fp8_cols", lambda: fq.fp4_to_fp8_cols(ou["q"], ou["s"], offu, 0,
                                                                  ou["yT"], ou["yTs"]),
                    b_cols(Mu, Kt, col_blocks(offs_u), 32))])
    del xu, offu, ou
    torch.cuda.empty_cache()
    # the bar: every call on a tensor of at least 4x L2 at >= 75 % alone
    big = [(n, lab, c["alone_frac"]) for n, cf in configs.items() for lab, c in cf["calls"].items()
           if c["bytes"] >= 4 * l2_bytes]
    worst = min(big, key=lambda t: t[2]) if big else None
    configs_summary = {"l2_bytes": l2_bytes, "reps": cfg_reps,
                       "calls_at_least_4x_l2": len(big),
                       "min_alone_frac_at_least_4x_l2": (
                           {"config": worst[0], "call": worst[1], "frac": worst[2]}
                           if worst else None)}

    # ---------------------------------------------------------------- end to end
    # through host buffers: every step copies its input (and the group
    # offsets) from pinned host memory, runs all casts and copies every
    # output back to pinned host memory.  Three streams pipeline the steps
    # (H2D of step i+1 and D2H of step i-1 overlap the casts of step i);
    # device inputs and outputs are double buffered, ordered by events.
    e2e_steps = max(3, min(args.steps, 30))
    xh = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).pin_memory()
    offs_h = torch.from_numpy(offs_np).pin_memory()
    xds = [torch.empty_like(x) for _ in range(2)]
    offds = [torch.empty_like(offs) for _ in range(2)]
    outs = [out, {k: torch.empty_like(v) for k, v in out.items()}]
    outs_h = {k: torch.empty(v.shape, dtype=v.dtype).pin_memory() for k, v in out.items()}
    h2d = xh.numel() * 2 + offs_h.numel() * 8
    d2h = sum(v.numel() * v.element_size() for k, v in out.items())
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def e2e_run(nsteps):
        ev_in = [torch.cuda.Event() for _ in range(nsteps)]
        ev_comp = [torch.cuda.Event() for _ in range(nsteps)]
        ev_out = [torch.cuda.Event() for _ in range(nsteps)]
        t0e, t1e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0e.record(s_in)
        for i in range(nsteps):
            b = i & 1
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_comp[i - 2])   # input buffer b is free
                xds[b].copy_(xh, non_blocking=True)
                offds[b].copy_(offs_h, non_blocking=True)
                ev_in[i].record(s_in)
            stream.wait_event(ev_in[i])
            if i >= 2:
                stream.wait_event(ev_out[i - 2])      # output buffer b was read back
            step(i, xds[b], o=outs[b], offs_d=offds[b])
            ev_comp[i].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_comp[i])
                for k, v in outs[b].items():
                    outs_h[k].copy_(v, non_blocking=True)
                ev_out[i].record(s_out)
        t1e.record(s_out)
        torch.cuda.synchronize(dev)
        return t0e.elapsed_time(t1e)

    e2e_run(2)  # warm-up
    if ws > 1:
        dist.barrier()
    e2e_ms = max_over_ranks(e2e_run(e2e_steps), dev) / e2e_steps
    e2e_value = ws * step_bytes / (e2e_ms * 1e-3) / 1e9
    link = link_rates(dev)
    # the link's bound on a step: its copies take at least the longer of each
    # direction alone, and of both directions' bytes at the two-way rate
    t_link = max(h2d / (link["h2d"] * 1e9), d2h / (link["d2h"] * 1e9),
                 (h2d + d2h) / (link["both_directions_total"] * 1e9))
    e2e_bound = ws * step_bytes / t_link / 1e9
    del xds, outs, outs_h

    cpu, errs = None, None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline()
        errs = oracle_error_stats(host)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": WORKLOAD, "M": M, "K": K, "experts": G,
                       "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU",
                       "l2": "flushed before every pass (256 MB write + read, outside the "
                             "timed events)",
                       "step_bytes": step_bytes,
                       "reps_per_step": reps,
                       "timing": f"each of the {args.steps} steps is one pass of the six casts "
                                 f"repeated {reps} times; ms_per_step is per pass"},
            "frac_of_hbm_peak": round(value / ws / peak, 4),
            "kernels": kernels,
            "roofline": roofline,
            "next_rows": next_rows,
            "configs": configs,
            "configs_summary": configs_summary,
            "e2e": {"value": round(e2e_value, 1), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 3),
                    "pipelining": "H2D / casts / D2H on three streams, double-buffered",
                    "link_gbs": link, "link_bound": round(e2e_bound, 1),
                    "frac_of_link_bound": round(e2e_value / e2e_bound, 4)},
            "gpu_launches": launches_per_pass * npass,
            "clocks": clocks,
            "cpu_baseline": cpu,
            "error_stats": errs,
            "wall_s_timed_region": round(t1 - t0, 4),
            "wall_s_total": round(time.time() - wall0, 1),
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()
    return 0


def run_sweep_rows(m):
    """The bandwidth-sweep chain at m rows x 7168 alone (mxfp4_quantize_rows,
    fp4_to_fp8_rows, fp4_to_fp8_cols with one group), one launch per call with
    L2 cleaned before each: a small case for a full ncu capture of one size."""
    import torch
    import numpy as np
    import fp8_quantization_gb300 as fq
    from fp8_quantization_gb300 import workloads
    dev = torch.device("cuda", 0)
    T = Timer(dev, 0)

    def run(fn):
        T.flush()
        return fn()

    bits = workloads.sweep(m, 7168, seed=0)
    x = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)
    del bits
    q, s = run(lambda: fq.mxfp4_quantize_rows(x))
    del x
    run(lambda: fq.fp4_to_fp8_rows(q, s, 0))
    offs = torch.tensor([0, m], dtype=torch.int64, device=dev)
    run(lambda: fq.fp4_to_fp8_cols(q, s, offs, 0))
    torch.cuda.synchronize(dev)
    print(json.dumps({"sweep_rows": m}), flush=True)
    return 0


def run_ncu_cols(m: int, k: int, reps: int = 3):
    """The transposed conversion alone on the MoE-dispatch recipe at m x k
    (32 Zipf groups), `reps` calls with L2 cleaned before each, after one
    MXFP4 row quantization that makes its input: a small case for an ncu
    capture of one instance of the kernel (any m, such as one that is not a
    multiple of 16)."""
    import torch
    import numpy as np
    import fp8_quantization_gb300 as fq
    from fp8_quantization_gb300 import workloads
    dev = torch.device("cuda", 0)
    T = Timer(dev, 0)
    bits = workloads.moe_dispatch(m, k, seed=0)
    offs = torch.from_numpy(workloads.zipf_group_offsets(m, EXPERTS, 1.1, 0)).to(dev)
    x = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)
    q, s = fq.mxfp4_quantize_rows(x)
    yT, yTs = fq.fp4_to_fp8_cols(q, s, offs, 0)
    for _ in range(reps):
        T.flush()
        fq.fp4_to_fp8_cols(q, s, offs, 0, yT, yTs)
    torch.cuda.synchronize(dev)
    print(json.dumps({"ncu_cols": [m, k], "reps": reps}), flush=True)
    return 0


def run_ncu_calls(reps: int = 3):
    """Every entry point of the DRAM-traffic record on the headline tensor
    (16384 x 7168, 32 Zipf groups), each `reps` times with L2 cleaned before
    each call, and nothing else: about 2 GB on the device and a few dozen
    launches, a small case for an ncu capture of DRAM bytes per call."""
    import torch
    import numpy as np
    import fp8_quantization_gb300 as fq
    from fp8_quantization_gb300 import workloads
    dev = torch.device("cuda", 0)
    T = Timer(dev, 0)
    M, K, G = M_ROWS, K_COLS, EXPERTS
    bits = workloads.moe_dispatch(M, K, seed=0)
    offs_np = workloads.zipf_group_offsets(M, G, 1.1, 0)
    x = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)
    del bits
    offs = torch.from_numpy(offs_np).to(dev)
    q, s = fq.mxfp4_quantize_rows(x)
    amax = fq.nvfp4_amax(x)
    ar = fq.nvfp4_amax_rht(x, 0x9E37)
    hist = fq.amax_history(64, device=dev)
    calls = [
        lambda: fq.mxfp4_quantize_rows(x, q, s),
        lambda: fq.fp4_to_fp8_rows(q, s, 0),
        lambda: fq.fp4_to_fp8_cols(q, s, offs, 0),
        lambda: fq.nvfp4_amax(x, amax),
        lambda: fq.nvfp4_quantize(x, amax, use_sr=True, seed=1000, offset=0),
        lambda: fq.nvfp4_quantize_2d(x, amax),
        lambda: fq.nvfp4_amax_rht(x, 0x9E37, ar),
        lambda: fq.nvfp4_quantize_rht(x, ar, 0x9E37, True, 4242, 0),
        lambda: fq.nvfp4_quantize_rht(x, ar, 0x9E37, False, 0, 0),
        lambda: fq.fp8_quantize_1x128(x),
        lambda: fq.fp8_quantize_128x128(x),
        lambda: fq.mxfp4_dequantize_rows(q, s),
        lambda: fq.nvfp4_quantize_2d_t(x, amax),
        lambda: fq.nvfp4_quantize_delayed(x, hist, 0, True, 99, 0),
        lambda: fq.bf16_to_mxfp4_fp8(x, offs, 0),
        lambda: fq.mxfp4_scales_mma_layout(s),
        lambda: fq.bf16_to_mxfp4_fp8_single_pass(x, offs, 0),
    ]
    for fn in calls:
        for _ in range(reps):
            T.flush()
            fn()
            torch.cuda.synchronize(dev)
    print(json.dumps({"ncu_calls": len(calls), "reps": reps}), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["fq", "reference"], default="fq")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sweep-rows", type=int, default=0,
                    help="run the bandwidth-sweep chain at this many rows once (for an ncu "
                         "capture of one size) and exit")
    ap.add_argument("--ncu-calls", action="store_true",
                    help="run every entry point of the DRAM-traffic record three times on the "
                         "headline tensor and exit (for an ncu capture of DRAM bytes per call)")
    ap.add_argument("--ncu-cols", type=int, nargs=2, metavar=("M", "K"), default=None,
                    help="run the transposed conversion alone on the MoE-dispatch recipe at "
                         "M x K (32 groups) four times and exit (for an ncu capture of one "
                         "instance)")
    args = ap.parse_args()
    if args.ncu_calls:
        return run_ncu_calls()
    if args.ncu_cols:
        return run_ncu_cols(*args.ncu_cols)
    if args.sweep_rows:
        return run_sweep_rows(args.sweep_rows)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
