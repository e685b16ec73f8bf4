#!/usr/bin/env python3
"""Benchmark of the block-scaled cast path on one GB300 (or N replicas).

One step = every cast of the path over one batch of the MoE-dispatch
activations workload (BF16 16384 x 7168, N(0,1) rows times a per-row
log-normal(0,1) magnitude, seed 0; the tokens are split over 32 experts with
Zipf(1.1) counts for the transposed ragged conversion):

  1. mxfp4_quantize_rows   BF16 -> MXFP4 (packed E2M1 + UE8M0)
  2. fp4_to_fp8_rows       MXFP4 -> E4M3, 128-element blocks, k = 0
  3. fp4_to_fp8_cols       MXFP4 -> E4M3 transposed, 32 ragged expert groups
  4. nvfp4_amax            per-tensor amax
  5. nvfp4_quantize        NVFP4 1x16, stochastic rounding (seed = step)
  6. nvfp4_quantize_2d     NVFP4 16x16 on the same tensor

The metric is effective bandwidth: algorithmic bytes read + written by the
kernels over their device time (CUDA events on the launching stream), as GB/s
and as a fraction of the measured HBM copy bandwidth.  L2 is flushed (256 MB
written, then read back) between steps, outside the timed events.

--impl reference times the CPU oracle (the plain C implementation the tests
compare against) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
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
# kernels of libfq.so each entry point launches (nvfp4_amax: the one-thread
# zeroing of the amax word, then the reduction)
LAUNCHES = {"mxfp4_quantize_rows": 1, "fp4_to_fp8_rows": 1, "fp4_to_fp8_cols": 2,  # or 1 (K)
            "nvfp4_amax": 2, "nvfp4_quantize": 1, "nvfp4_quantize_2d": 1}
# source file of each kernel (for the ncu traffic record's staleness check)
KERNEL_SRC = {
    "mxfp4_quantize_rows": "fq_mxfp4.cu", "fp4_to_fp8_rows": "fq_mxfp4.cu",
    "fp4_to_fp8_cols": "fq_cols.cu", "nvfp4_amax": "fq_nvfp4.cu",
    "nvfp4_quantize": "fq_nvfp4.cu", "nvfp4_quantize_2d": "fq_nvfp4.cu",
    "bf16_to_mxfp4_fp8": "fq_mxfp4.cu", "nvfp4_amax_rht": "fq_nvfp4.cu",
    "nvfp4_quantize_rht": "fq_nvfp4.cu", "fp8_quantize_1x128": "fq_fp8.cu",
    "fp8_quantize_128x128": "fq_fp8.cu", "mxfp4_dequantize_rows": "fq_fp8.cu",
    "nvfp4_quantize_delayed": "fq_nvfp4.cu", "nvfp4_quantize_2d_t": "fq_nvfp4.cu",
}
FALLBACK_HBM_GBS = 6800.0


def algorithmic_bytes(M: int, K: int, nblocks_cols: int, G: int) -> dict:
    """Bytes each kernel must read + write (inputs once, outputs once)."""
    E = M * K
    return {
        "mxfp4_quantize_rows": 2 * E + E // 2 + E // 32,
        "fp4_to_fp8_rows": E // 2 + E // 32 + E + 4 * (E // 128),
        "fp4_to_fp8_cols": E // 2 + E // 32 + E + 4 * K * nblocks_cols + 8 * (G + 1),
        "nvfp4_amax": 2 * E + 4,
        "nvfp4_quantize": 2 * E + E // 2 + E // 16 + 8,
        "nvfp4_quantize_2d": 2 * E + E // 2 + E // 256 + 8,
    }


def hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def file_sha(name: str) -> str:
    """sha256[:16] of a kernel's source file followed by the shared header."""
    h = hashlib.sha256()
    for part in (name, "fq_common.cuh"):
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
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            f = [x.strip() for x in r.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
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
    import numpy as np
    nb = int(((np.diff(offs_rows) + 127) // 128).sum())
    return dt, sum(algorithmic_bytes(M, K, nb, G).values())


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

    M, K, G = M_ROWS, K_COLS, EXPERTS
    bits = workloads.moe_dispatch(M, K, seed=0)
    offs_np = workloads.zipf_group_offsets(M, G, 1.1, 0)
    nb_cols = int(((np.diff(offs_np) + 127) // 128).sum())
    nbytes = algorithmic_bytes(M, K, nb_cols, G)
    launches_per_step = sum(LAUNCHES.values()) - LAUNCHES["fp4_to_fp8_cols"] + \
        fq.fp4_to_fp8_cols_launch_count(K)
    step_bytes = sum(nbytes.values())

    x = torch.from_numpy(bits.view(np.int16)).to(dev).view(torch.bfloat16)
    offs = torch.from_numpy(offs_np).to(dev)
    cap = fq.fp4_to_fp8_cols_scale_capacity(M, G)
    u8 = dict(dtype=torch.uint8, device=dev)
    f32 = dict(dtype=torch.float32, device=dev)
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
    flush_buf = torch.empty((256 << 20,), dtype=torch.uint8, device=dev)

    def flush():
        # evict L2 (2x its size): write a buffer, then read it back so that
        # the flush's own dirty lines are written out here, not in the next step
        flush_buf.fill_(1)
        flush_buf.sum(dtype=torch.int64)

    stream = torch.cuda.current_stream(dev)

    def step(i, xin, ev=None, o=None, offs_d=None):
        o = out if o is None else o
        offs_d = offs if offs_d is None else offs_d
        if ev:
            ev[0].record(stream)
        fq.mxfp4_quantize_rows(xin, o["q"], o["s"])
        if ev:
            ev[1].record(stream)
        fq.fp4_to_fp8_rows(o["q"], o["s"], 0, o["y"], o["ys"])
        if ev:
            ev[2].record(stream)
        fq.fp4_to_fp8_cols(o["q"], o["s"], offs_d, 0, o["yT"], o["yTs"])
        if ev:
            ev[3].record(stream)
        fq.nvfp4_amax(xin, o["amax"])
        if ev:
            ev[4].record(stream)
        fq.nvfp4_quantize(xin, o["amax"], use_sr=True, seed=1000 + i, offset=0, q=o["q4"],
                          sb=o["sb4"], g=o["g4"])
        if ev:
            ev[5].record(stream)
        fq.nvfp4_quantize_2d(xin, o["amax"], o["q2"], o["sb2"], o["g2"])
        if ev:
            ev[6].record(stream)

    for i in range(args.warmup):
        flush()
        step(i, x)
    torch.cuda.synchronize(dev)

    # The timed region: CUDA events at the two ends of every step only.  An
    # event recorded between two kernels holds the next launch until it is
    # processed (about 2 us per kernel boundary), so the split of the step
    # over its kernels is measured in a second pass below.
    sevs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    sampler = ClockSampler(dev.index)
    sampler.start()
    time.sleep(0.3)  # let the sampler start before the timed region
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    t0 = time.time()
    for i in range(args.steps):
        flush()
        sevs[i][0].record(stream)
        step(i, x)
        sevs[i][1].record(stream)
    torch.cuda.synchronize(dev)
    t1 = time.time()
    if ws > 1:
        dist.barrier()
    clocks = sampler.stop(t0, t1)
    step_ms = sum(a.elapsed_time(b) for a, b in sevs)
    step_ms_max = max_over_ranks(step_ms, dev)
    ms_per_step = step_ms_max / args.steps
    value = ws * step_bytes * args.steps / (step_ms_max * 1e-3) / 1e9

    # the split: the same steps with an event between every two kernels
    split_steps = max(3, min(args.steps, 200))
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(7)] for _ in range(split_steps)]
    for i in range(split_steps):
        flush()
        step(i, x, evs[i])
    torch.cuda.synchronize(dev)
    per_kernel_ms = {k: 0.0 for k in KERNELS}
    split_ms = 0.0
    for ev in evs:
        for j, k in enumerate(KERNELS):
            per_kernel_ms[k] += ev[j].elapsed_time(ev[j + 1])
        split_ms += ev[0].elapsed_time(ev[6])
    for k in KERNELS:
        per_kernel_ms[k] = max_over_ranks(per_kernel_ms[k], dev) / split_steps
    split_ms_per_step = max_over_ranks(split_ms, dev) / split_steps

    peak, peak_kind = hbm_peak()
    kernels = {}
    for k in KERNELS:
        ms = per_kernel_ms[k]
        gbs = nbytes[k] / (ms * 1e-3) / 1e9
        kernels[k] = {"us": round(ms * 1e3, 2), "bytes": nbytes[k], "GB/s": round(gbs, 1),
                      "frac": round(gbs / peak, 4)}
    dom = max(KERNELS, key=lambda k: per_kernel_ms[k])
    traffic = ncu_traffic(dom)
    roofline = {"bound": "hbm", "kernel": dom, "achieved": kernels[dom]["GB/s"],
                "peak": peak, "unit": "GB/s", "frac": kernels[dom]["frac"],
                "traffic": traffic, "peak_source": f"hbm_gbs of {peak_kind}",
                "algorithmic_bytes": nbytes[dom]}

    # ---- calls beyond the six casts, on the same tensor, each timed alone
    # (L2 flushed before every call)
    extra_steps = max(3, min(args.steps, 200))

    def timed_us(fn):
        for _ in range(args.warmup):
            flush()
            fn()
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(extra_steps)]
        for i in range(extra_steps):
            flush()
            ev[i][0].record(stream)
            fn()
            ev[i][1].record(stream)
        torch.cuda.synchronize(dev)
        return max_over_ranks(sum(a.elapsed_time(b) for a, b in ev), dev) / extra_steps * 1e3

    def entry(call, us, nbytes, launches, **kw):
        gbs = nbytes / (us * 1e-6) / 1e9
        return {"call": call, "us": round(us, 2), "bytes": nbytes, "GB/s": round(gbs, 1),
                "frac": round(gbs / peak, 4), "launches_per_call": launches,
                "traffic": ncu_traffic(call), **kw}

    # the six casts again, each alone with L2 flushed before every call: the
    # per-kernel figure without the previous kernel's dirty lines (written
    # back during the next kernel in the step)
    alone = {
        "mxfp4_quantize_rows": lambda: fq.mxfp4_quantize_rows(x, out["q"], out["s"]),
        "fp4_to_fp8_rows": lambda: fq.fp4_to_fp8_rows(out["q"], out["s"], 0, out["y"], out["ys"]),
        "fp4_to_fp8_cols": lambda: fq.fp4_to_fp8_cols(out["q"], out["s"], offs, 0, out["yT"],
                                                      out["yTs"]),
        "nvfp4_amax": lambda: fq.nvfp4_amax(x, out["amax"]),
        "nvfp4_quantize": lambda: fq.nvfp4_quantize(x, out["amax"], use_sr=True, seed=7, offset=0,
                                                    q=out["q4"], sb=out["sb4"], g=out["g4"]),
        "nvfp4_quantize_2d": lambda: fq.nvfp4_quantize_2d(x, out["amax"], out["q2"], out["sb2"],
                                                          out["g2"]),
    }
    for k, fn in alone.items():
        us = timed_us(fn)
        gbs = nbytes[k] / (us * 1e-6) / 1e9
        kernels[k]["alone"] = {"us": round(us, 2), "GB/s": round(gbs, 1), "frac": round(gbs / peak, 4)}

    E = M * K
    fo = {k: torch.empty_like(out[k]) for k in ("q", "s", "y", "ys", "yT", "yTs")}
    fused_us = timed_us(lambda: fq.bf16_to_mxfp4_fp8(x, offs, 0, fo["q"], fo["s"], fo["y"],
                                                      fo["ys"], fo["yT"], fo["yTs"]))
    sep_us = sum(kernels[k]["us"] for k in ("mxfp4_quantize_rows", "fp4_to_fp8_rows",
                                             "fp4_to_fp8_cols"))
    rht_mask = 0x9E37
    ar = torch.empty((1,), dtype=torch.float32, device=dev)
    amax_rht_us = timed_us(lambda: fq.nvfp4_amax_rht(x, rht_mask, ar))
    rht_us = timed_us(lambda: fq.nvfp4_quantize_rht(x, ar, rht_mask, True, 4242, 0, out["q4"],
                                                     out["sb4"], out["g4"]))
    fy = torch.empty((M, K), dtype=torch.uint8, device=dev)
    fs1 = torch.empty((M, K // 128), dtype=torch.float32, device=dev)
    fs2 = torch.empty((M // 128, K // 128), dtype=torch.float32, device=dev)
    fp8_1x128_us = timed_us(lambda: fq.fp8_quantize_1x128(x, fy, fs1))
    fp8_128_us = timed_us(lambda: fq.fp8_quantize_128x128(x, fy, fs2))
    deq = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
    deq_us = timed_us(lambda: fq.mxfp4_dequantize_rows(out["q"], out["s"], deq))
    hist = fq.amax_history(64, device=dev)
    dstep = [0]

    def delayed_call():
        fq.nvfp4_quantize_delayed(x, hist, dstep[0], True, 99, 0, out["q4"], out["sb4"], out["g4"])
        dstep[0] += 1

    delayed_us = timed_us(delayed_call)
    qT = torch.empty((K, M // 2), dtype=torch.uint8, device=dev)
    sbT = torch.empty((K // 16, M // 16), dtype=torch.uint8, device=dev)
    w2t_us = timed_us(lambda: fq.nvfp4_quantize_2d_t(x, out["amax"], out["q2"], out["sb2"], qT,
                                                     sbT, out["g2"]))
    next_rows = {
        "bf16_to_mxfp4_fp8": entry(
            "bf16_to_mxfp4_fp8", fused_us,
            2 * E + E // 2 + E // 32 + E + 4 * (E // 128) + E + 4 * K * nb_cols + 8 * (G + 1),
            1 + fq.fp4_to_fp8_cols_launch_count(K), separate_calls_us=round(sep_us, 2)),
        "nvfp4_amax_rht": entry("nvfp4_amax_rht", amax_rht_us, 2 * E + 4, 1),
        "nvfp4_quantize_rht_sr": entry("nvfp4_quantize_rht", rht_us, 2 * E + E // 2 + E // 16 + 8,
                                       1, sign_mask=rht_mask),
        "fp8_quantize_1x128": entry("fp8_quantize_1x128", fp8_1x128_us, 3 * E + 4 * (E // 128), 1),
        "fp8_quantize_128x128": entry("fp8_quantize_128x128", fp8_128_us,
                                      3 * E + 4 * (E // 16384), 1),
        "mxfp4_dequantize_rows": entry("mxfp4_dequantize_rows", deq_us,
                                       E // 2 + E // 32 + 2 * E, 1),
        "nvfp4_quantize_delayed_sr": entry(
            "nvfp4_quantize_delayed", delayed_us, 2 * E + E // 2 + E // 16 + 16 * 65, 1, window=64,
            amax_then_quantize_us=round(kernels["nvfp4_amax"]["us"] +
                                        kernels["nvfp4_quantize"]["us"], 2)),
        "nvfp4_quantize_2d_t": entry(
            "nvfp4_quantize_2d_t", w2t_us, 2 * E + E // 2 + E // 256 + E // 2 + E // 256 + 8, 1,
            without_transpose_us=kernels["nvfp4_quantize_2d"]["us"]),
        "steps": extra_steps,
    }

    # ---- end to end through host buffers: every step copies its input (and
    # the group offsets) from pinned host memory, runs all casts and copies
    # every output back to pinned host memory.  Three streams pipeline the
    # steps (H2D of step i+1 and D2H of step i-1 overlap the casts of step i);
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

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline()

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": WORKLOAD, "M": M, "K": K, "experts": G,
                       "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU",
                       "l2": "flushed between steps (256 MB write + read, outside the timed events)",
                       "step_bytes": step_bytes},
            "frac_of_hbm_peak": round(value / ws / peak, 4),
            "kernels": kernels,
            "kernels_pass": {"steps": split_steps, "ms_per_step": round(split_ms_per_step, 4),
                             "events": "one between every two kernels (the timed steps have "
                                       "events at their ends only)"},
            "roofline": roofline,
            "next_rows": next_rows,
            "e2e": {"value": round(e2e_value, 1), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 3),
                    "pipelining": "H2D / casts / D2H on three streams, double-buffered"},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clocks,
            "cpu_baseline": cpu,
            "wall_s_timed_region": round(t1 - t0, 4),
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()
    return 0


# Launch order of --profile-configs (our kernels only), for reading an ncu
# capture of it: (configuration, call) per launch.
PROFILE_SWEEP = [1024 << i for i in range(9)]
PROFILE_ORDER = (
    [("cfg1 pr1 256x512", c) for c in ("mxfp4_quantize_rows", "fp4_to_fp8_rows k=0",
                                        "fp4_to_fp8_rows k=6")] +
    [("cfg2 moe_dispatch 16384x7168", c) for c in (
        "mxfp4_quantize_rows", "fp4_to_fp8_rows", "fp4_to_fp8_cols (32 Zipf groups)",
        "nvfp4_amax", "nvfp4_quantize SR", "nvfp4_quantize_2d")] +
    [("cfg3 ragged_experts 65536x2048", c) for c in (
        "mxfp4_quantize_rows", "fp4_to_fp8_cols (32 Zipf groups)")] +
    [("cfg4 nvfp4 activations 16384x14336", c) for c in (
        "nvfp4_amax", "nvfp4_quantize SR", "nvfp4_quantize RNE")] +
    [("cfg4 nvfp4 weights 14336x4096", c) for c in ("nvfp4_amax", "nvfp4_quantize_2d")] +
    [(f"cfg5 sweep {m}x7168", c) for m in PROFILE_SWEEP
     for c in ("mxfp4_quantize_rows", "fp4_to_fp8_rows", "fp4_to_fp8_cols (1 group)")])


def run_sweep_rows(m):
    """The bandwidth-sweep chain at m rows x 7168 alone (mxfp4_quantize_rows,
    fp4_to_fp8_rows, fp4_to_fp8_cols with one group), one launch per call with
    L2 cleaned before each: a small case for a full ncu capture of one size."""
    import torch
    import numpy as np
    import fp8_quantization_gb300 as fq
    from fp8_quantization_gb300 import workloads
    dev = torch.device("cuda", 0)
    flush_buf = torch.empty((256 << 20,), dtype=torch.uint8, device=dev)

    def run(fn):
        flush_buf.fill_(1)
        flush_buf.sum(dtype=torch.int64)
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


def run_profile_configs():
    """Every configuration's chain, one launch per call in PROFILE_ORDER, L2
    cleaned before each: the launches an ncu pass over the configurations
    captures.  Nothing is timed here; outputs are not checked (the tests do)."""
    import torch
    import numpy as np
    import fp8_quantization_gb300 as fq
    from fp8_quantization_gb300 import workloads
    dev = torch.device("cuda", 0)
    flush_buf = torch.empty((256 << 20,), dtype=torch.uint8, device=dev)

    def flush():
        flush_buf.fill_(1)
        flush_buf.sum(dtype=torch.int64)

    def run(fn):
        flush()
        return fn()

    def dev_bf16(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)

    def offs_dev(o):
        return torch.from_numpy(np.asarray(o, dtype=np.int64)).to(dev)

    x = dev_bf16(workloads.pr1(256, 512, seed=0))
    q, s = run(lambda: fq.mxfp4_quantize_rows(x))
    run(lambda: fq.fp4_to_fp8_rows(q, s, 0))
    run(lambda: fq.fp4_to_fp8_rows(q, s, 6))

    x = dev_bf16(workloads.moe_dispatch(16384, 7168, seed=0))
    o = offs_dev(workloads.zipf_group_offsets(16384, 32, 1.1, 0))
    q, s = run(lambda: fq.mxfp4_quantize_rows(x))
    run(lambda: fq.fp4_to_fp8_rows(q, s, 0))
    run(lambda: fq.fp4_to_fp8_cols(q, s, o, 0))
    amax = run(lambda: fq.nvfp4_amax(x))
    run(lambda: fq.nvfp4_quantize(x, amax, use_sr=True, seed=1234))
    run(lambda: fq.nvfp4_quantize_2d(x, amax))

    bits, offs = workloads.ragged_experts(65536, 2048, 32, seed=0)
    x = dev_bf16(bits)
    q, s = run(lambda: fq.mxfp4_quantize_rows(x))
    run(lambda: fq.fp4_to_fp8_cols(q, s, offs_dev(offs), 0))

    x = dev_bf16(workloads.nvfp4_act(16384, 14336, seed=0))
    amax = run(lambda: fq.nvfp4_amax(x))
    run(lambda: fq.nvfp4_quantize(x, amax, use_sr=True, seed=1234))
    run(lambda: fq.nvfp4_quantize(x, amax))
    w = dev_bf16(workloads.nvfp4_weight(14336, 4096, seed=0))
    wamax = run(lambda: fq.nvfp4_amax(w))
    run(lambda: fq.nvfp4_quantize_2d(w, wamax))

    del x, q, s, w
    big = workloads.sweep(PROFILE_SWEEP[-1], 7168, seed=0)
    xb = dev_bf16(big)
    del big
    for m in PROFILE_SWEEP:
        xm = xb[:m]
        q, s = run(lambda: fq.mxfp4_quantize_rows(xm))
        run(lambda: fq.fp4_to_fp8_rows(q, s, 0))
        run(lambda: fq.fp4_to_fp8_cols(q, s, offs_dev([0, m]), 0))
        del q, s
        torch.cuda.empty_cache()
    torch.cuda.synchronize()
    print(json.dumps({"profile_configs": len(PROFILE_ORDER)}), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["fq", "reference"], default="fq")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile-configs", action="store_true",
                    help="run every configuration's calls once (for an ncu capture) and exit")
    ap.add_argument("--sweep-rows", type=int, default=0,
                    help="run the bandwidth-sweep chain at this many rows once (for an ncu "
                         "capture of one size) and exit")
    args = ap.parse_args()
    if args.profile_configs:
        return run_profile_configs()
    if args.sweep_rows:
        return run_sweep_rows(args.sweep_rows)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
