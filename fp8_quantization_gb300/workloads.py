"""Seeded synthetic inputs for the cast kernels.

This module only draws random numbers and rounds them to BF16; it holds none
of the quantisation arithmetic, so both the CUDA path's tests/bench and the
CPU oracle's tests can use it.  Each generator states the value distribution
and shape of the workload it stands in for:

* ``pr1``            256x512 N(0,1), 0.1% of entries scaled by 100 (outliers).
* ``moe_dispatch``   MoE dispatch activations of a 671B-class model
                     (hidden 7168): N(0,1) rows times a per-row log-normal(0,1)
                     magnitude.
* ``ragged_experts`` routed rows of width 2048 over 32 local experts, expert
                     sizes drawn Zipf(s=1.1) (group offsets, no padding).
* ``nvfp4_act``      Student-t(nu=4) activations (MLP width 14336).
* ``nvfp4_weight``   N(0, 0.02) weights 14336x4096.
* ``sweep``          Student-t(nu=3) rows x 7168 for the bandwidth sweep.

All arrays are returned as BF16 bit patterns (``numpy.uint16``), row-major.
BF16 rounding is round-to-nearest-even, done by ``torch`` on the host.  Every
generator but ``pr1`` draws blocks of rows (about 4M elements each) from
child seeds of one seed, in parallel threads, so that the largest tensors
take seconds; a block's values do not depend on the row count, so a smaller
tensor is a prefix of a larger one drawn with the same seed.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """float32 array -> BF16 bit patterns (round to nearest even)."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bits_to_float(bits: np.ndarray) -> np.ndarray:
    """BF16 bit patterns -> float32 values (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def pr1(M: int = 256, K: int = 512, seed: int = 0) -> np.ndarray:
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((M, K))
    mask = rng.random((M, K)) < 1e-3
    x[mask] *= 100.0
    return bf16_bits(x.astype(np.float32))


def moe_dispatch(M: int = 16384, K: int = 7168, seed: int = 0) -> np.ndarray:
    def draw(rng, shape):
        x = rng.standard_normal(shape, dtype=np.float32)
        x *= rng.lognormal(0.0, 1.0, (shape[0], 1)).astype(np.float32)
        return x
    return _bf16_row_blocks(M, K, seed, draw)


def zipf_group_offsets(M: int, G: int = 32, s: float = 1.1, seed: int = 0) -> np.ndarray:
    """Exclusive prefix sum of per-expert token counts; expert e has Zipf rank
    e+1, i.e. probability proportional to (e+1)^-s.  Returns int64 [G+1]."""
    rng = np.random.default_rng(seed + 1)
    p = np.arange(1, G + 1, dtype=np.float64) ** (-s)
    p /= p.sum()
    ids = rng.choice(G, size=M, p=p)
    counts = np.bincount(ids, minlength=G).astype(np.int64)
    return np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)


def ragged_experts(M: int = 65536, K: int = 2048, G: int = 32, seed: int = 0):
    x = _bf16_row_blocks(M, K, seed, lambda rng, shape: rng.standard_normal(shape, dtype=np.float32))
    return x, zipf_group_offsets(M, G, 1.1, seed)


def _bf16_row_blocks(M: int, K: int, seed: int, draw) -> np.ndarray:
    """BF16 bits [M, K]; rows c*R .. (c+1)*R - 1 (R rows of about 4M
    elements) are draw(rng, shape) with rng seeded by the c-th child of
    SeedSequence(seed).  A block's values do not depend on M."""
    R = max(1, (1 << 22) // max(K, 1))
    n = max(1, -(-M // R))
    kids = np.random.SeedSequence(seed).spawn(n)
    out = np.empty((M, K), dtype=np.uint16)

    def work(c):
        r0, r1 = c * R, min(M, (c + 1) * R)
        if r1 > r0:
            rng = np.random.default_rng(kids[c])
            out[r0:r1] = bf16_bits(draw(rng, (r1 - r0, K)).astype(np.float32))

    with ThreadPoolExecutor(max(1, min(n, os.cpu_count() or 1))) as ex:
        list(ex.map(work, range(n)))
    return out


def nvfp4_act(M: int = 16384, K: int = 14336, seed: int = 0) -> np.ndarray:
    return _bf16_row_blocks(M, K, seed, lambda rng, shape: rng.standard_t(4, shape))


def nvfp4_weight(N: int = 14336, K: int = 4096, seed: int = 0) -> np.ndarray:
    return _bf16_row_blocks(N, K, seed, lambda rng, shape: rng.normal(0.0, 0.02, shape))


def sweep(M: int, K: int = 7168, seed: int = 0) -> np.ndarray:
    return _bf16_row_blocks(M, K, seed, lambda rng, shape: rng.standard_t(3, shape))


def random_group_offsets(M: int, G: int, seed: int = 0, empty_frac: float = 0.2) -> np.ndarray:
    """Arbitrary ragged split of M rows into G groups (some empty), for edge
    cases: sizes are unrelated to 128 so group starts are misaligned."""
    rng = np.random.default_rng(seed)
    w = rng.random(G)
    w[rng.random(G) < empty_frac] = 0.0
    if w.sum() == 0:
        w[0] = 1.0
    counts = np.floor(w / w.sum() * M).astype(np.int64)
    counts[int(np.argmax(w))] += M - counts.sum()
    return np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
