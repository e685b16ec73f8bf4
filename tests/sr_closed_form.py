"""Inputs and closed-form expectations for the statistical tests of NVFP4
stochastic rounding, on the device and on the oracle.

The NVFP4 page ("Train models faster with JAX and MaxText using NVFP4 on
NVIDIA Blackwell", section "Receta de pre-entrenamiento NVFP4", item
"Redondeo estocástico") asks for unbiased rounding and says it is native to
Blackwell's FP4 conversion instructions.  The closed form checked here: a
magnitude y with lo <= y < hi on the E2M1 grid {0, 0.5, 1, 1.5, 2, 3, 4, 6}
rounds up with probability floor(2^16 (y - lo) / (hi - lo)) / 2^16 when the
element's 16 random bits are uniform; y >= 6 gives 6.  So wherever
2^16 (y - lo) / (hi - lo) is an integer the expected decoded value is y
itself.  Nothing here uses the mapping of Philox words to elements: a wrong
mapping that left some position's bits non-uniform (or a wrong rounding rule)
moves that position's up-rate away from the closed form.

Test tensors hold blocks of 16 values whose block maximum sits at position
(block index mod 16) and whose other 15 values all share one magnitude (the
block's "type"), so every position of a block is measured for every type.
Per-tensor amax values are chosen so that the block scale arithmetic (the
library's binary32 rule: g = A / 2688, enc = 1 / (6 g), t = amax_blk * enc,
b = E4M3(t), r = 1 / (b g), y = |x| r) gives:

* setup "pow2": A = 2688 (g = 1), block maximum 1536 (b = 256), r = 2^-8
  exactly, so y = |x| / 256 and fractions such as 2^-16, 1/4, 1/2, 7/8 are
  hit exactly;
* setup "near1": A = 2688 (1 + 2^-16) (g = 1 + 2^-16), block maximum 768
  (b = 128), r = 2^-7 (1 - 2^-16): y = 64 r = (1 - 2^-16) / 2 sits at
  fraction 1 - 2^-16 of [0, 0.5].

For the random Hadamard transform variant the tensor is built so that the
transform of each block is exactly such a block: x = 1/4 diag(d) H16 z
(H16 H16 = 16 I and d_i = +-1), with z small integers so that x is exact in
BF16 and every butterfly sum is exact in binary32.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np
import torch

GRID = [Fraction(0), Fraction(1, 2), Fraction(1), Fraction(3, 2), Fraction(2), Fraction(3),
        Fraction(4), Fraction(6)]

SETUPS = {
    # name: (A, block maximum, magnitudes of the other 15 values)
    "pow2": (2688.0, 1536.0, [2.0 ** -9, 64.0, 320.0, 576.0, 1472.0]),
    "near1": (None, 768.0, [64.0, 192.0]),
}
# Magnitudes whose transformed block stays exact in BF16 (x_0 = 4 v + (max - v) / 4
# needs at most 8 significant bits).
RHT_SETUPS = {
    "pow2": (2688.0, 1536.0, [64.0, 320.0, 576.0, 1408.0]),
    "near1": (None, 768.0, [64.0, 192.0]),
}


def f32(v):
    return np.float32(v)


def setup_amax(name: str) -> np.float32:
    if name == "pow2":
        return f32(2688.0)
    # A with fl(A / 2688) = 1 + 2^-16 (checked by the caller via scale_chain)
    return f32(np.float32(2688.0) * np.float32(1.0 + 2.0 ** -16))


def e4m3_byte(t: np.float32) -> int:
    """E4M3 byte of a non-negative binary32 value (torch's float8_e4m3fn cast:
    round to nearest even; finite here)."""
    return int(torch.tensor([float(t)], dtype=torch.float32).to(torch.float8_e4m3fn)
               .view(torch.uint8).item())


def e4m3_value(b: int) -> np.float32:
    return np.float32(torch.tensor([b], dtype=torch.uint8).view(torch.float8_e4m3fn)
                      .to(torch.float32).item())


def scale_chain(A: np.float32, amax_blk: np.float32):
    """(g, block-scale byte b, r) in binary32, one rounding per operation."""
    g = f32(A) / f32(2688.0) if A > 0 else f32(1.0)
    enc = f32(1.0) / (f32(6.0) * g)
    t = f32(amax_blk) * enc
    b = e4m3_byte(t)
    r = f32(1.0) / (e4m3_value(b) * g)
    return g, b, r


def closed_form(y: np.float32):
    """(lo code, hi code, P(up) as a Fraction, E[decoded] as a Fraction) for
    magnitude y >= 0."""
    fy = Fraction(float(y))
    if fy >= 6:
        return 7, 7, Fraction(0), Fraction(6)
    lo = max(i for i in range(8) if GRID[i] <= fy)
    frac = (fy - GRID[lo]) / (GRID[lo + 1] - GRID[lo])
    p = Fraction(int(frac * 65536), 65536)   # floor for a non-negative value
    return lo, lo + 1, p, GRID[lo] + p * (GRID[lo + 1] - GRID[lo])


def h16() -> np.ndarray:
    i = np.arange(16)
    return np.array([[(-1) ** bin(a & b).count("1") for b in i] for a in i], dtype=np.float64)


def build(setup: str, nblocks: int, rht_mask: int | None = None, K: int = 4096):
    """Test tensor and expectations.

    Returns a dict with: bits (BF16 bit patterns [M, K]), A (per-tensor amax
    to pass), g, b (expected block-scale byte, the same for every block),
    etype [M, K] (type index of each element, -1 for the block maxima),
    epos [M, K] (position in the block), and types: a list of
    (magnitude y, lo code, hi code, P(up), E[decoded]) per type, the last
    entry being the block maxima."""
    table = RHT_SETUPS if rht_mask is not None else SETUPS
    _, vmax, mags = table[setup]
    A = setup_amax(setup)
    g, b, r = scale_chain(A, f32(vmax))
    assert nblocks % 16 == 0 and (nblocks * 16) % K == 0
    nt = len(mags)
    blk = np.arange(nblocks)
    pmax = blk % 16
    tix = (blk // 16) % nt
    z = np.empty((nblocks, 16), dtype=np.float64)
    z[:] = np.asarray(mags, dtype=np.float64)[tix][:, None]
    z[blk, pmax] = vmax
    etype = np.repeat(tix[:, None], 16, axis=1)
    etype[blk, pmax] = -1
    epos = np.broadcast_to(np.arange(16), (nblocks, 16)).copy()
    # signs: negative where (position + block) is odd -- the sign is kept,
    # so only magnitudes are rounded
    sign = np.where((epos + blk[:, None]) % 2 == 1, -1.0, 1.0)
    if rht_mask is None:
        x = z * sign
    else:
        # the transform of x is z exactly: x = 1/4 diag(d) H z (signs of z
        # stay positive here; the RHT's output signs are what they are)
        d = np.array([-1.0 if (rht_mask >> i) & 1 else 1.0 for i in range(16)])
        x = 0.25 * (h16() @ z.T).T * d
    xf = x.astype(np.float32)
    assert np.array_equal(xf.astype(np.float64), x), "inputs must be exact in binary32"
    bits = (xf.view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal(((bits.astype(np.uint32) << 16).view(np.float32)).astype(np.float64),
                          x), "inputs must be exact in BF16"
    types = []
    for v in list(mags) + [vmax]:
        y = f32(v) * r
        types.append((y,) + closed_form(y))
    return {"bits": bits.reshape(-1, K), "A": A, "g": g, "b": b,
            "etype": etype.reshape(-1, K), "epos": epos.reshape(-1, K), "types": types}


def check_counts(ups: np.ndarray, trials: np.ndarray, probs, what: str, z: float = 4.0):
    """Binomial check of up counts against P(up) per (type, position)."""
    for ti, p in enumerate(probs):
        pf = float(p)
        for pos in range(16):
            n = int(trials[ti, pos])
            if n == 0:
                continue
            k = int(ups[ti, pos])
            mean, sd = n * pf, np.sqrt(n * pf * (1 - pf))
            assert abs(k - mean) <= z * sd + 1.0, (
                f"{what}: type {ti} position {pos}: {k} ups in {n} trials, expected "
                f"{mean:.1f} +- {sd:.1f} (P = {p})")
