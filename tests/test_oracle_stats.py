"""The oracle's statistics functions (dequantization error per block, and the
exact / rounded / flushed classification of the FP4 -> FP8 conversion)
checked against the same numbers computed another way: numpy decoding of the
quantizers' outputs, and decoding of the actual FP8 conversion outputs."""
import numpy as np
import pytest

from fp8_quantization_gb300 import workloads


def f64(bits):
    return workloads.bits_to_float(bits).astype(np.float64)


def per_block_ratio(x, xhat, rows, cols):
    M, K = x.shape
    err = np.abs(x - xhat).reshape(M // rows, rows, K // cols, cols).max(axis=(1, 3))
    amax = np.abs(x).reshape(M // rows, rows, K // cols, cols).max(axis=(1, 3))
    return err, amax


@pytest.mark.parametrize("seed", [0, 1])
def test_mxfp4_error_stats(oracle_mod, seed):
    bits = workloads.pr1(64, 256, seed=seed)
    bits[0, :32] = 0                      # an all-zero block is not counted
    bits[1, 5] = 0x7FC0                   # nor is a NaN block
    q, s = oracle_mod.mxfp4_quantize_rows(bits)
    st = oracle_mod.mxfp4_error_stats(bits, q, s)
    x = f64(bits)
    scale = np.repeat(2.0 ** (s.astype(np.float64) - 127), 32, axis=1)
    xhat = oracle_mod.e2m1_decode(oracle_mod.unpack_nibbles(q)) * scale
    err, amax = per_block_ratio(np.nan_to_num(x), xhat, 1, 32)
    keep = (s != 0xFF) & (amax > 0)
    ratio = err[keep] / amax[keep]
    assert st["blocks"] == keep.sum() == 64 * 8 - 2
    assert st["max_ratio"] == ratio.max()
    assert np.isclose(st["mean_ratio"], ratio.mean(), rtol=1e-12)
    assert st["over_bound"] == 0 and st["max_ratio"] <= 0.25


@pytest.mark.parametrize("tile_rows", [1, 16])
def test_nvfp4_error_stats(oracle_mod, tile_rows):
    bits = workloads.nvfp4_act(64, 256, seed=3)
    bits[2, :16] = 0x0001                 # a tiny block: subnormal or zero scale byte
    A = oracle_mod.nvfp4_amax(bits)
    if tile_rows == 1:
        q, sb, g = oracle_mod.nvfp4_quantize(bits, A)
    else:
        q, sb, g = oracle_mod.nvfp4_quantize_2d(bits, A)
    st = oracle_mod.nvfp4_error_stats(bits, q, sb, g, tile_rows)
    x = f64(bits)
    scale = np.repeat(np.repeat(oracle_mod.e4m3_decode(sb) * float(g), tile_rows, axis=0), 16,
                      axis=1)
    xhat = oracle_mod.e2m1_decode(oracle_mod.unpack_nibbles(q)) * scale
    err, amax = per_block_ratio(x, xhat, tile_rows, 16)
    normal = (sb & 0x78) != 0
    keep = normal & (amax > 0)
    assert st["blocks"] == keep.sum()
    assert st["max_ratio"] == (err[keep] / amax[keep]).max()
    assert np.isclose(st["mean_ratio"], (err[keep] / amax[keep]).mean(), rtol=1e-12)
    small = ~normal & (amax > 0)
    assert st["small_scale_blocks"] == small.sum() and (tile_rows == 16 or small.sum() >= 1)


def classify_from_outputs(oracle_mod, q, s, y, ys_elem):
    """exact / rounded / flushed / zero counts from decoded conversion outputs."""
    v = oracle_mod.e2m1_decode(oracle_mod.unpack_nibbles(q)) * \
        np.repeat(2.0 ** (s.astype(np.float64) - 127), 32, axis=1)
    w = oracle_mod.e4m3_decode(y) * ys_elem
    nz = v != 0
    return {"exact": int((nz & (w == v)).sum()), "rounded": int((nz & (w != v) & (w != 0)).sum()),
            "flushed": int((nz & (w == 0)).sum()), "zero": int((~nz).sum()), "nan_block": 0}


@pytest.mark.parametrize("k", [0, 6])
def test_fp4_to_fp8_counts_rows_and_cols(oracle_mod, k):
    rng = np.random.default_rng(5)
    M, K = 200, 256
    q = rng.integers(0, 256, (M, K // 2), dtype=np.uint8)
    s = (100 + rng.integers(0, 24, (M, K // 32))).astype(np.uint8)   # shifts up to 23: flushes
    y, ys = oracle_mod.fp4_to_fp8_rows(q, s, k)
    want = classify_from_outputs(oracle_mod, q, s, y, np.repeat(ys.astype(np.float64), 128, axis=1))
    got = oracle_mod.fp4_to_fp8_counts(q, s, k)
    assert got == want
    assert got["rounded"] > 0 and got["flushed"] > 0
    offs = np.array([0, 60, 60, 200], dtype=np.int64)
    yT, yTs = oracle_mod.fp4_to_fp8_cols(q, s, offs, k)
    # the scale of element (feature f, token t) is row (block of t) of yTs
    blk = np.empty(M, dtype=np.int64)
    base = 0
    for g in range(3):
        c = offs[g + 1] - offs[g]
        blk[offs[g]:offs[g + 1]] = base + np.arange(c) // 128
        base += (c + 127) // 128
    sc = yTs[blk].astype(np.float64)                     # [M, K]
    want = classify_from_outputs(oracle_mod, q, s, np.ascontiguousarray(yT.T), sc)
    assert oracle_mod.fp4_to_fp8_counts(q, s, k, offs) == want


def test_fp4_to_fp8_counts_nan_blocks(oracle_mod):
    q = np.full((2, 64), 0x33, dtype=np.uint8)
    s = np.full((2, 4), 120, dtype=np.uint8)
    s[1, 2] = 0xFF
    got = oracle_mod.fp4_to_fp8_counts(q, s, 0)
    assert got == {"exact": 128, "rounded": 0, "flushed": 0, "zero": 0, "nan_block": 128}
