"""Pins of the oracle's BF16 -> FP8 E4M3 block quantizer (1x128 and 128x128)
and of its MXFP4 -> BF16 dequantizer.

Reading of the quantizer (the pages fix the format, E4M3 with 128-element
blocks and FP32 scales, not the scale rule): per block r = min(448 / amax,
FLT_MAX), s = amax / 448 (binary32), code = E4M3_RNE_satfinite(x r); NaN or Inf
in a block -> s = NaN, codes 0x7F.  The dequantizer is exact: BF16(v 2^(e-127)),
infinity on overflow, NaN for scale 0xFF."""
import numpy as np
import pytest
import torch

import oracle
from fp8_quantization_gb300 import workloads


def bf16(a):
    return workloads.bits_to_float(workloads.bf16_bits(np.asarray(a, dtype=np.float32)))


def torch_bf16_bits(v64):
    """float64 values exactly representable in float32 -> BF16 bits (torch RNE)."""
    t = torch.from_numpy(np.asarray(v64, dtype=np.float64).astype(np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def test_bf16_rounding_helper_matches_torch():
    rng = np.random.default_rng(0)
    f = (rng.standard_normal(20000) * np.exp2(rng.integers(-140, 126, 20000))).astype(np.float32)
    assert np.array_equal(oracle.bf16_rne(f.astype(np.float64)), torch_bf16_bits(f))
    top = np.ldexp(2.0 - 2.0 ** -7, 127)                      # largest finite BF16
    mid = np.ldexp(2.0 - 2.0 ** -8, 127)                      # midpoint to 2^128
    got = oracle.bf16_rne(np.array([top, mid, -mid, np.nextafter(mid, 0), 2.0 ** -133,
                                    2.0 ** -134, 3 * 2.0 ** -134, -0.0]))
    assert got.tolist() == [0x7F7F, 0x7F80, 0xFF80, 0x7F7F, 0x0001, 0x0000, 0x0002, 0x8000]


def test_dequantize_every_code_and_scale():
    """All 256 code bytes (two codes each) under all 256 scale bytes against
    an independent float64 computation rounded by torch."""
    mags = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    q = np.tile(np.arange(256, dtype=np.uint8), (256, 1))    # [256 scales, 256 bytes] -> K = 512
    q = np.repeat(q, 1, axis=0)
    s = np.repeat(np.arange(256, dtype=np.uint8)[:, None], 512 // 32, axis=1)
    out = oracle.mxfp4_dequantize_rows(q, s)
    codes = np.stack([q & 0xF, q >> 4], axis=-1).reshape(256, 512)
    val = np.where(codes & 8, -1.0, 1.0) * mags[codes & 7] * np.exp2(np.arange(256)[:, None] - 127.0)
    with np.errstate(over="ignore"):
        want = torch_bf16_bits(val)  # exact or overflow -> inf (float32 overflow, then inf)
    want[255] = 0x7FC0
    assert np.array_equal(out, want)


def identity_block_values(rng, n):
    """E4M3-representable BF16 values with |max| exactly 448 (so r = s = 1)."""
    codes = rng.integers(0, 0x7F, n)
    codes[codes == 0x7F] = 0
    vals = np.array([oracle.e4m3_magnitude(int(c)) for c in codes]) * rng.choice([-1, 1], n)
    vals[rng.integers(0, n)] = 448.0 * rng.choice([-1, 1])
    return vals.astype(np.float32)


def test_identity_blocks_give_the_e4m3_codes():
    rng = np.random.default_rng(1)
    x = identity_block_values(rng, 4 * 256).reshape(4, 256)
    for h in range(2):
        x[:, 128 * h + 3] = 448.0
    y, sc = oracle.fp8_quantize_blocks(workloads.bf16_bits(x), 1)
    assert np.all(sc == 1.0)
    want = (oracle.e4m3_rne(np.abs(x)).reshape(x.shape).astype(np.uint8) |
            np.where(np.signbit(x), 0x80, 0).astype(np.uint8))
    assert np.array_equal(y, want)


@pytest.mark.parametrize("block_rows", [1, 128])
def test_error_bound_and_block_max(block_rows):
    rng = np.random.default_rng(2)
    M, K = 256, 384
    x = bf16(rng.standard_normal((M, K)) * np.exp2(rng.integers(-30, 30, (M, 1))))
    y, sc = oracle.fp8_quantize_blocks(workloads.bf16_bits(x), block_rows)
    dec = oracle.e4m3_decode(y).astype(np.float64)
    s_full = np.repeat(np.repeat(sc.astype(np.float64), block_rows, axis=0), 128, axis=1)
    approx = dec * s_full
    blk = np.abs(x).reshape(M // block_rows, block_rows, K // 128, 128).max(axis=(1, 3))
    assert np.array_equal(sc, (blk / np.float32(448.0)).astype(np.float32))
    # E4M3: 3 mantissa bits -> relative error <= 2^-4 in the normal range, and
    # absolute <= 2^-10 s below it; plus the binary32 roundings of r and s
    tol = np.maximum(np.abs(x) * (2.0 ** -4 + 2.0 ** -20), s_full * (2.0 ** -10 + 2.0 ** -20))
    assert np.all(np.abs(approx - x) <= tol)
    # the element holding the block max encodes +-448
    mx = np.abs(x).reshape(M // block_rows, block_rows, K // 128, 128)
    codes = y.reshape(M // block_rows, block_rows, K // 128, 128)
    hit = mx == blk[:, None, :, None]
    assert np.all(codes[hit] & 0x7F == 0x7E)


def test_special_blocks():
    x = np.ones((2, 512), dtype=np.float32)
    x[0, :128] = 0.0
    x[0, 128:256] = -0.0
    x[0, 300] = np.nan
    x[1, 10] = np.inf
    x[1, 400] = -np.inf
    x[1, 128:256] = np.float32(2.0 ** -130)  # BF16 subnormals: r saturates at FLT_MAX
    y, sc = oracle.fp8_quantize_blocks(workloads.bf16_bits(x), 1)
    assert np.all(y[0, :128] == 0) and sc[0, 0] == 0.0
    assert np.all(y[0, 128:256] == 0x80) and sc[0, 1] == 0.0
    assert np.all(y[0, 256:384] == 0x7F) and np.isnan(sc[0, 2])
    assert np.all(y[1, :128] == 0x7F) and np.isnan(sc[1, 0])
    assert np.all(y[1, 384:] == 0x7F) and np.isnan(sc[1, 3])
    with np.errstate(over="ignore"):
        assert not np.isfinite(np.float32(448.0) / np.float32(2.0 ** -130))  # r saturates
    want = oracle.e4m3_rne(np.array([np.float32(2.0 ** -130) * np.finfo(np.float32).max]))[0]
    assert np.all(y[1, 128:256] == want) and sc[1, 1] == np.float32(2.0 ** -130) / np.float32(448)


def test_tiles_use_the_tile_max():
    rng = np.random.default_rng(3)
    x = bf16(rng.standard_normal((256, 256)))
    x[5, 7] = 1000.0  # tile (0, 0) max
    y1, s1 = oracle.fp8_quantize_blocks(workloads.bf16_bits(x), 1)
    y2, s2 = oracle.fp8_quantize_blocks(workloads.bf16_bits(x), 128)
    assert s2.shape == (2, 2) and s2[0, 0] == np.float32(1000.0) / np.float32(448.0)
    assert s1[5, 0] == s2[0, 0] and s1[6, 0] < s2[0, 0]
    # rows of tile (0, 0) other than row 5 quantize coarser than with row blocks
    assert not np.array_equal(y1[:128, :128], y2[:128, :128])
    assert np.array_equal(y1[5, :128], y2[5, :128])
