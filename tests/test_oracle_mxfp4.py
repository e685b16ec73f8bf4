"""Pins of the oracle's MXFP4 row quantization (BF16ToFP4Row) and of the
direct FP4->FP8 conversions (FP4RowToFP8Row / FP4RowToFP8Col).

Sources: "Practical FP4 Training for Large-Scale MoE Models on Hopper GPUs",
technical overview section 2: 32-element blocks with a UE8M0 power-of-two
scale and E2M1 elements; direct bitwise FP4->FP8 conversion that maps four MX
blocks onto one 128-element E4M3 block by aligning exponents to the largest
scale, which keeps the numbers equivalent; transposed conversion for Wgrad and
ragged per-expert groups without padding."""
from fractions import Fraction

import numpy as np
import pytest

from fp8_quantization_gb300 import workloads

ml_dtypes = pytest.importorskip("ml_dtypes")


def f32(bits):
    return workloads.bits_to_float(bits)


def special_tensor(M=16, K=128, seed=3):
    """Tiny tensor with zero blocks, signed zeros, BF16 subnormals, huge
    values, exact E2M1 ties after scaling, and ordinary values."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((M, K)).astype(np.float32)
    x[0, :32] = 0.0
    x[0, 32:64] = -0.0
    x[1, :32] = np.float32(2.0 ** -130) * rng.integers(1, 127, 32)      # subnormal bf16
    x[2, :32] = np.float32(3.0e38) * rng.standard_normal(32).clip(-1, 1)
    x[3, :32] = np.float32(4.0) * np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0] * 4)
    x[3, 31] = 7.0   # amax in [4,8): scale exponent stays 127 + 0
    x[4, :32] = np.float32(2.0 ** -120)
    bits = workloads.bf16_bits(x)
    return bits


def test_mxfp4_brute_force_tiny(oracle_mod):
    bits = special_tensor()
    q, s = oracle_mod.mxfp4_quantize_rows(bits)
    codes = oracle_mod.unpack_nibbles(q)
    x = f32(bits).astype(np.float64)
    M, K = x.shape
    grid = np.array([oracle_mod.e2m1_magnitude(c) for c in range(8)])
    for r in range(M):
        for j in range(K // 32):
            xb = x[r, 32 * j:32 * j + 32]
            e = int(s[r, j])
            amax = np.abs(xb).max()
            # closed form of the scale rule
            if amax == 0:
                assert e == 0
            elif e > 0:
                assert 4.0 <= amax * 2.0 ** (127 - e) < 8.0
            scale = 2.0 ** (e - 127)
            for i in range(32):
                # exhaustive search over the 8 magnitudes, ties to even code
                d = [abs(abs(xb[i]) - g * scale) for g in grid]
                best = min(d)
                cands = [c for c in range(8) if d[c] == best]
                c = min(cands, key=lambda c: (c % 2, c))
                c |= 8 if np.signbit(xb[i]) else 0
                assert codes[r, 32 * j + i] == c, (r, j, i, xb[i], e)


def test_mxfp4_matches_library_cast_after_scaling(oracle_mod):
    bits = workloads.pr1(64, 512, seed=4)
    q, s = oracle_mod.mxfp4_quantize_rows(bits)
    x = f32(bits).reshape(64, 16, 32).astype(np.float64)
    scaled = (x * 2.0 ** (127 - s.astype(np.float64))[:, :, None]).astype(np.float32)
    lib = scaled.astype(ml_dtypes.float4_e2m1fn).view(np.uint8).reshape(64, 512) & 0xF
    np.testing.assert_array_equal(oracle_mod.unpack_nibbles(q), lib)


def test_mxfp4_error_bound_pr1(oracle_mod):
    # |x - xhat| <= amax_blk / 4 for every element (grid half-gap at most 1 in
    # the top binade and saturation loss below 2, over amax >= 4 after scaling)
    bits = workloads.pr1()
    q, s = oracle_mod.mxfp4_quantize_rows(bits)
    x = f32(bits).astype(np.float64).reshape(256, 16, 32)
    xhat = oracle_mod.e2m1_decode(oracle_mod.unpack_nibbles(q)).reshape(256, 16, 32)
    xhat = xhat * 2.0 ** (s.astype(np.float64) - 127)[:, :, None]
    amax = np.abs(x).max(axis=2, keepdims=True)
    err = np.abs(x - xhat)
    assert np.all(err <= amax / 4)
    ratio = (err / np.where(amax > 0, amax, 1)).max()
    assert ratio <= 0.25
    print(f"max |x - xhat| / amax_blk over PR1 = {ratio:.4f}")


def test_mxfp4_nonfinite_block(oracle_mod):
    x = np.zeros((2, 64), dtype=np.float32)
    x[0, 5] = np.nan
    x[1, 40] = -np.inf
    x[1, :32] = 1.0
    q, s = oracle_mod.mxfp4_quantize_rows(workloads.bf16_bits(x))
    assert s.tolist() == [[0xFF, 0], [127 - 2, 0xFF]]
    codes = oracle_mod.unpack_nibbles(q)
    assert np.all(codes[0, :32] == 0) and np.all(codes[1, 32:] == 0)


def test_mxfp4_packing_order(oracle_mod):
    x = np.zeros((1, 32), dtype=np.float32)
    x[0, 0] = 1.0   # amax 6 gives e = 127 (scale 1): code 2
    x[0, 1] = -6.0
    q, s = oracle_mod.mxfp4_quantize_rows(workloads.bf16_bits(x))
    assert s[0, 0] == 127
    assert q[0, 0] == (2 | (0xF << 4))  # element 0 low nibble, element 1 high nibble


# ------------------------------------------------------------------ FP4 -> FP8

def e4m3_exact_table():
    """All finite E4M3 magnitudes as exact Fractions, by code."""
    out = []
    for c in range(127):
        E, m = c >> 3, c & 7
        out.append(Fraction(m, 512) if E == 0 else Fraction(8 + m, 8) * Fraction(2) ** (E - 7))
    return out


def test_fp4_to_fp8_element_map_exhaustive(oracle_mod):
    # 16 codes x every shift d in [0, 254] x every offset k in [0, 6] against
    # an exact rational nearest-value search (ties to even code, saturate).
    table = e4m3_exact_table()
    grid = [Fraction(0), Fraction(1, 2), Fraction(1), Fraction(3, 2), Fraction(2), Fraction(3),
            Fraction(4), Fraction(6)]
    codes = np.repeat(np.arange(16, dtype=np.uint8), 255)
    d = np.tile(np.arange(255, dtype=np.int32), 16)
    for k in range(7):
        got = oracle_mod.fp4_to_fp8_element(codes, d, k)
        for idx in range(codes.size):
            c, dd = int(codes[idx]), int(d[idx])
            v = grid[c & 7] * Fraction(2) ** (k - dd)
            if v >= 448:
                want = 0x7E
            elif v == 0 or v < Fraction(1, 2048):
                want = 0
            else:
                dist = [abs(v - t) for t in table]
                best = min(dist)
                cands = [i for i in range(127) if dist[i] == best]
                want = min(cands, key=lambda i: (i % 2, i))
            want |= 0x80 if c & 8 else 0
            assert got[idx] == want, (c, dd, k, got[idx], want)


def test_fp4_to_fp8_equivalence_invariant(oracle_mod):
    # The alignment keeps dequantised values identical wherever the shifted
    # value is representable: for every code, d <= k + 8 is exact.
    codes = np.repeat(np.arange(16, dtype=np.uint8), 40)
    d = np.tile(np.arange(40, dtype=np.int32), 16)
    for k in range(7):
        y = oracle_mod.fp4_to_fp8_element(codes, d, k)
        v4 = oracle_mod.e2m1_decode(codes) * 2.0 ** (k - d.astype(np.float64))
        v8 = oracle_mod.e4m3_decode(y)
        exact = d <= k + 8
        np.testing.assert_array_equal(v8[exact], v4[exact])
        assert np.all(np.signbit(v8) == np.signbit(v4))


def test_fp4_to_fp8_rows_structure_pr1(oracle_mod):
    bits = workloads.pr1()
    q, s = oracle_mod.mxfp4_quantize_rows(bits)
    for k in (0, 6):
        y, ys = oracle_mod.fp4_to_fp8_rows(q, s, k)
        S = s.reshape(256, 4, 4).max(axis=2).astype(np.float64)
        np.testing.assert_array_equal(ys.astype(np.float64), 2.0 ** (S - 127 - k))
        # dequantised FP8 equals dequantised FP4 wherever d <= k + 8
        v4 = oracle_mod.e2m1_decode(oracle_mod.unpack_nibbles(q)) * \
            np.repeat(2.0 ** (s.astype(np.float64) - 127), 32, axis=1)
        v8 = oracle_mod.e4m3_decode(y) * np.repeat(ys.astype(np.float64), 128, axis=1)
        d = np.repeat(np.repeat(S, 4, axis=1) - s, 32, axis=1)
        ok = d <= k + 8
        np.testing.assert_array_equal(v8[ok], v4[ok])
        print(f"k={k}: {int((~ok).sum())} of {ok.size} elements beyond the exact range")


def test_fp4_to_fp8_rows_equal_scales_is_value_cast(oracle_mod):
    # With all four MX exponents equal and k = 0 every E2M1 value is
    # representable in E4M3, so the FP8 code is the library's cast of it.
    rng = np.random.default_rng(9)
    codes = rng.integers(0, 16, (8, 256), dtype=np.uint8)
    q = oracle_mod.pack_nibbles(codes)
    s = np.full((8, 8), 120, dtype=np.uint8)
    y, ys = oracle_mod.fp4_to_fp8_rows(q, s, 0)
    vals = oracle_mod.e2m1_decode(codes).astype(np.float32)
    np.testing.assert_array_equal(y, vals.astype(ml_dtypes.float8_e4m3fn).view(np.uint8))
    assert np.all(ys == np.float32(2.0 ** (120 - 127)))


def test_fp4_to_fp8_rows_nan_block(oracle_mod):
    rng = np.random.default_rng(2)
    q = rng.integers(0, 256, (2, 128), dtype=np.uint8)
    s = np.full((2, 8), 100, dtype=np.uint8)
    s[1, 6] = 0xFF
    y, ys = oracle_mod.fp4_to_fp8_rows(q, s, 0)
    assert np.all(y[1, 128:] == 0x7F) and np.isnan(ys[1, 1])
    assert ys.view(np.uint32)[1, 1] == 0x7FC00000
    assert not np.any(np.isnan(ys[0])) and not np.isnan(ys[1, 0])


# ------------------------------------------------------------------ transposed, ragged

def rand_mx(M, K, seed, lo=100, hi=140):
    rng = np.random.default_rng(seed)
    q = rng.integers(0, 256, (M, K // 2), dtype=np.uint8)
    s = rng.integers(lo, hi, (M, K // 32), dtype=np.uint8)
    return q, s


def test_cols_equal_scales_is_transpose_of_rows(oracle_mod):
    # With one exponent everywhere no shift happens, so the column conversion
    # is the transpose of the row conversion, whatever the groups.
    M, K = 300, 256
    q, _ = rand_mx(M, K, 1)
    s = np.full((M, K // 32), 117, dtype=np.uint8)
    offs = workloads.random_group_offsets(M, 5, seed=2)
    for k in (0, 3):
        y, ys = oracle_mod.fp4_to_fp8_rows(q, s, k)
        yT, yTs = oracle_mod.fp4_to_fp8_cols(q, s, offs, k)
        np.testing.assert_array_equal(yT, y.T)
        counts = np.diff(offs)
        nb = int(((counts + 127) // 128).sum())
        assert np.all(yTs[:nb] == np.float32(2.0 ** (117 - 127 - k)))
        assert np.all(np.isnan(yTs[nb:]))   # unused rows untouched


def test_cols_ragged_equals_per_group_calls(oracle_mod):
    M, K = 700, 256
    q, s = rand_mx(M, K, 5)
    offs = workloads.random_group_offsets(M, 7, seed=6)
    yT, yTs = oracle_mod.fp4_to_fp8_cols(q, s, offs, 2)
    base = 0
    for g in range(7):
        a, b = int(offs[g]), int(offs[g + 1])
        nb = (b - a + 127) // 128
        if b > a:
            yg, ygs = oracle_mod.fp4_to_fp8_cols(q[a:b], s[a:b], np.array([0, b - a]), 2)
            np.testing.assert_array_equal(yT[:, a:b], yg)
            np.testing.assert_array_equal(yTs[base:base + nb], ygs[:nb])
        base += nb


def test_cols_block_agrees_with_rows_on_runs(oracle_mod):
    # One 128-token block whose exponents come in four runs of 32 tokens is,
    # for every feature, the same problem as one 128-element row block with
    # four MX scales: the column conversion must agree with the row one.
    rng = np.random.default_rng(8)
    M, K = 128, 128
    codes = rng.integers(0, 16, (M, K), dtype=np.uint8)
    q = oracle_mod.pack_nibbles(codes)
    sig = rng.integers(90, 140, (4, K // 32)).astype(np.uint8)   # run r, column block j
    sig[2, 1] = sig[0, 1] + 14                                     # force a flushing shift
    s = np.repeat(sig, 32, axis=0)                                 # token t -> run t // 32
    for k in (0, 6):
        yT, yTs = oracle_mod.fp4_to_fp8_cols(q, s, np.array([0, M]), k)
        for f in range(K):
            j = f // 32
            row_codes = codes[:, f][None, :]
            y, ys = oracle_mod.fp4_to_fp8_rows(oracle_mod.pack_nibbles(row_codes),
                                               sig[:, j][None, :], k)
            np.testing.assert_array_equal(yT[f], y[0])
            assert yTs[0, f] == ys[0, 0]


def test_cols_rejects_bad_offsets(oracle_mod):
    q, s = rand_mx(10, 128, 0)
    for offs in ([0, 11], [1, 10], [0, 6, 4, 10]):
        with pytest.raises(ValueError):
            oracle_mod.fp4_to_fp8_cols(q, s, np.array(offs))
