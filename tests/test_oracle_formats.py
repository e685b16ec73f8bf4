"""Pins of the oracle's scalar encoders against things other than itself:
the format definitions (golden files), brute-force nearest-value search,
library casts (ml_dtypes, torch) and published known-answer vectors."""
import numpy as np
import pytest
import torch

from conftest import read_golden

ml_dtypes = pytest.importorskip("ml_dtypes")


def all_bf16_finite():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    finite = ((bits >> 7) & 0xFF) != 0xFF
    bits = bits[finite]
    vals = (bits.astype(np.uint32) << 16).view(np.float32)
    return bits, vals


def brute_e2m1(y):
    """Nearest of the 8 grid magnitudes by exhaustive search, ties to the even
    code; the sign bit copied from the input.  Independent of the oracle."""
    grid = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    # values above 16 are clipped to 16 (which is still nearest to 6) so that
    # float64 distances stay exact for huge inputs
    a = np.minimum(np.abs(np.asarray(y, dtype=np.float64)), 16.0)[:, None]
    dist = np.abs(a - grid[None, :])
    best = dist.min(axis=1, keepdims=True)
    cand = dist == best
    # among the nearest, prefer the even code (there are at most two)
    even = cand & (np.arange(8)[None, :] % 2 == 0)
    code = np.where(even.any(axis=1), even.argmax(axis=1), cand.argmax(axis=1))
    return (code | np.where(np.signbit(y), 8, 0)).astype(np.uint8)


def test_e2m1_grid_matches_format(oracle_mod):
    for code, value in read_golden("e2m1_grid.txt"):
        c, v = int(code), float(value)
        mag = oracle_mod.e2m1_magnitude(c & 7)
        assert mag == abs(v), (c, v, mag)
        assert oracle_mod.e2m1_decode(np.uint8(c)) == v
        assert np.signbit(oracle_mod.e2m1_decode(np.uint8(c))) == bool(c & 8)


def test_e4m3_limits_match_format(oracle_mod):
    for code, value in read_golden("e4m3_limits.txt"):
        c, v = int(code, 16), float(value)
        assert oracle_mod.e4m3_decode(np.uint8(c)) == v
        assert oracle_mod.e4m3_rne(np.array([v]))[0] == c


def test_e2m1_rne_exhaustive_over_bf16_values(oracle_mod):
    # Every BF16 value (the MXFP4 element path only ever sees BF16 values times
    # a power of two) against brute force and against ml_dtypes' cast.
    _, vals = all_bf16_finite()
    got = oracle_mod.e2m1_rne(vals.astype(np.float64))
    np.testing.assert_array_equal(got, brute_e2m1(vals))
    lib_codes = vals.astype(ml_dtypes.float4_e2m1fn).view(np.uint8) & 0xF
    np.testing.assert_array_equal(got, lib_codes)


def test_e2m1_rne_random_float32(oracle_mod):
    rng = np.random.default_rng(11)
    y = (rng.random(400_000) * 8).astype(np.float32)
    y[::3] *= -1
    # exact ties and their neighbours
    ties = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0, 7.0], dtype=np.float32)
    y = np.concatenate([y, ties, np.nextafter(ties, 0), np.nextafter(ties, 10), -ties])
    got = oracle_mod.e2m1_rne(y.astype(np.float64))
    np.testing.assert_array_equal(got, brute_e2m1(y))
    np.testing.assert_array_equal(got, y.astype(ml_dtypes.float4_e2m1fn).view(np.uint8) & 0xF)


def test_e2m1_sign_of_zero(oracle_mod):
    got = oracle_mod.e2m1_rne(np.array([-0.1, -0.0, 0.0, 0.1, -0.25, 0.25]))
    np.testing.assert_array_equal(got, [8, 8, 0, 0, 8, 0])


def e4m3_torch(t):
    return torch.from_numpy(np.asarray(t, dtype=np.float32)).to(torch.float8_e4m3fn).view(
        torch.uint8).numpy()


def test_e4m3_rne_against_torch_cast(oracle_mod):
    # (a) every code value, every midpoint, and one float32 ulp either side
    vals = np.array([oracle_mod.e4m3_magnitude(c) for c in range(127)])
    mids = (vals[:-1] + vals[1:]) / 2
    pts = np.concatenate([vals, mids]).astype(np.float32)
    pts = np.concatenate([pts, np.nextafter(pts, np.float32(0)), np.nextafter(pts, np.float32(1e9))])
    # (b) a stride through all float32 patterns of [0, 464)
    hi = np.float32(464.0).view(np.uint32)
    stride = np.arange(0, hi, 97, dtype=np.uint32).view(np.float32)
    # (c) random values
    rnd = np.random.default_rng(5).random(1 << 20).astype(np.float32) * np.float32(464.0)
    t = np.concatenate([pts, stride, rnd])
    t = t[(t >= 0) & (t < 464)]
    got = oracle_mod.e4m3_rne(t.astype(np.float64))
    np.testing.assert_array_equal(got, e4m3_torch(t))


def test_e4m3_saturates_above_448(oracle_mod):
    t = np.array([448.0, 450.0, 464.0, 465.0, 1e6, 3.4e38, np.inf])
    np.testing.assert_array_equal(oracle_mod.e4m3_rne(t), [0x7E] * len(t))
    assert oracle_mod.e4m3_rne(np.array([np.nan]))[0] == 0x7F


def test_ue8m0_scale_closed_form(oracle_mod):
    # For every positive finite BF16 amax: e = floor(log2 amax) - 2 + 127,
    # clamped at 0; whenever not clamped, amax / 2^(e-127) lies in [4, 8).
    _, vals = all_bf16_finite()
    vals = vals[vals > 0]
    for a in vals[:: 7]:
        e = oracle_mod.mx_scale_exponent(float(a))
        scaled = float(a) * 2.0 ** (127 - e)
        if e > 0:
            assert 4.0 <= scaled < 8.0, (a, e)
        else:
            assert scaled < 8.0
        # the UE8M0 byte e encodes 2^(e-127) (library cast)
        if 0 < e < 255:
            enc = np.array([2.0 ** (e - 127)], dtype=np.float32).astype(ml_dtypes.float8_e8m0fnu)
            assert enc.view(np.uint8)[0] == e
    assert oracle_mod.mx_scale_exponent(0.0) == 0
    assert oracle_mod.mx_scale_exponent(4.0) == 127
    assert oracle_mod.mx_scale_exponent(7.99) == 127
    assert oracle_mod.mx_scale_exponent(8.0) == 128


def test_philox_known_answers(oracle_mod):
    rows = read_golden("philox4x32_10_kat.txt")
    for row in rows:
        v = [int(h, 16) for h in row]
        out = oracle_mod.philox4x32_10([v[0:4]], [v[4:6]])[0]
        assert [int(o) for o in out] == v[6:10]
