"""Pins of the oracle's NVFP4 quantizers.

Source: "Train models faster with JAX and MaxText using NVFP4 on NVIDIA
Blackwell", section "Receta de pre-entrenamiento NVFP4": 16-element
micro-blocks, E4M3 block scales under one FP32 per-tensor scale (two-level
micro-scaling), 16x16 2D weight scaling so that FPROP and the transposed
DGRAD share scales, stochastic rounding for unbiased gradient quantization.

The exact order of the scale arithmetic is a reading (the page gives none);
these tests pin its consequences: special cases, the error bound, symmetry and
scale invariance, the E4M3 rounding of the block scale against a library cast,
the stochastic-rounding probability exactly over every random value, and the
transpose relation of the 2D scaling."""
from fractions import Fraction

import numpy as np
import pytest
import torch

from fp8_quantization_gb300 import workloads


def f32(bits):
    return workloads.bits_to_float(bits)


def dequant(oracle_mod, q, sb, g, block_shape):
    codes = oracle_mod.unpack_nibbles(q)
    v = oracle_mod.e2m1_decode(codes)
    scale = oracle_mod.e4m3_decode(sb).astype(np.float64) * float(g)
    br, bc = block_shape
    scale = np.repeat(np.repeat(scale, br, axis=0), bc, axis=1)
    return v * scale


def test_amax_is_max_abs(oracle_mod):
    bits = workloads.nvfp4_act(64, 256, seed=1)
    a = oracle_mod.nvfp4_amax(bits)
    assert a == np.abs(f32(bits)).max()
    x = f32(bits).copy()
    x[3, 3] = np.nan
    assert np.isnan(oracle_mod.nvfp4_amax(workloads.bf16_bits(x)))


def test_zero_tensor(oracle_mod):
    bits = workloads.bf16_bits(np.zeros((16, 64), dtype=np.float32))
    for sr in (False, True):
        q, sb, g = oracle_mod.nvfp4_quantize(bits, 0.0, use_sr=sr, seed=3)
        assert np.all(q == 0) and np.all(sb == 0) and g == 1.0
    q, sb, g = oracle_mod.nvfp4_quantize_2d(bits, 0.0)
    assert np.all(q == 0) and np.all(sb == 0)


def test_block_scale_and_error_bound(oracle_mod):
    bits = workloads.nvfp4_act(128, 512, seed=2)
    A = oracle_mod.nvfp4_amax(bits)
    q, sb, g = oracle_mod.nvfp4_quantize(bits, A)
    x = f32(bits).astype(np.float64)
    xb = np.abs(x).reshape(128, 32, 16)
    amax_blk = xb.max(axis=2)
    # per-tensor scale: g * 2688 recovers A to binary32 rounding
    assert abs(float(g) * 2688.0 - float(A)) <= float(A) * 2.0 ** -23
    # the block holding the tensor maximum gets the top E4M3 code (448)
    r, c = np.unravel_index(np.argmax(amax_blk), amax_blk.shape)
    assert sb[r, c] == 0x7E
    # block scale byte = library E4M3 cast of t = amax_blk * (1 / (6 g)) (binary32)
    enc = np.float32(1.0) / (np.float32(6.0) * np.float32(g))
    t = (amax_blk.astype(np.float32) * enc).astype(np.float32)
    lib = torch.from_numpy(t).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(sb, lib)
    # error bound: one E2M1 half-gap (<= 1) or the saturation loss (< 0.4)
    # of the block scale, i.e. |x - xhat| <= b * g, and b * g <= amax/6 * 17/16
    xhat = dequant(oracle_mod, q, sb, g, (1, 16))
    bg = np.repeat(oracle_mod.e4m3_decode(sb) * float(g), 16, axis=1)
    err = np.abs(x - xhat)
    normal = np.repeat(sb >= 8, 16, axis=1)
    assert np.all(err[normal] <= bg[normal] * (1 + 1e-6))
    ratio = (err / np.repeat(np.where(amax_blk > 0, amax_blk, 1), 16, axis=1).reshape(128, 512))
    assert ratio[normal].max() <= 6.0 ** -1 * 17 / 16 + 1e-6
    print(f"NVFP4 max |x - xhat| / amax_blk = {ratio[normal].max():.4f}")
    # the largest element of every block with a normal scale encodes to +-6
    codes = oracle_mod.unpack_nibbles(q).reshape(128, 32, 16)
    top = np.take_along_axis(codes, np.argmax(xb, axis=2)[:, :, None], axis=2)[:, :, 0] & 7
    assert np.all(top[sb >= 8] == 7)


def test_sign_symmetry(oracle_mod):
    bits = workloads.nvfp4_act(32, 128, seed=4)
    A = oracle_mod.nvfp4_amax(bits)
    neg = bits ^ np.uint16(0x8000)
    for sr in (False, True):
        q1, sb1, _ = oracle_mod.nvfp4_quantize(bits, A, use_sr=sr, seed=77)
        q2, sb2, _ = oracle_mod.nvfp4_quantize(neg, A, use_sr=sr, seed=77)
        np.testing.assert_array_equal(sb1, sb2)
        np.testing.assert_array_equal(q1 ^ 0x88, q2)


def test_power_of_two_invariance(oracle_mod):
    # Scaling the tensor by 2^k scales g by 2^k and leaves every code and
    # block-scale byte unchanged (binary32 rounding commutes with 2^k).
    bits = workloads.nvfp4_act(32, 256, seed=5)
    A = oracle_mod.nvfp4_amax(bits)
    q, sb, g = oracle_mod.nvfp4_quantize(bits, A)
    q2d, sb2d, _ = oracle_mod.nvfp4_quantize_2d(bits, A)
    for k in (-20, -3, 5, 30):
        bk = workloads.bf16_bits(f32(bits) * np.float32(2.0 ** k))
        Ak = oracle_mod.nvfp4_amax(bk)
        assert Ak == np.float32(A * 2.0 ** k)
        qk, sbk, gk = oracle_mod.nvfp4_quantize(bk, Ak)
        np.testing.assert_array_equal(q, qk)
        np.testing.assert_array_equal(sb, sbk)
        assert gk == np.float32(g * 2.0 ** k)
        qk2, sbk2, _ = oracle_mod.nvfp4_quantize_2d(bk, Ak)
        np.testing.assert_array_equal(q2d, qk2)
        np.testing.assert_array_equal(sb2d, sbk2)


def test_sr_probability_exact_over_all_random_values(oracle_mod):
    # For fixed y, enumerate all 2^16 random values R: the number that round
    # up (F + R >= 2^16) is floor(frac * 2^16) exactly, and the result is
    # always lo or hi.
    grid = [Fraction(0), Fraction(1, 2), Fraction(1), Fraction(3, 2), Fraction(2), Fraction(3),
            Fraction(4), Fraction(6)]
    rng = np.random.default_rng(12)
    ys = np.concatenate([rng.random(24) * 6, [0.0, 0.5, 1.0, 5.999, 2.0 + 2 ** -20,
                                              0.5 - 2 ** -30, 6.0, 7.5]]).astype(np.float32)
    R = np.arange(1 << 16, dtype=np.uint32)
    for y in ys:
        codes = oracle_mod.e2m1_sr(np.full(R.size, float(y)), R)
        fy = Fraction(float(y))
        if fy >= 6:
            assert np.all(codes == 7)
            continue
        lo = max(i for i in range(8) if grid[i] <= fy)
        frac = (fy - grid[lo]) / (grid[lo + 1] - grid[lo])
        ups = int((codes == lo + 1).sum())
        assert set(np.unique(codes)) <= {lo, lo + 1}
        assert ups == int(frac * 65536) // 1, (y, ups)


def test_sr_unbiased_in_expectation(oracle_mod):
    x = np.full((16, 16), 0.0, dtype=np.float32)
    x[:, 0] = 6.0                   # block max fixes the scale: t = 6/(6g) ...
    x[:, 1:] = 2.3                  # ... and the rest sit between grid points
    bits = workloads.bf16_bits(x)
    A = oracle_mod.nvfp4_amax(bits)
    vals = []
    for seed in range(64):
        q, sb, g = oracle_mod.nvfp4_quantize(bits, A, use_sr=True, seed=seed)
        vals.append(dequant(oracle_mod, q, sb, g, (1, 16))[:, 1:])
    vals = np.concatenate([v.ravel() for v in vals])
    target = float(f32(bits)[0, 1])
    sigma = vals.std() / np.sqrt(vals.size)
    assert abs(vals.mean() - target) < 4 * sigma + 1e-3 * target
    assert len(np.unique(vals)) == 2   # exactly the two neighbours


def test_sr_shards_match_whole(oracle_mod):
    # Row shards quantized with the element offset of their first row (and
    # the global amax) reproduce the unsharded stochastic result.
    bits = workloads.nvfp4_act(48, 160, seed=6)
    A = oracle_mod.nvfp4_amax(bits)
    q, sb, g = oracle_mod.nvfp4_quantize(bits, A, use_sr=True, seed=2024)
    parts = []
    for r0, r1 in ((0, 16), (16, 17), (17, 48)):
        qp, sbp, gp = oracle_mod.nvfp4_quantize(bits[r0:r1], A, use_sr=True, seed=2024,
                                                offset=r0 * 160)
        assert gp == g
        parts.append((qp, sbp))
    np.testing.assert_array_equal(np.concatenate([p[0] for p in parts]), q)
    np.testing.assert_array_equal(np.concatenate([p[1] for p in parts]), sb)


def bitrev16(v):
    return int(f"{int(v):016b}"[::-1], 2)


def test_sr_stream_definition(oracle_mod):
    """A definition check, not a pin: it restates the library's mapping of
    Philox words onto elements (reading R12) and confirms the oracle follows
    it, so it cannot catch a wrong mapping.  What pins the stream's
    statistics is test_sr_up_rate_closed_form_every_position below (oracle)
    and test_gpu_sr_closed_form.py (device)."""
    # Element j = offset + i draws 16 bits from word (j/4) mod 4 of
    # Philox4x32-10(key=seed, counter=(j/16, 0, 0)): with W that word,
    # P = W[23:16]W[7:0], Q = W[31:24]W[15:8], and elements j mod 4 = 0..3
    # use P, rev(P), Q, rev(Q).  Reproduce one block from the raw words.
    x = np.full((1, 16), 2.5, dtype=np.float32)
    x[0, 0] = 6.0
    bits = workloads.bf16_bits(x)
    A = oracle_mod.nvfp4_amax(bits)
    seed = 0x1234_5678_9ABC_DEF0
    q, sb, g = oracle_mod.nvfp4_quantize(bits, A, use_sr=True, seed=seed, offset=32)
    codes = oracle_mod.unpack_nibbles(q)[0]
    key = [seed & 0xFFFFFFFF, seed >> 32]
    words = oracle_mod.philox4x32_10([[2, 0, 0, 0]], [key])[0]   # elements 32..47 -> counter 2
    R = []
    for W in words:
        W = int(W)
        P = (((W >> 16) & 0xFF) << 8) | (W & 0xFF)
        Q = (((W >> 24) & 0xFF) << 8) | ((W >> 8) & 0xFF)
        R += [P, bitrev16(P), Q, bitrev16(Q)]
    r = np.float32(1.0) / (np.float32(448.0) * np.float32(g))   # b = 448 here
    y = np.float32(2.5) * r
    assert sb[0, 0] == 0x7E
    want = oracle_mod.e2m1_sr(np.full(16, float(y)), np.array(R, dtype=np.uint32))
    np.testing.assert_array_equal(codes[1:], want[1:])
    # y = 2.5 * 6 / 6 sits between 2 and 3 with frac ~ 1/2: both outcomes occur
    assert set(codes[1:].tolist()) <= {4, 5}


def test_sr_random_numbers_are_uniform(oracle_mod):
    # Each element's 16-bit number is uniform: over many blocks the up-rate of
    # a value with frac = 1/2 is 1/2 for every position in the block.
    x = np.full((4096, 16), 1.25, dtype=np.float32)   # frac 1/2 between 1 and 1.5
    x[:, 0] = 6.0
    bits = workloads.bf16_bits(x)
    A = oracle_mod.nvfp4_amax(bits)
    q, sb, g = oracle_mod.nvfp4_quantize(bits, A, use_sr=True, seed=99)
    assert np.all(sb == 0x7E)
    codes = oracle_mod.unpack_nibbles(q)[:, 1:]
    up = (codes == 3).mean(axis=0)
    assert np.all(np.abs(up - 0.5) < 4 * 0.5 / np.sqrt(4096)), up


@pytest.mark.parametrize("setup", ["pow2", "near1"])
@pytest.mark.parametrize("rht", [False, True])
def test_sr_up_rate_closed_form_every_position(oracle_mod, setup, rht):
    """The oracle's stochastic rounding against the closed form of unbiased
    rounding (sr_closed_form): per value and per position in the block, the
    up-rate over seeds is floor(2^16 frac) / 2^16 within 4 sigma, at
    fractions derived from the E2M1 grid -- independent of how the Philox
    words are mapped onto elements."""
    import sr_closed_form as S
    seeds, nblocks, mask = 48, 16384, 0xA5C3
    d = S.build(setup, nblocks, mask if rht else None, K=1024)
    types = d["types"]
    nt = len(types)
    tix = np.where(d["etype"] < 0, nt - 1, d["etype"])
    lo = np.array([t[1] for t in types], dtype=np.uint8)[tix]
    hi = np.array([t[2] for t in types], dtype=np.uint8)[tix]
    ups = np.zeros(d["bits"].shape, dtype=np.int64)
    for seed in range(seeds):
        if rht:
            q, sb, g = oracle_mod.nvfp4_quantize_rht(d["bits"], d["A"], mask, use_sr=True,
                                                     seed=seed)
        else:
            q, sb, g = oracle_mod.nvfp4_quantize(d["bits"], d["A"], use_sr=True, seed=seed)
        assert np.all(sb == d["b"]) and g == d["g"]
        mag = oracle_mod.unpack_nibbles(q) & 7
        assert np.all((mag == lo) | (mag == hi))
        ups += (mag == hi) & (hi != lo)
    idx = (tix * 16 + d["epos"]).ravel()
    up_tp = np.bincount(idx, weights=ups.ravel(), minlength=nt * 16).reshape(nt, 16)
    trials = np.bincount(idx, minlength=nt * 16).reshape(nt, 16) * seeds
    S.check_counts(up_tp, trials, [t[3] for t in types], f"oracle rht={rht} {setup}")


def test_2d_transpose_relation(oracle_mod):
    # The point of 16x16 scaling: quantizing W^T gives the transpose of
    # quantizing W, codes and scales, bit for bit.
    w = workloads.nvfp4_weight(64, 96, seed=7)
    A = oracle_mod.nvfp4_amax(w)
    q, sb, g = oracle_mod.nvfp4_quantize_2d(w, A)
    qt, sbt, gt = oracle_mod.nvfp4_quantize_2d(np.ascontiguousarray(w.T), A)
    np.testing.assert_array_equal(oracle_mod.unpack_nibbles(q).T, oracle_mod.unpack_nibbles(qt))
    np.testing.assert_array_equal(sb.T, sbt)
    assert g == gt


def test_2d_equals_1d_when_each_row_block_holds_tile_max(oracle_mod):
    # If every 1x16 row block of a tile reaches the tile's max magnitude, the
    # tile scale equals each row-block scale and the two quantizers agree.
    rng = np.random.default_rng(13)
    w = rng.normal(0, 0.02, (32, 64)).astype(np.float32)
    tiles = np.abs(w).reshape(2, 16, 4, 16).max(axis=(1, 3))
    for tr in range(2):
        for tc in range(4):
            for i in range(16):
                w[16 * tr + i, 16 * tc + (i % 16)] = tiles[tr, tc] * (1 if i % 2 else -1)
    bits = workloads.bf16_bits(w)
    A = oracle_mod.nvfp4_amax(bits)
    q2, sb2, _ = oracle_mod.nvfp4_quantize_2d(bits, A)
    q1, sb1, _ = oracle_mod.nvfp4_quantize(bits, A)
    np.testing.assert_array_equal(q1, q2)
    np.testing.assert_array_equal(np.repeat(sb2, 16, axis=0), sb1)


def test_2d_error_bound_and_top_tile(oracle_mod):
    w = workloads.nvfp4_weight(128, 128, seed=8)
    A = oracle_mod.nvfp4_amax(w)
    q, sb, g = oracle_mod.nvfp4_quantize_2d(w, A)
    x = f32(w).astype(np.float64)
    tiles = np.abs(x).reshape(8, 16, 8, 16).max(axis=(1, 3))
    r, c = np.unravel_index(np.argmax(tiles), tiles.shape)
    assert sb[r, c] == 0x7E
    xhat = dequant(oracle_mod, q, sb, g, (16, 16))
    bg = np.repeat(np.repeat(oracle_mod.e4m3_decode(sb) * float(g), 16, axis=0), 16, axis=1)
    normal = np.repeat(np.repeat(sb >= 8, 16, axis=0), 16, axis=1)
    assert np.all(np.abs(x - xhat)[normal] <= bg[normal] * (1 + 1e-6))


# ---- non-finite values (reading R21: NaN ranks above +Inf in a block's amax,
# so a block holding NaN takes the NaN scale byte 0x7F; a NaN product encodes
# as code 7 (+6, sign clear), which is what Blackwell's FP4 conversion gives
# for any NaN; +-Inf saturates to +-6)

def _codes(oracle_mod, q):
    return oracle_mod.unpack_nibbles(q)


@pytest.mark.parametrize("sr", [False, True])
def test_nan_block_takes_the_nan_scale_and_nan_codes_are_plus_six(oracle_mod, sr):
    rng = np.random.default_rng(21)
    x = rng.standard_normal((2, 64)).astype(np.float32)
    x[0, 3] = np.nan
    bits = workloads.bf16_bits(x)
    bits[1, 17] = 0xFFC1                       # a negative NaN with a payload
    clean = bits.copy()
    clean[0, 3] = 0
    clean[1, 17] = 0
    A = float(np.abs(f32(clean)).max())
    q, sb, g = oracle_mod.nvfp4_quantize(bits, A, use_sr=sr, seed=5)
    rq, rsb, rg = oracle_mod.nvfp4_quantize(clean, A, use_sr=sr, seed=5)
    assert sb[0, 0] == 0x7F and sb[1, 1] == 0x7F          # the NaN blocks
    others = np.ones(sb.shape, dtype=bool)
    others[0, 0] = others[1, 1] = False
    assert np.array_equal(sb[others], rsb[others])          # no other block moves
    c, rc = _codes(oracle_mod, q), _codes(oracle_mod, rq)
    assert c[0, 3] == 7 and c[1, 17] == 7                   # NaN of either sign -> +6
    keep = np.ones(c.shape, dtype=bool)
    keep[0, :16] = keep[1, 16:32] = False
    assert np.array_equal(c[keep], rc[keep])


def test_infinities_saturate_and_give_the_largest_block_scale(oracle_mod):
    x = np.full((1, 32), 0.5, dtype=np.float32)
    x[0, 2] = np.inf
    x[0, 20] = -np.inf
    bits = workloads.bf16_bits(x)
    q, sb, g = oracle_mod.nvfp4_quantize(bits, 1.0)
    # amax = Inf: t = Inf * enc saturates to the largest E4M3 scale, 448
    assert sb.tolist() == [[0x7E, 0x7E]]
    c = _codes(oracle_mod, q)
    assert c[0, 2] == 0x7 and c[0, 20] == 0xF               # +6 and -6
    # 0.5 * r with r = 1 / (448 g), g = 1/2688: 0.5 * 6 = 3 -> code 5
    assert np.all(np.delete(c[0], [2, 20]) == 5)


def test_infinite_tensor_scale(oracle_mod):
    """A = +Inf: g = Inf and enc = 0, so finite blocks get scale 0 (codes +-0)
    and a block holding +-Inf gets t = Inf * 0 = NaN -> the NaN scale byte,
    r = 0, and its infinities give NaN products -> code 7."""
    x = np.full((1, 48), -0.25, dtype=np.float32)
    x[0, 1] = 2.0
    x[0, 20] = -np.inf
    bits = workloads.bf16_bits(x)
    q, sb, g = oracle_mod.nvfp4_quantize(bits, float("inf"))
    assert np.isinf(g)
    assert sb.tolist() == [[0, 0x7F, 0]]
    c = _codes(oracle_mod, q)[0]
    assert c[1] == 0 and c[0] == 8 and np.all(c[32:] == 8)  # +0 for 2.0, -0 elsewhere
    assert c[20] == 7 and np.all(np.delete(c[16:32], 4) == 8)


def test_nan_tile_in_2d_scaling(oracle_mod):
    rng = np.random.default_rng(22)
    w = rng.normal(0.0, 0.02, (32, 32)).astype(np.float32)
    bits = workloads.bf16_bits(w)
    A = float(np.abs(f32(bits)).max())
    rq, rsb, _ = oracle_mod.nvfp4_quantize_2d(bits, A)
    bits[20, 5] = 0x7FC0
    q, sb, _ = oracle_mod.nvfp4_quantize_2d(bits, A)
    assert sb[1, 0] == 0x7F
    assert sb[0, 0] == rsb[0, 0] and sb[0, 1] == rsb[0, 1] and sb[1, 1] == rsb[1, 1]
    assert _codes(oracle_mod, q)[20, 5] == 7
    _, _, qT, sbT, _ = oracle_mod.nvfp4_quantize_2d_t(bits, A)
    assert sbT[0, 1] == 0x7F and _codes(oracle_mod, qT)[5, 20] == 7
