"""Pins of the oracle's 16-point random Hadamard transform and of the NVFP4
quantizer fed by it (reading: per 16 consecutive elements, y = (1/4) H16
diag(d) x with H16 the Sylvester Hadamard matrix and d from a 16-bit sign
mask, binary32 fast Walsh-Hadamard butterflies, then x 0.25).

The pins tie the transform to the mathematics, not to itself: one-hot blocks
give the signed Hadamard columns exactly (order, signs and the 1/4 factor);
on inputs whose sums are exact it equals the matrix product computed in
float64 and is its own inverse (H16 H16 = 16 I); and the quantizer of the
transformed tensor equals the already pinned BF16 quantizer wherever the
transform is exactly representable in BF16."""
import numpy as np
import pytest

import oracle
from fp8_quantization_gb300 import workloads


def hadamard16():
    i = np.arange(16)
    pc = np.vectorize(lambda v: bin(v).count("1"))(i[:, None] & i[None, :])
    return np.where(pc % 2 == 0, 1.0, -1.0)


def signs(mask):
    return np.where((mask >> np.arange(16)) & 1, -1.0, 1.0)


def bf16(a):
    return workloads.bf16_bits(np.asarray(a, dtype=np.float32))


@pytest.mark.parametrize("mask", [0x0000, 0xFFFF, 0x5A3C, 0x8001])
def test_one_hot_blocks_give_signed_hadamard_columns(mask):
    H = hadamard16()
    d = signs(mask)
    x = np.eye(16, dtype=np.float32)  # block j = e_j
    y = oracle.rht16(bf16(x), mask)
    want = 0.25 * (H * d[None, :]).T  # row j: 0.25 * d_j * column j of H
    assert np.array_equal(y, want.astype(np.float32))


def test_equals_exact_matrix_product_on_small_integers():
    rng = np.random.default_rng(1)
    H = hadamard16()
    for mask in (0, 0x1234, 0xFFFF, 0x0F0F):
        x = rng.integers(-200, 201, (64, 16)).astype(np.float32)  # every sum exact
        y = oracle.rht16(bf16(x), mask)
        want = 0.25 * (x.astype(np.float64) * signs(mask)[None, :]) @ H.T
        assert np.array_equal(y.astype(np.float64), want)


def test_transform_is_its_own_inverse_without_signs():
    rng = np.random.default_rng(2)
    x = (rng.integers(-4, 5, (32, 16)) * 4).astype(np.float32)
    y = oracle.rht16(bf16(x), 0)  # y = H x / 4: integers, |y| <= 64, exact in BF16
    assert np.array_equal(workloads.bits_to_float(bf16(y)), y)
    z = oracle.rht16(bf16(y), 0)  # H H x / 16 = x
    assert np.array_equal(z, x)


def test_norm_preserved_within_rounding():
    rng = np.random.default_rng(3)
    bits = workloads.nvfp4_act(40, 64, seed=4)
    x = workloads.bits_to_float(bits).astype(np.float64).reshape(-1, 16)
    y = oracle.rht16(bits, 0xBEEF).astype(np.float64).reshape(-1, 16)
    nx, ny = np.linalg.norm(x, axis=1), np.linalg.norm(y, axis=1)
    assert np.allclose(nx, ny, rtol=4e-6, atol=0.0)


def test_amax_of_the_transform():
    bits = workloads.nvfp4_act(33, 48, seed=5)
    y = oracle.rht16(bits, 0x7777)
    assert oracle.nvfp4_amax_rht(bits, 0x7777) == np.float32(np.abs(y).max())
    assert oracle.nvfp4_amax_rht(np.zeros((2, 16), np.uint16), 3) == 0.0
    bad = bits.copy()
    bad[3, 7] = 0x7FC0  # NaN spreads through its block
    assert np.isnan(oracle.nvfp4_amax_rht(bad, 0x7777))


@pytest.mark.parametrize("sr", [False, True])
def test_quantizer_is_the_bf16_quantizer_of_the_transform(sr):
    """x = blocks whose transform is exactly BF16: one-hot blocks scaled by
    random powers of two and signs (y entries are +-2^k / 4).  Quantizing x
    with the transform must equal quantizing the BF16 transform directly."""
    rng = np.random.default_rng(6)
    M, K = 24, 64
    x = np.zeros((M, K), dtype=np.float32)
    for r in range(M):
        for b in range(K // 16):
            j = rng.integers(0, 16)
            x[r, 16 * b + j] = rng.choice([-1.0, 1.0]) * np.float32(2.0) ** rng.integers(-8, 9)
    bits = bf16(x)
    mask = 0x3C5A
    y = oracle.rht16(bits, mask)
    ybits = bf16(y)
    assert np.array_equal(workloads.bits_to_float(ybits), y)  # exactly representable
    A = oracle.nvfp4_amax_rht(bits, mask)
    assert A == oracle.nvfp4_amax(ybits)
    got = oracle.nvfp4_quantize_rht(bits, A, mask, use_sr=sr, seed=99, offset=160)
    want = oracle.nvfp4_quantize(ybits, A, use_sr=sr, seed=99, offset=160)
    for a, b in zip(got, want):
        assert np.array_equal(np.asarray(a), np.asarray(b))
