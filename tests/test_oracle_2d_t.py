"""Pins of the oracle's 2D weight quantization with the transposed (DGRAD)
operand (reading: one FP8 scale per 16x16 weight block, shared by FPROP and its
transposed DGRAD, so W^T's operand is W's codes and scales transposed).

The transposed outputs are checked against the 2D quantizer applied to the
transposed BF16 tensor (a computation that never runs the transposition code),
against a brute-force unpack of the nibbles, and by decoding both operands to
the same values."""
import numpy as np
import pytest

import oracle
from fp8_quantization_gb300 import workloads


def weight(N, K, seed):
    rng = np.random.default_rng(seed)
    w = rng.normal(0.0, 0.02, (N, K)).astype(np.float32)
    w[:16, 16:32] *= 300.0      # one loud tile
    w[16:32, :16] = 0.0         # one silent tile
    w[rng.random((N, K)) < 1e-3] *= -50.0
    return workloads.bf16_bits(w)


def amax_of(bits):
    return float(np.abs(workloads.bits_to_float(bits)).max())


@pytest.mark.parametrize("N,K", [(32, 32), (48, 96), (256, 64), (64, 272)])
def test_dgrad_operand_is_the_2d_quantization_of_the_transpose(N, K):
    w = weight(N, K, seed=N + K)
    A = amax_of(w)
    q, sb, qT, sbT, g = oracle.nvfp4_quantize_2d_t(w, A)
    rq, rsb, rg = oracle.nvfp4_quantize_2d(w, A)
    assert np.array_equal(q, rq) and np.array_equal(sb, rsb) and g == rg
    tq, tsb, tg = oracle.nvfp4_quantize_2d(np.ascontiguousarray(w.T), A)
    assert qT.shape == (K, N // 2) and sbT.shape == (K // 16, N // 16)
    assert np.array_equal(qT, tq)
    assert np.array_equal(sbT, tsb)
    assert tg == g


def test_codes_and_scales_are_transposed_element_by_element():
    N, K = 48, 80
    w = weight(N, K, seed=3)
    q, sb, qT, sbT, _ = oracle.nvfp4_quantize_2d_t(w, amax_of(w))
    codes, codesT = oracle.unpack_nibbles(q), oracle.unpack_nibbles(qT)
    for n in range(N):
        for k in range(K):
            assert codesT[k, n] == codes[n, k]
    for i in range(N // 16):
        for j in range(K // 16):
            assert sbT[j, i] == sb[i, j]


def test_both_operands_decode_to_the_same_values():
    N, K = 64, 128
    w = weight(N, K, seed=4)
    q, sb, qT, sbT, g = oracle.nvfp4_quantize_2d_t(w, amax_of(w))
    mags = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])

    def decode(qq, ss):
        c = oracle.unpack_nibbles(qq)
        val = np.where(c & 8, -1.0, 1.0) * mags[c & 7]
        s = oracle.e4m3_decode(ss).astype(np.float64)
        return val * np.repeat(np.repeat(s, 16, axis=0), 16, axis=1) * float(g)

    assert np.array_equal(decode(qT, sbT), decode(q, sb).T)
