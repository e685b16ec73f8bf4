"""Pins of the oracle's delayed per-tensor scaling with a Max-Window amax
history (reading: a ring of W+1 entries (step tag << 32 | amax bits); the
estimate at step t is the largest amax tagged t-W .. t-1, 0 if none; the
tensor is quantized by the 1x16 NVFP4 rule with that amax and its own amax is
recorded under tag t).

The window maximum is checked against a plain Python sliding-window max over a
sequence of steps; the quantized output against the already pinned NVFP4
quantizer at the estimate."""
import numpy as np
import pytest

import oracle
from fp8_quantization_gb300 import workloads


def tensor_with_amax(rng, M, K, amax):
    """BF16 tensor whose largest |value| is exactly `amax` (a BF16 number)."""
    x = rng.uniform(-1.0, 1.0, (M, K)).astype(np.float32) * np.float32(amax) * np.float32(0.5)
    x[rng.integers(0, M), rng.integers(0, K)] = np.float32(amax) * rng.choice([-1, 1])
    bits = workloads.bf16_bits(x)
    assert oracle.nvfp4_amax(bits) == np.float32(amax)
    return bits


@pytest.mark.parametrize("W", [1, 4, 64])
def test_estimate_is_the_window_max(W):
    rng = np.random.default_rng(W)
    hist = np.zeros(W + 1, dtype=np.uint64)
    seen = []
    for t in range(3 * W + 20):
        amax = float(workloads.bits_to_float(workloads.bf16_bits(
            np.array([np.exp2(rng.uniform(-8, 8))], dtype=np.float32)))[0])
        if t % 17 == 5:
            amax = 2.0 ** 100  # a spike that must expire after W steps
        bits = tensor_with_amax(rng, 4, 32, amax)
        want = max(seen[max(0, t - W):t], default=0.0)
        assert oracle.window_estimate(hist, W, t) == np.float32(want)
        q, sb, g, hist = oracle.nvfp4_quantize_delayed(bits, hist, W, t, use_sr=(t % 2 == 1),
                                                       seed=t, offset=0)
        rq, rsb, rg = oracle.nvfp4_quantize(bits, np.float32(want), use_sr=(t % 2 == 1), seed=t)
        assert np.array_equal(q, rq) and np.array_equal(sb, rsb) and g == rg
        seen.append(amax)
        e = int(hist[t % (W + 1)])
        assert e >> 32 == t and np.uint32(e & 0xFFFFFFFF).view(np.float32) == np.float32(amax)


def test_gap_longer_than_the_window_resets_the_estimate():
    W = 8
    rng = np.random.default_rng(0)
    hist = np.zeros(W + 1, dtype=np.uint64)
    for t in range(5):
        *_, hist = oracle.nvfp4_quantize_delayed(tensor_with_amax(rng, 2, 16, 4.0), hist, W, t)
    assert oracle.window_estimate(hist, W, 5) == 4.0
    assert oracle.window_estimate(hist, W, 4 + W) == 4.0       # step 4 is still in the window
    assert oracle.window_estimate(hist, W, 5 + W) == 0.0       # every entry expired


def test_tag_wraps_around():
    W = 3
    rng = np.random.default_rng(1)
    hist = np.zeros(W + 1, dtype=np.uint64)
    start = 2**32 - 2
    for i in range(5):
        t = (start + i) % 2**32
        *_, hist = oracle.nvfp4_quantize_delayed(tensor_with_amax(rng, 2, 16, float(2 ** i)), hist,
                                                 W, t)
    # steps start..start+4 had amax 1, 2, 4, 8, 16; at step start+5 the window
    # is start+2 .. start+4 (tags 0, 1, 2 after the wrap)
    assert oracle.window_estimate(hist, W, (start + 5) % 2**32) == 16.0
    assert oracle.window_estimate(hist, W, (start + 4) % 2**32) == 8.0


def test_current_tensor_above_the_estimate_saturates():
    """Delayed scaling's failure mode: a tensor larger than its estimate
    clips at the largest code (6) under the largest block scale (448)."""
    W = 4
    rng = np.random.default_rng(2)
    hist = np.zeros(W + 1, dtype=np.uint64)
    *_, hist = oracle.nvfp4_quantize_delayed(tensor_with_amax(rng, 2, 16, 1.0), hist, W, 0)
    big = tensor_with_amax(rng, 2, 16, 1024.0)
    q, sb, g, hist = oracle.nvfp4_quantize_delayed(big, hist, W, 1)
    x = workloads.bits_to_float(big)
    i = np.unravel_index(np.argmax(np.abs(x)), x.shape)
    codes = oracle.unpack_nibbles(q)
    assert g == np.float32(1.0) / np.float32(2688.0)
    assert codes[i] & 7 == 7 and sb[i[0], i[1] // 16] == 0x7E
