"""Plain CPU oracle for the block-scaled FP4/FP8 casts.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline / reference legs of ``bench.py`` may import this package.
The product path (``fp8_quantization_gb300``) never imports it and shares no
code with it: the C source here (``fq_oracle.c``) is compiled on its own with
gcc into ``oracle/_build/liboracle.so``.

What each routine computes, and the readings taken where the pages are silent,
is documented beside the routine in ``fq_oracle.c``.  Sources:

* "Practical FP4 Training for Large-Scale MoE Models on Hopper GPUs",
  technical overview section 2 (MXFP4 spec, direct FP4->FP8 conversion with
  hierarchical scale alignment, BF16ToFP4Row / FP4RowToFP8Row /
  FP4RowToFP8Col, ragged tensors).
* "Train models faster with JAX and MaxText using NVFP4 on NVIDIA Blackwell",
  section "Receta de pre-entrenamiento NVFP4" (16-element blocks, E4M3 block
  scales under an FP32 per-tensor scale, 16x16 2D weight scaling, stochastic
  rounding).

Pins (in ``tests/test_oracle_*.py``): exhaustive and brute-force checks of the
E2M1/E4M3 encoders, closed forms of the UE8M0 rule, the exact-equivalence
invariant of the FP4->FP8 alignment, metamorphic relations of the transposed
ragged conversion and of the 2D weight scaling, Philox known-answer vectors,
error bounds and special cases of NVFP4.  The exact operation order of the
NVFP4 scale arithmetic is a reading; its arithmetic is pinned by those
properties, not by a printed example (none exists).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fq_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (plain scalar code, OpenMP over rows)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-fno-fast-math", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB_PATH)
            vp, i64, i32, u64 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_uint64
            sig = {
                "oracle_e2m1_magnitude": (ctypes.c_double, [ctypes.c_int]),
                "oracle_e4m3_magnitude": (ctypes.c_double, [ctypes.c_int]),
                "oracle_mx_scale_exponent": (ctypes.c_int, [ctypes.c_double]),
                "oracle_philox4x32_10": (None, [vp, vp, vp]),
                "oracle_philox4x32_10_array": (None, [vp, vp, i64, vp]),
                "oracle_e2m1_rne_array": (None, [vp, i64, vp]),
                "oracle_e2m1_sr_array": (None, [vp, vp, i64, vp]),
                "oracle_e4m3_rne_array": (None, [vp, i64, vp]),
                "oracle_fp4_to_fp8_element_array": (None, [vp, vp, ctypes.c_int, i64, vp]),
                "oracle_num_threads": (ctypes.c_int, []),
                "oracle_set_num_threads": (None, [ctypes.c_int]),
                "oracle_mxfp4_quantize_rows": (ctypes.c_int, [vp, i64, i64, vp, vp]),
                "oracle_fp4_to_fp8_rows": (ctypes.c_int, [vp, vp, i64, i64, ctypes.c_int, vp, vp]),
                "oracle_fp4_to_fp8_cols_scale_capacity": (i64, [i64, i32]),
                "oracle_fp4_to_fp8_cols": (ctypes.c_int, [vp, vp, i64, i64, vp, i32, ctypes.c_int,
                                                          vp, vp, i64]),
                "oracle_nvfp4_amax": (ctypes.c_float, [vp, i64]),
                "oracle_nvfp4_quantize": (ctypes.c_int, [vp, i64, i64, ctypes.c_float, ctypes.c_int,
                                                         u64, u64, vp, vp, vp]),
                "oracle_nvfp4_quantize_2d": (ctypes.c_int, [vp, i64, i64, ctypes.c_float, vp, vp,
                                                            vp]),
                "oracle_nvfp4_quantize_2d_t": (ctypes.c_int, [vp, i64, i64, ctypes.c_float, vp,
                                                              vp, vp, vp, vp]),
                "oracle_rht16": (ctypes.c_int, [vp, i64, ctypes.c_uint32, vp]),
                "oracle_fp8_quantize_blocks": (ctypes.c_int, [vp, i64, i64, ctypes.c_int, vp, vp]),
                "oracle_window_estimate": (ctypes.c_float, [vp, i32, ctypes.c_uint32]),
                "oracle_nvfp4_quantize_delayed": (ctypes.c_int, [vp, i64, i64, vp, i32,
                                                                 ctypes.c_uint32, ctypes.c_int,
                                                                 u64, u64, vp, vp, vp]),
                "oracle_mxfp4_dequantize_rows": (ctypes.c_int, [vp, vp, i64, i64, vp]),
                "oracle_mxfp4_scales_mma_layout": (ctypes.c_int, [vp, i64, i64, vp]),
                "oracle_bf16_rne_array": (None, [vp, i64, vp]),
                "oracle_nvfp4_amax_rht": (ctypes.c_float, [vp, i64, ctypes.c_uint32]),
                "oracle_nvfp4_quantize_rht": (ctypes.c_int, [vp, i64, i64, ctypes.c_float,
                                                             ctypes.c_uint32, ctypes.c_int, u64,
                                                             u64, vp, vp, vp]),
                "oracle_mxfp4_error_stats": (ctypes.c_int, [vp, i64, i64, vp, vp, vp]),
                "oracle_nvfp4_error_stats": (ctypes.c_int, [vp, i64, i64, vp, vp, ctypes.c_float,
                                                            ctypes.c_int, vp]),
                "oracle_fp4_to_fp8_counts": (ctypes.c_int, [vp, vp, i64, i64, ctypes.c_int, vp,
                                                            i32, vp]),
            }
            for name, (res, args) in sig.items():
                f = getattr(L, name)
                f.restype = res
                f.argtypes = args
            _lib = L
        return _lib


def num_threads() -> int:
    return int(lib().oracle_num_threads())


def set_num_threads(n: int) -> None:
    """Threads of the oracle's later calls from this thread (for timing)."""
    lib().oracle_set_num_threads(int(n))


# ---------------------------------------------------------------- scalars

def e2m1_magnitude(code: int) -> float:
    return lib().oracle_e2m1_magnitude(int(code))


def e4m3_magnitude(code: int) -> float:
    return lib().oracle_e4m3_magnitude(int(code))


def mx_scale_exponent(amax: float) -> int:
    return int(lib().oracle_mx_scale_exponent(float(amax)))


def philox4x32_10(ctr, key) -> np.ndarray:
    ctr = np.ascontiguousarray(np.asarray(ctr, dtype=np.uint32).reshape(-1, 4))
    key = np.ascontiguousarray(np.asarray(key, dtype=np.uint32).reshape(-1, 2))
    assert ctr.shape[0] == key.shape[0]
    out = np.empty_like(ctr)
    lib().oracle_philox4x32_10_array(_p(ctr), _p(key), ctr.shape[0], _p(out))
    return out


def e2m1_rne(y) -> np.ndarray:
    y = np.ascontiguousarray(np.asarray(y, dtype=np.float64).ravel())
    out = np.empty(y.size, dtype=np.uint8)
    lib().oracle_e2m1_rne_array(_p(y), y.size, _p(out))
    return out


def e2m1_sr(y, R) -> np.ndarray:
    y = np.ascontiguousarray(np.asarray(y, dtype=np.float64).ravel())
    R = np.ascontiguousarray(np.asarray(R, dtype=np.uint32).ravel())
    assert R.size == y.size
    out = np.empty(y.size, dtype=np.uint8)
    lib().oracle_e2m1_sr_array(_p(y), _p(R), y.size, _p(out))
    return out


def e4m3_rne(t) -> np.ndarray:
    t = np.ascontiguousarray(np.asarray(t, dtype=np.float64).ravel())
    out = np.empty(t.size, dtype=np.uint8)
    lib().oracle_e4m3_rne_array(_p(t), t.size, _p(out))
    return out


def fp4_to_fp8_element(codes, d, k: int) -> np.ndarray:
    codes = np.ascontiguousarray(np.asarray(codes, dtype=np.uint8).ravel())
    d = np.ascontiguousarray(np.asarray(d, dtype=np.int32).ravel())
    assert d.size == codes.size
    out = np.empty(codes.size, dtype=np.uint8)
    lib().oracle_fp4_to_fp8_element_array(_p(codes), _p(d), int(k), codes.size, _p(out))
    return out


# ---------------------------------------------------------------- tensors
# Inputs are bf16 bit patterns as numpy uint16 arrays (row-major).

def _bits(x) -> np.ndarray:
    x = np.ascontiguousarray(x)
    assert x.dtype == np.uint16, "bf16 inputs are passed as uint16 bit patterns"
    return x


def mxfp4_quantize_rows(x):
    x = _bits(x)
    M, K = x.shape
    q = np.zeros((M, K // 2), dtype=np.uint8)
    s = np.zeros((M, K // 32), dtype=np.uint8)
    rc = lib().oracle_mxfp4_quantize_rows(_p(x), M, K, _p(q), _p(s))
    if rc:
        raise ValueError(f"oracle_mxfp4_quantize_rows: bad arguments M={M} K={K}")
    return q, s


def fp4_to_fp8_rows(q, s, k: int = 0):
    q = np.ascontiguousarray(q, dtype=np.uint8)
    s = np.ascontiguousarray(s, dtype=np.uint8)
    M, K = q.shape[0], q.shape[1] * 2
    y = np.zeros((M, K), dtype=np.uint8)
    ys = np.zeros((M, K // 128), dtype=np.float32)
    rc = lib().oracle_fp4_to_fp8_rows(_p(q), _p(s), M, K, int(k), _p(y), _p(ys))
    if rc:
        raise ValueError(f"oracle_fp4_to_fp8_rows: bad arguments M={M} K={K} k={k}")
    return y, ys


def fp4_to_fp8_cols_scale_capacity(M: int, G: int) -> int:
    return int(lib().oracle_fp4_to_fp8_cols_scale_capacity(int(M), int(G)))


def fp4_to_fp8_cols(q, s, offs, k: int = 0, cap: int | None = None, fill_scale=np.nan):
    q = np.ascontiguousarray(q, dtype=np.uint8)
    s = np.ascontiguousarray(s, dtype=np.uint8)
    offs = np.ascontiguousarray(offs, dtype=np.int64)
    M, K = q.shape[0], q.shape[1] * 2
    G = offs.size - 1
    if cap is None:
        cap = fp4_to_fp8_cols_scale_capacity(M, G)
    yT = np.zeros((K, M), dtype=np.uint8)
    yTs = np.full((cap, K), fill_scale, dtype=np.float32)
    rc = lib().oracle_fp4_to_fp8_cols(_p(q), _p(s), M, K, _p(offs), G, int(k), _p(yT), _p(yTs),
                                      int(cap))
    if rc:
        raise ValueError("oracle_fp4_to_fp8_cols: bad arguments")
    return yT, yTs


def nvfp4_amax(x) -> np.float32:
    x = _bits(x)
    return np.float32(lib().oracle_nvfp4_amax(_p(x), x.size))


def nvfp4_quantize(x, amax, use_sr: bool = False, seed: int = 0, offset: int = 0):
    x = _bits(x)
    M, K = x.shape
    q = np.zeros((M, K // 2), dtype=np.uint8)
    sb = np.zeros((M, K // 16), dtype=np.uint8)
    g = np.zeros(1, dtype=np.float32)
    rc = lib().oracle_nvfp4_quantize(_p(x), M, K, float(np.float32(amax)), int(bool(use_sr)),
                                     int(seed), int(offset), _p(q), _p(sb), _p(g))
    if rc:
        raise ValueError("oracle_nvfp4_quantize: bad arguments")
    return q, sb, g[0]


def nvfp4_quantize_2d(w, amax):
    w = _bits(w)
    N, K = w.shape
    q = np.zeros((N, K // 2), dtype=np.uint8)
    sb = np.zeros((N // 16, K // 16), dtype=np.uint8)
    g = np.zeros(1, dtype=np.float32)
    rc = lib().oracle_nvfp4_quantize_2d(_p(w), N, K, float(np.float32(amax)), _p(q), _p(sb), _p(g))
    if rc:
        raise ValueError("oracle_nvfp4_quantize_2d: bad arguments")
    return q, sb, g[0]


def nvfp4_quantize_2d_t(w, amax):
    """2D weight quantization with the transposed (DGRAD) operand: (q [N, K/2],
    sb [N/16, K/16], qT [K, N/2], sbT [K/16, N/16], g)."""
    w = _bits(w)
    N, K = w.shape
    q = np.zeros((N, K // 2), dtype=np.uint8)
    sb = np.zeros((N // 16, K // 16), dtype=np.uint8)
    qT = np.zeros((K, N // 2), dtype=np.uint8)
    sbT = np.zeros((K // 16, N // 16), dtype=np.uint8)
    g = np.zeros(1, dtype=np.float32)
    rc = lib().oracle_nvfp4_quantize_2d_t(_p(w), N, K, float(np.float32(amax)), _p(q), _p(sb),
                                          _p(qT), _p(sbT), _p(g))
    if rc:
        raise ValueError("oracle_nvfp4_quantize_2d_t: bad arguments")
    return q, sb, qT, sbT, g[0]


# ---------------------------------------------------------------- decoding helpers
# Plain table-free decoders used by tests to read results back as numbers.

def rht16(x, sign_mask: int) -> np.ndarray:
    """The 16-point random Hadamard transform of every 16-element block of
    x (BF16 bits, size a multiple of 16): float32 array of x's shape."""
    x = _bits(x)
    y = np.zeros(x.shape, dtype=np.float32)
    rc = lib().oracle_rht16(_p(x), x.size, int(sign_mask) & 0xFFFF, _p(y))
    if rc:
        raise ValueError("oracle_rht16: size must be a multiple of 16")
    return y


def nvfp4_amax_rht(x, sign_mask: int) -> np.float32:
    x = _bits(x)
    return np.float32(lib().oracle_nvfp4_amax_rht(_p(x), x.size, int(sign_mask) & 0xFFFF))


def nvfp4_quantize_rht(x, amax, sign_mask: int, use_sr: bool = False, seed: int = 0,
                       offset: int = 0):
    x = _bits(x)
    M, K = x.shape
    q = np.zeros((M, K // 2), dtype=np.uint8)
    sb = np.zeros((M, K // 16), dtype=np.uint8)
    g = np.zeros(1, dtype=np.float32)
    rc = lib().oracle_nvfp4_quantize_rht(_p(x), M, K, float(np.float32(amax)),
                                         int(sign_mask) & 0xFFFF, int(bool(use_sr)), int(seed),
                                         int(offset), _p(q), _p(sb), _p(g))
    if rc:
        raise ValueError("oracle_nvfp4_quantize_rht: bad arguments")
    return q, sb, g[0]


def fp8_quantize_blocks(x, block_rows: int):
    """BF16 bits [M, K] -> (E4M3 codes uint8 [M, K], float32 scales
    [M / block_rows, K / 128]); block_rows is 1 or 128."""
    x = _bits(x)
    M, K = x.shape
    y = np.zeros((M, K), dtype=np.uint8)
    sc = np.zeros((M // block_rows, K // 128), dtype=np.float32)
    rc = lib().oracle_fp8_quantize_blocks(_p(x), M, K, int(block_rows), _p(y), _p(sc))
    if rc:
        raise ValueError("oracle_fp8_quantize_blocks: bad arguments")
    return y, sc


def mxfp4_dequantize_rows(q, s):
    q = np.ascontiguousarray(q, dtype=np.uint8)
    s = np.ascontiguousarray(s, dtype=np.uint8)
    M, K = q.shape[0], q.shape[1] * 2
    out = np.zeros((M, K), dtype=np.uint16)
    rc = lib().oracle_mxfp4_dequantize_rows(_p(q), _p(s), M, K, _p(out))
    if rc:
        raise ValueError("oracle_mxfp4_dequantize_rows: bad arguments")
    return out


def mxfp4_scales_mma_layout(s, M: int, K: int):
    """MXFP4 scales [M, K/32] in the tiled layout of a block-scaled MMA
    operand: ceil(M/128) * K/128 atoms of 512 bytes (see the C oracle)."""
    s = np.ascontiguousarray(s, dtype=np.uint8)
    assert s.shape == (M, K // 32)
    out = np.full(((M + 127) // 128) * (K // 128) * 512, 0xA5, dtype=np.uint8)
    rc = lib().oracle_mxfp4_scales_mma_layout(_p(s), M, K, _p(out))
    if rc:
        raise ValueError("oracle_mxfp4_scales_mma_layout: bad arguments")
    return out


def bf16_rne(v) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.zeros(v.shape, dtype=np.uint16)
    lib().oracle_bf16_rne_array(_p(v), v.size, _p(out))
    return out


def window_estimate(history, window: int, step: int) -> np.float32:
    h = np.ascontiguousarray(history, dtype=np.uint64)
    assert h.size == window + 1
    return np.float32(lib().oracle_window_estimate(_p(h), int(window), int(step) & 0xFFFFFFFF))


def nvfp4_quantize_delayed(x, history, window: int, step: int, use_sr: bool = False,
                           seed: int = 0, offset: int = 0):
    """Returns (q, sb, g, history after the step); `history` is not modified."""
    x = _bits(x)
    M, K = x.shape
    h = np.array(history, dtype=np.uint64, copy=True)
    assert h.size == window + 1
    q = np.zeros((M, K // 2), dtype=np.uint8)
    sb = np.zeros((M, K // 16), dtype=np.uint8)
    g = np.zeros(1, dtype=np.float32)
    rc = lib().oracle_nvfp4_quantize_delayed(_p(x), M, K, _p(h), int(window),
                                             int(step) & 0xFFFFFFFF, int(bool(use_sr)), int(seed),
                                             int(offset), _p(q), _p(sb), _p(g))
    if rc:
        raise ValueError("oracle_nvfp4_quantize_delayed: bad arguments")
    return q, sb, g[0], h


def e2m1_decode(codes) -> np.ndarray:
    codes = np.asarray(codes, dtype=np.uint8)
    mag = np.array([e2m1_magnitude(c) for c in range(8)], dtype=np.float64)
    v = mag[codes & 7]
    return np.where(codes & 8, -v, v)


def e4m3_decode(codes) -> np.ndarray:
    codes = np.asarray(codes, dtype=np.uint8)
    mag = np.array([e4m3_magnitude(c) for c in range(128)], dtype=np.float64)
    mag[0x7F] = np.nan
    v = mag[codes & 0x7F]
    return np.where(codes & 0x80, -v, v)


def unpack_nibbles(q) -> np.ndarray:
    """[..., n/2] packed bytes -> [..., n] codes (low nibble first)."""
    q = np.asarray(q, dtype=np.uint8)
    out = np.empty(q.shape[:-1] + (q.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = q & 0xF
    out[..., 1::2] = q >> 4
    return out


def pack_nibbles(c) -> np.ndarray:
    c = np.asarray(c, dtype=np.uint8)
    return (c[..., 0::2] & 0xF) | ((c[..., 1::2] & 0xF) << 4)


# ---------------------------------------------------------------- statistics of the method
# Numbers about the formats on a given input (see fq_oracle.c): the
# dequantization error of the quantizers and the exactness of the FP4 -> FP8
# conversion.

def mxfp4_error_stats(x, q, s) -> dict:
    """Per 32-element block, max |x - xhat| / amax_blk over finite nonzero
    blocks: largest and mean ratio, block count, blocks above the 1/4 bound."""
    x = _bits(x)
    M, K = x.shape
    q = np.ascontiguousarray(q, dtype=np.uint8)
    s = np.ascontiguousarray(s, dtype=np.uint8)
    out = np.zeros(4, dtype=np.float64)
    if lib().oracle_mxfp4_error_stats(_p(x), M, K, _p(q), _p(s), _p(out)):
        raise ValueError("oracle_mxfp4_error_stats: bad arguments")
    return {"max_ratio": float(out[0]), "mean_ratio": float(out[1]), "blocks": int(out[2]),
            "over_bound": int(out[3]), "bound": 0.25}


def nvfp4_error_stats(x, q, sb, g, tile_rows: int = 1) -> dict:
    """Per 1x16 block (tile_rows = 1) or 16x16 tile, max |x - xhat| / amax_blk
    over finite nonzero blocks with a normal scale byte (and, separately, the
    count and largest ratio of blocks whose scale byte is subnormal or 0)."""
    x = _bits(x)
    M, K = x.shape
    q = np.ascontiguousarray(q, dtype=np.uint8)
    sb = np.ascontiguousarray(sb, dtype=np.uint8)
    out = np.zeros(5, dtype=np.float64)
    if lib().oracle_nvfp4_error_stats(_p(x), M, K, _p(q), _p(sb), float(np.float32(g)),
                                      int(tile_rows), _p(out)):
        raise ValueError("oracle_nvfp4_error_stats: bad arguments")
    return {"max_ratio": float(out[0]), "mean_ratio": float(out[1]), "blocks": int(out[2]),
            "small_scale_blocks": int(out[3]), "small_scale_max_ratio": float(out[4])}


def fp4_to_fp8_counts(q, s, k: int = 0, offs=None) -> dict:
    """Elements of the FP4 -> FP8 conversion (row blocks, or the ragged
    transposed blocks of `offs`) that are exact, rounded, flushed to zero,
    zero codes, or in blocks with a NaN scale."""
    q = np.ascontiguousarray(q, dtype=np.uint8)
    s = np.ascontiguousarray(s, dtype=np.uint8)
    M, K = q.shape[0], q.shape[1] * 2
    counts = np.zeros(5, dtype=np.int64)
    if offs is None:
        rc = lib().oracle_fp4_to_fp8_counts(_p(q), _p(s), M, K, int(k), None, 0, _p(counts))
    else:
        o = np.ascontiguousarray(offs, dtype=np.int64)
        rc = lib().oracle_fp4_to_fp8_counts(_p(q), _p(s), M, K, int(k), _p(o), o.size - 1,
                                            _p(counts))
    if rc:
        raise ValueError("oracle_fp4_to_fp8_counts: bad arguments")
    return dict(zip(("exact", "rounded", "flushed", "zero", "nan_block"), map(int, counts)))
