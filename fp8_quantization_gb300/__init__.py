"""Block-scaled FP4 / FP8 casts for GB300 -- Python binding of libfq.so.

Every function here only marshals arguments: it checks the dtype, layout and
size of every tensor and that it lives on the current CUDA device, allocates
outputs with ``torch.empty`` when none are given, and calls
the C entry point of the same name (declared in ``include/fq.h``) on the
current CUDA stream.  All arithmetic runs in the sm_103a kernels of libfq.so;
there is no CPU or PyTorch fallback -- if the library is missing, every call
raises.

Sources (page title, section):
* "Practical FP4 Training for Large-Scale MoE Models on Hopper GPUs",
  technical overview section 2: MXFP4 (BF16ToFP4Row), direct FP4->FP8
  conversion with hierarchical scale alignment (FP4RowToFP8Row,
  FP4RowToFP8Col), ragged expert groups.
* "Train models faster with JAX and MaxText using NVFP4 on NVIDIA Blackwell",
  section "Receta de pre-entrenamiento NVFP4": NVFP4 1x16 and 16x16 scaling,
  stochastic rounding.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libfq.so")

FQ_COLS_MAX_GROUPS = 1024

_vp, _i64, _i32, _u64, _int = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_uint64,
                               ctypes.c_int)

# C signatures, by entry point (restype, argtypes); must match include/fq.h.
SIGNATURES = {
    "fq_status_string": (ctypes.c_char_p, [_int]),
    "fq_last_cuda_error": (_int, []),
    "fq_version": (_int, []),
    "mxfp4_quantize_rows": (_int, [_vp, _i64, _i64, _vp, _vp, _vp]),
    "fp4_to_fp8_rows": (_int, [_vp, _vp, _i64, _i64, _int, _vp, _vp, _vp]),
    "fp4_to_fp8_cols_scale_capacity": (_i64, [_i64, _i32]),
    "fp4_to_fp8_cols_launch_count": (_int, [_i64]),
    "fp4_to_fp8_cols": (_int, [_vp, _vp, _i64, _i64, _vp, _i32, _int, _vp, _vp, _i64, _vp, _vp]),
    "bf16_to_mxfp4_fp8": (_int, [_vp, _i64, _i64, _vp, _i32, _int, _vp, _vp, _vp, _vp, _vp, _vp,
                                 _i64, _vp, _vp]),
    "bf16_to_mxfp4_fp8_single_pass": (_int, [_vp, _i64, _i64, _vp, _i32, _int, _vp, _vp, _vp, _vp,
                                             _vp, _vp, _i64, _vp, _vp]),
    "nvfp4_amax": (_int, [_vp, _i64, _vp, _vp]),
    "nvfp4_quantize": (_int, [_vp, _i64, _i64, _vp, _int, _u64, _u64, _vp, _vp, _vp, _vp]),
    "nvfp4_quantize_2d": (_int, [_vp, _i64, _i64, _vp, _vp, _vp, _vp, _vp]),
    "nvfp4_quantize_2d_t": (_int, [_vp, _i64, _i64, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "nvfp4_amax_rht": (_int, [_vp, _i64, ctypes.c_uint32, _vp, _vp]),
    "fp8_quantize_1x128": (_int, [_vp, _i64, _i64, _vp, _vp, _vp]),
    "nvfp4_quantize_delayed": (_int, [_vp, _i64, _i64, _vp, _i32, ctypes.c_uint32, _int, _u64, _u64,
                                      _vp, _vp, _vp, _vp]),
    "fp8_quantize_128x128": (_int, [_vp, _i64, _i64, _vp, _vp, _vp]),
    "mxfp4_dequantize_rows": (_int, [_vp, _vp, _i64, _i64, _vp, _vp]),
    "mxfp4_scales_mma_bytes": (_i64, [_i64, _i64]),
    "mxfp4_scales_mma_layout": (_int, [_vp, _i64, _i64, _vp, _vp]),
    "nvfp4_quantize_rht": (_int, [_vp, _i64, _i64, _vp, ctypes.c_uint32, _int, _u64, _u64, _vp,
                                  _vp, _vp, _vp]),
}

_lock = threading.Lock()
_lib = None


class FQError(RuntimeError):
    """A libfq.so entry point returned a status other than FQ_OK."""

    def __init__(self, name: str, status: int):
        self.status = status
        msg = abi().fq_status_string(status).decode()
        if status == 5:
            msg += f" (cudaError {abi().fq_last_cuda_error()})"
        super().__init__(f"{name}: {msg}")


def abi() -> ctypes.CDLL:
    """The loaded libfq.so with typed entry points (raises if not built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"libfq.so not found at {LIB_PATH}: build it with "
                    "`python -c 'import __graft_entry__ as g; g.build()'` (nvcc, sm_103a)")
            L = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
        return _lib


def _call(name: str, *args) -> None:
    status = getattr(abi(), name)(*args)
    if status != 0:
        raise FQError(name, status)


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _p(t: torch.Tensor | None):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _need(t: torch.Tensor, dtype, name: str, ndim: int | None = None,
          numel: int | None = None, shape: tuple | None = None):
    """dtype, contiguity and size of a tensor argument (placement is checked
    by _on_device just before the call)."""
    if not isinstance(t, torch.Tensor):
        raise ValueError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if numel is not None and t.numel() != numel:
        raise ValueError(f"{name} must have {numel} elements, got {t.numel()}")


def _on_device(**tensors):
    """Every tensor given is a CUDA tensor on the current device (the library
    launches there); None entries are skipped."""
    cur = torch.cuda.current_device() if torch.cuda.is_available() else None
    for name, t in tensors.items():
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if t.device.index != cur:
            raise ValueError(f"{name} is on {t.device}, the current device is cuda:{cur}")


def _bf16(x: torch.Tensor, name: str, ndim: int | None = None):
    if not isinstance(x, torch.Tensor) or x.dtype not in (torch.bfloat16, torch.int16,
                                                           torch.uint16):
        raise ValueError(f"{name} must be bfloat16 (or its 16-bit pattern)")
    _need(x, x.dtype, name, ndim)


def _bf16_2d(x: torch.Tensor, name: str):
    _bf16(x, name, 2)


def _empty(shape, dtype, like: torch.Tensor):
    return torch.empty(shape, dtype=dtype, device=like.device)


# ---------------------------------------------------------------- MXFP4
# Sizes are checked wherever the block size divides the tensor; a size the
# block does not divide is passed on, and the library rejects it with
# FQ_ERR_SHAPE.

def mxfp4_quantize_rows(x: torch.Tensor, q: torch.Tensor | None = None,
                        s: torch.Tensor | None = None):
    """BF16 [M, K] -> (q uint8 [M, K/2] packed E2M1, s uint8 [M, K/32] UE8M0)."""
    _bf16_2d(x, "x")
    M, K = x.shape
    q = _empty((M, K // 2), torch.uint8, x) if q is None else q
    s = _empty((M, K // 32), torch.uint8, x) if s is None else s
    ok = K % 32 == 0
    _need(q, torch.uint8, "q", numel=M * K // 2 if ok else None)
    _need(s, torch.uint8, "s", numel=M * K // 32 if ok else None)
    _on_device(x=x, q=q, s=s)
    _call("mxfp4_quantize_rows", _p(x), M, K, _p(q), _p(s), _stream())
    return q, s


def fp4_to_fp8_rows(q: torch.Tensor, s: torch.Tensor, exp_offset_k: int = 0,
                    y: torch.Tensor | None = None, ys: torch.Tensor | None = None):
    """MXFP4 -> (y uint8 [M, K] E4M3, ys float32 [M, K/128])."""
    _need(q, torch.uint8, "q", 2)
    M, K = q.shape[0], q.shape[1] * 2
    _need(s, torch.uint8, "s", 2, shape=(M, K // 32))
    y = _empty((M, K), torch.uint8, q) if y is None else y
    ys = _empty((M, max(K // 128, 0)), torch.float32, q) if ys is None else ys
    ok = K % 128 == 0
    _need(y, torch.uint8, "y", numel=M * K if ok else None)
    _need(ys, torch.float32, "ys", numel=M * K // 128 if ok else None)
    _on_device(q=q, s=s, y=y, ys=ys)
    _call("fp4_to_fp8_rows", _p(q), _p(s), M, K, int(exp_offset_k), _p(y), _p(ys), _stream())
    return y, ys


def fp4_to_fp8_cols_scale_capacity(M: int, G: int) -> int:
    return int(abi().fp4_to_fp8_cols_scale_capacity(int(M), int(G)))


def fp4_to_fp8_cols_launch_count(K: int) -> int:
    return int(abi().fp4_to_fp8_cols_launch_count(int(K)))


def _groups(group_offsets: torch.Tensor) -> int:
    _need(group_offsets, torch.int64, "group_offsets", 1)
    G = group_offsets.numel() - 1
    if G < 1:
        raise ValueError("group_offsets must hold at least two entries (G >= 1)")
    return G


def fp4_to_fp8_cols(q: torch.Tensor, s: torch.Tensor, group_offsets: torch.Tensor,
                    exp_offset_k: int = 0, yT: torch.Tensor | None = None,
                    yT_scale: torch.Tensor | None = None, dev_status: torch.Tensor | None = None):
    """MXFP4 [M tokens, K] with int64 group offsets [G+1] (device) ->
    (yT uint8 [K, M] E4M3, yT_scale float32 [cap, K]: one row of K scales per
    128-token block)."""
    _need(q, torch.uint8, "q", 2)
    M, K = q.shape[0], q.shape[1] * 2
    _need(s, torch.uint8, "s", 2, shape=(M, K // 32))
    G = _groups(group_offsets)
    cap = fp4_to_fp8_cols_scale_capacity(M, G)
    yT = _empty((K, M), torch.uint8, q) if yT is None else yT
    yT_scale = _empty((cap, K), torch.float32, q) if yT_scale is None else yT_scale
    _need(yT, torch.uint8, "yT", numel=K * M)
    _need(yT_scale, torch.float32, "yT_scale", 2)
    if yT_scale.shape[1] != K or yT_scale.shape[0] < cap:
        raise ValueError(f"yT_scale must be [>= {cap}, {K}], got {tuple(yT_scale.shape)}")
    if dev_status is not None:
        _need(dev_status, torch.int32, "dev_status")
        if dev_status.numel() < 1:
            raise ValueError("dev_status must hold one int32")
    _on_device(q=q, s=s, group_offsets=group_offsets, yT=yT, yT_scale=yT_scale,
               dev_status=dev_status)
    _call("fp4_to_fp8_cols", _p(q), _p(s), M, K, _p(group_offsets), G, int(exp_offset_k), _p(yT),
          _p(yT_scale), int(yT_scale.shape[0]), _p(dev_status), _stream())
    return yT, yT_scale


def bf16_to_mxfp4_fp8(x: torch.Tensor, group_offsets: torch.Tensor, exp_offset_k: int = 0,
                      q=None, s=None, y=None, ys=None, yT=None, yT_scale=None,
                      dev_status: torch.Tensor | None = None):
    """BF16 [M, K] + int64 group offsets [G+1] (device) -> (q, s, y, ys, yT,
    yT_scale): the MXFP4 codes and scales, the FP8 rows and the transposed
    FP8 columns, equal to the three separate calls (two kernels)."""
    return _forward_cast("bf16_to_mxfp4_fp8", x, group_offsets, exp_offset_k, q, s, y, ys, yT,
                         yT_scale, dev_status)


def bf16_to_mxfp4_fp8_single_pass(x: torch.Tensor, group_offsets: torch.Tensor,
                                  exp_offset_k: int = 0, q=None, s=None, y=None, ys=None,
                                  yT=None, yT_scale=None, dev_status: torch.Tensor | None = None):
    """bf16_to_mxfp4_fp8 as one kernel that reads BF16 once and reads no
    output back (slower on GB300)."""
    return _forward_cast("bf16_to_mxfp4_fp8_single_pass", x, group_offsets, exp_offset_k, q, s, y,
                         ys, yT, yT_scale, dev_status)


def _forward_cast(entry, x, group_offsets, exp_offset_k, q, s, y, ys, yT, yT_scale, dev_status):
    _bf16_2d(x, "x")
    M, K = x.shape
    G = _groups(group_offsets)
    cap = fp4_to_fp8_cols_scale_capacity(M, G)
    q = _empty((M, K // 2), torch.uint8, x) if q is None else q
    s = _empty((M, K // 32), torch.uint8, x) if s is None else s
    y = _empty((M, K), torch.uint8, x) if y is None else y
    ys = _empty((M, K // 128), torch.float32, x) if ys is None else ys
    yT = _empty((K, M), torch.uint8, x) if yT is None else yT
    yT_scale = _empty((cap, K), torch.float32, x) if yT_scale is None else yT_scale
    ok = K % 128 == 0
    for t, name, dt, n in ((q, "q", torch.uint8, M * K // 2), (s, "s", torch.uint8, M * K // 32),
                           (y, "y", torch.uint8, M * K), (ys, "ys", torch.float32, M * K // 128),
                           (yT, "yT", torch.uint8, M * K)):
        _need(t, dt, name, numel=n if ok else None)
    _need(yT_scale, torch.float32, "yT_scale", 2)
    if yT_scale.shape[1] != K or yT_scale.shape[0] < cap:
        raise ValueError(f"yT_scale must be [>= {cap}, {K}], got {tuple(yT_scale.shape)}")
    if dev_status is not None:
        _need(dev_status, torch.int32, "dev_status")
        if dev_status.numel() < 1:
            raise ValueError("dev_status must hold one int32")
    _on_device(x=x, group_offsets=group_offsets, q=q, s=s, y=y, ys=ys, yT=yT, yT_scale=yT_scale,
               dev_status=dev_status)
    _call(entry, _p(x), M, K, _p(group_offsets), G, int(exp_offset_k), _p(q), _p(s),
          _p(y), _p(ys), _p(yT), _p(yT_scale), int(yT_scale.shape[0]), _p(dev_status), _stream())
    return q, s, y, ys, yT, yT_scale


# ---------------------------------------------------------------- NVFP4

def _one_float(t: torch.Tensor, name: str):
    _need(t, torch.float32, name)
    if t.numel() < 1:
        raise ValueError(f"{name} must hold one float32")


def nvfp4_amax(x: torch.Tensor, out: torch.Tensor | None = None) -> torch.Tensor:
    """max |x| of a BF16 tensor into a 1-element float32 device tensor."""
    _bf16(x, "x")
    out = _empty((1,), torch.float32, x) if out is None else out
    _one_float(out, "out")
    _on_device(x=x, out=out)
    _call("nvfp4_amax", _p(x), x.numel(), _p(out), _stream())
    return out


def _nvfp4_outputs(x, q, sb, g, sb_shape, ok):
    M, K = x.shape
    q = _empty((M, K // 2), torch.uint8, x) if q is None else q
    sb = _empty(sb_shape, torch.uint8, x) if sb is None else sb
    g = _empty((1,), torch.float32, x) if g is None else g
    _need(q, torch.uint8, "q", numel=M * K // 2 if ok else None)
    _need(sb, torch.uint8, "sb", numel=sb_shape[0] * sb_shape[1] if ok else None)
    _one_float(g, "g")
    return q, sb, g


def nvfp4_quantize(x: torch.Tensor, amax: torch.Tensor | None = None, use_sr: bool = False,
                   seed: int = 0, offset: int = 0, q: torch.Tensor | None = None,
                   sb: torch.Tensor | None = None, g: torch.Tensor | None = None):
    """BF16 [M, K] -> (q uint8 [M, K/2], sb uint8 [M, K/16] E4M3, g float32 [1])."""
    _bf16_2d(x, "x")
    M, K = x.shape
    q, sb, g = _nvfp4_outputs(x, q, sb, g, (M, K // 16), K % 16 == 0)
    amax = nvfp4_amax(x) if amax is None else amax
    _one_float(amax, "amax")
    _on_device(x=x, amax=amax, q=q, sb=sb, g=g)
    _call("nvfp4_quantize", _p(x), M, K, _p(amax), int(bool(use_sr)), int(seed) & (2**64 - 1),
          int(offset), _p(q), _p(sb), _p(g), _stream())
    return q, sb, g


def nvfp4_quantize_2d(w: torch.Tensor, amax: torch.Tensor | None = None,
                      q: torch.Tensor | None = None, sb: torch.Tensor | None = None,
                      g: torch.Tensor | None = None):
    """BF16 [N, K] -> (q uint8 [N, K/2], sb uint8 [N/16, K/16] E4M3, g float32 [1])."""
    _bf16_2d(w, "w")
    N, K = w.shape
    q, sb, g = _nvfp4_outputs(w, q, sb, g, (N // 16, K // 16), N % 16 == 0 and K % 16 == 0)
    amax = nvfp4_amax(w) if amax is None else amax
    _one_float(amax, "amax")
    _on_device(w=w, amax=amax, q=q, sb=sb, g=g)
    _call("nvfp4_quantize_2d", _p(w), N, K, _p(amax), _p(q), _p(sb), _p(g), _stream())
    return q, sb, g


def nvfp4_quantize_2d_t(w: torch.Tensor, amax: torch.Tensor | None = None, q=None, sb=None,
                        qT=None, sbT=None, g=None):
    """BF16 [N, K] -> (q uint8 [N, K/2], sb uint8 [N/16, K/16], qT uint8
    [K, N/2], sbT uint8 [K/16, N/16], g float32 [1]): the 2D-scaled weight for
    FPROP and its transpose for DGRAD, sharing the 16x16 scales, in one read."""
    _bf16_2d(w, "w")
    N, K = w.shape
    ok = N % 16 == 0 and K % 16 == 0
    q, sb, g = _nvfp4_outputs(w, q, sb, g, (N // 16, K // 16), ok)
    qT = _empty((K, N // 2), torch.uint8, w) if qT is None else qT
    sbT = _empty((K // 16, N // 16), torch.uint8, w) if sbT is None else sbT
    _need(qT, torch.uint8, "qT", numel=N * K // 2 if ok else None)
    _need(sbT, torch.uint8, "sbT", numel=N * K // 256 if ok else None)
    amax = nvfp4_amax(w) if amax is None else amax
    _one_float(amax, "amax")
    _on_device(w=w, amax=amax, q=q, sb=sb, qT=qT, sbT=sbT, g=g)
    _call("nvfp4_quantize_2d_t", _p(w), N, K, _p(amax), _p(q), _p(sb), _p(qT), _p(sbT), _p(g),
          _stream())
    return q, sb, qT, sbT, g


# ---------------------------------------------------------------- NVFP4 with the Hadamard transform

def nvfp4_amax_rht(x: torch.Tensor, sign_mask: int, out: torch.Tensor | None = None) -> torch.Tensor:
    """max |y| of the 16-point random Hadamard transform y of a BF16 tensor."""
    _bf16(x, "x")
    out = _empty((1,), torch.float32, x) if out is None else out
    _one_float(out, "out")
    _on_device(x=x, out=out)
    _call("nvfp4_amax_rht", _p(x), x.numel(), int(sign_mask) & 0xFFFF, _p(out), _stream())
    return out


def nvfp4_quantize_rht(x: torch.Tensor, amax: torch.Tensor, sign_mask: int, use_sr: bool = False,
                       seed: int = 0, offset: int = 0, q=None, sb=None, g=None):
    """NVFP4 1x16 quantization of the transformed BF16 tensor [M, K] ->
    (q uint8 [M, K/2], sb uint8 [M, K/16], g float32 [1])."""
    _bf16_2d(x, "x")
    M, K = x.shape
    q, sb, g = _nvfp4_outputs(x, q, sb, g, (M, K // 16), K % 16 == 0)
    _one_float(amax, "amax")
    _on_device(x=x, amax=amax, q=q, sb=sb, g=g)
    _call("nvfp4_quantize_rht", _p(x), M, K, _p(amax), int(sign_mask) & 0xFFFF, int(bool(use_sr)),
          int(seed) & (2**64 - 1), int(offset), _p(q), _p(sb), _p(g), _stream())
    return q, sb, g


# ---------------------------------------------------------------- FP8 backward flow and dequantization

def _fp8_blocks(name, x, block_rows, y=None, s=None):
    _bf16_2d(x, "x")
    M, K = x.shape
    y = _empty((M, K), torch.uint8, x) if y is None else y
    s = _empty((M // block_rows, K // 128), torch.float32, x) if s is None else s
    ok = K % 128 == 0 and M % block_rows == 0
    _need(y, torch.uint8, "y", numel=M * K)
    _need(s, torch.float32, "s", numel=(M // block_rows) * (K // 128) if ok else None)
    _on_device(x=x, y=y, s=s)
    _call(name, _p(x), M, K, _p(y), _p(s), _stream())
    return y, s


def fp8_quantize_1x128(x: torch.Tensor, y=None, s=None):
    """BF16 [M, K] -> (E4M3 codes uint8 [M, K], float32 scales [M, K/128])."""
    return _fp8_blocks("fp8_quantize_1x128", x, 1, y, s)


def fp8_quantize_128x128(w: torch.Tensor, y=None, s=None):
    """BF16 [N, K] -> (E4M3 codes uint8 [N, K], float32 scales [N/128, K/128])."""
    return _fp8_blocks("fp8_quantize_128x128", w, 128, y, s)


def mxfp4_dequantize_rows(q: torch.Tensor, s: torch.Tensor, out: torch.Tensor | None = None):
    """MXFP4 (q uint8 [M, K/2], s uint8 [M, K/32]) -> BF16 [M, K]."""
    _need(q, torch.uint8, "q", 2)
    M, K = q.shape[0], q.shape[1] * 2
    _need(s, torch.uint8, "s", 2, shape=(M, K // 32))
    out = torch.empty((M, K), dtype=torch.bfloat16, device=q.device) if out is None else out
    _need(out, torch.bfloat16, "out", numel=M * K)
    _on_device(q=q, s=s, out=out)
    _call("mxfp4_dequantize_rows", _p(q), _p(s), M, K, _p(out), _stream())
    return out


def mxfp4_scales_mma_bytes(M: int, K: int) -> int:
    """Bytes of the block-scaled-MMA scale layout of an [M, K] MXFP4 tensor
    (-1 for a rejected shape)."""
    return int(abi().mxfp4_scales_mma_bytes(int(M), int(K)))


def mxfp4_scales_mma_layout(s: torch.Tensor, out: torch.Tensor | None = None):
    """MXFP4 scales uint8 [M, K/32] -> uint8 [mxfp4_scales_mma_bytes(M, K)]:
    512-byte atoms of 128 rows x 4 scale columns for a block-scaled MMA
    operand (layout in include/fq.h)."""
    _need(s, torch.uint8, "s", 2)
    M, K = s.shape[0], s.shape[1] * 32
    n = mxfp4_scales_mma_bytes(M, K)
    if n < 0:
        raise ValueError(f"s of shape {tuple(s.shape)}: K = {K} must be a positive multiple of 128")
    out = torch.empty((n,), dtype=torch.uint8, device=s.device) if out is None else out
    _need(out, torch.uint8, "out", numel=n)
    _on_device(s=s, out=out)
    _call("mxfp4_scales_mma_layout", _p(s), M, K, _p(out), _stream())
    return out


# ---------------------------------------------------------------- delayed scaling (Max-Window)

def amax_history(window: int = 64, device="cuda") -> torch.Tensor:
    """A zeroed Max-Window history for nvfp4_quantize_delayed: window + 1
    entries (step tag << 32 | amax bits), held as int64."""
    return torch.zeros((window + 1,), dtype=torch.int64, device=device)


def nvfp4_quantize_delayed(x: torch.Tensor, history: torch.Tensor, step: int,
                           use_sr: bool = False, seed: int = 0, offset: int = 0,
                           q=None, sb=None, g=None):
    """NVFP4 1x16 quantization of BF16 [M, K] with the per-tensor amax taken
    from the Max-Window history (window = history.numel() - 1); records this
    tensor's amax under `step`.  Returns (q, sb, g)."""
    _bf16_2d(x, "x")
    _need(history, torch.int64, "history", 1)
    if history.numel() < 2:
        raise ValueError("history must hold window + 1 >= 2 entries")
    M, K = x.shape
    q, sb, g = _nvfp4_outputs(x, q, sb, g, (M, K // 16), K % 16 == 0)
    _on_device(x=x, history=history, q=q, sb=sb, g=g)
    _call("nvfp4_quantize_delayed", _p(x), M, K, _p(history), history.numel() - 1,
          int(step) & 0xFFFFFFFF, int(bool(use_sr)), int(seed) & (2**64 - 1), int(offset), _p(q),
          _p(sb), _p(g), _stream())
    return q, sb, g
