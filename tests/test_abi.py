"""The C ABI boundary on the CPU: libfq.so builds, loads, exports every entry
point declared in include/fq.h (and the binding types each of them), and
rejects bad arguments on the host before touching the GPU.  No call here
reaches a CUDA API."""
import ctypes
import os
import re
import subprocess

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "fq.h")


@pytest.fixture(scope="module")
def lib():
    from fp8_quantization_gb300 import build
    build.build()
    import fp8_quantization_gb300 as fq
    return fq.abi()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w \t\*]*?\b([a-z_][a-z0-9_]*)\s*\([^;{]*\)\s*;", text, re.M)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("mxfp4_quantize_rows", "fp4_to_fp8_rows", "fp4_to_fp8_cols",
              "fp4_to_fp8_cols_scale_capacity", "fp4_to_fp8_cols_launch_count",
              "bf16_to_mxfp4_fp8", "bf16_to_mxfp4_fp8_single_pass", "nvfp4_amax", "nvfp4_amax_rht", "nvfp4_quantize_rht",
              "fp8_quantize_1x128", "fp8_quantize_128x128", "mxfp4_dequantize_rows",
              "nvfp4_quantize_delayed", "nvfp4_quantize",
              "nvfp4_quantize_2d", "mxfp4_scales_mma_bytes", "mxfp4_scales_mma_layout",
              "fq_status_string", "fq_last_cuda_error", "fq_version"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    import fp8_quantization_gb300 as fq
    out = subprocess.run(["nm", "-D", "--defined-only", fq.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in declared_functions():
        assert name in exported, name
        assert getattr(lib, name) is not None
        assert name in fq.SIGNATURES, f"binding does not type {name}"
    assert set(fq.SIGNATURES) == set(declared_functions())


def test_no_torch_in_the_library(lib):
    import fp8_quantization_gb300 as fq
    out = subprocess.run(["ldd", fq.LIB_PATH], capture_output=True, text=True).stdout
    assert "torch" not in out and "c10" not in out


def test_status_strings_and_version(lib):
    assert lib.fq_version() >= 100
    for st, name in enumerate(["FQ_OK", "FQ_ERR_NULL", "FQ_ERR_SHAPE", "FQ_ERR_ALIGN",
                               "FQ_ERR_ARG", "FQ_ERR_CUDA"]):
        assert lib.fq_status_string(st).decode().startswith(name)
    assert lib.fq_last_cuda_error() == 0


OK, NULL, SHAPE, ALIGN, ARG = 0, 1, 2, 3, 4
P = ctypes.c_void_p(0x1000)        # 16-byte aligned fake device pointer (never dereferenced)
PM = ctypes.c_void_p(0x1008)       # misaligned


def test_host_validation_mxfp4(lib):
    f = lib.mxfp4_quantize_rows
    assert f(P, -1, 64, P, P, None) == SHAPE
    assert f(P, 4, 33, P, P, None) == SHAPE
    assert f(P, 4, 0, P, P, None) == SHAPE
    assert f(None, 0, 64, None, None, None) == OK          # empty: no-op
    assert f(None, 4, 64, P, P, None) == NULL
    assert f(PM, 4, 64, P, P, None) == ALIGN
    assert f(P, 2**40, 2**30, P, P, None) == SHAPE         # M*K overflows


def test_host_validation_rows_and_cols(lib):
    f = lib.fp4_to_fp8_rows
    assert f(P, P, 4, 96, 0, P, P, None) == SHAPE
    assert f(P, P, 4, 128, 7, P, P, None) == ARG
    assert f(P, P, 4, 128, -1, P, P, None) == ARG
    assert f(P, P, 0, 128, 0, None, None, None) == OK
    assert f(P, P, 4, 128, 0, P, None, None) == NULL
    assert f(P, P, 4, 128, 0, PM, P, None) == ALIGN
    cap = lib.fp4_to_fp8_cols_scale_capacity
    assert cap(0, 1) == 1 and cap(1, 1) == 2 and cap(128, 1) == 2 and cap(129, 3) == 5
    assert cap(-1, 1) == -1 and cap(5, 0) == -1
    # launch count: invalid K -> 0 (decided without a CUDA call; a valid K asks
    # the driver for its tensor-map encoder and is checked on the GPU)
    lc = lib.fp4_to_fp8_cols_launch_count
    assert lc(0) == 0 and lc(-128) == 0 and lc(64) == 0 and lc(200) == 0
    c = lib.fp4_to_fp8_cols
    assert c(P, P, 100, 128, P, 0, 0, P, P, 100, None, None) == ARG          # G < 1
    assert c(P, P, 100, 128, P, 1025, 0, P, P, 2000, None, None) == ARG      # G too large
    assert c(P, P, 100, 128, P, 4, 0, P, P, 4, None, None) == ARG            # cap too small
    assert c(P, P, 100, 64, P, 4, 0, P, P, 5, None, None) == SHAPE
    assert c(P, P, 2**31, 128, P, 4, 0, P, P, 2**25, None, None) == SHAPE    # M >= 2^31
    assert c(P, P, 100, 128, None, 4, 0, P, P, 5, None, None) == NULL
    assert c(P, P, 100, 128, PM, 4, 0, P, P, 5, None, None) == ALIGN
    assert c(P, P, 0, 128, P, 4, 0, P, P, 4, None, None) == OK


@pytest.mark.parametrize("entry", ["bf16_to_mxfp4_fp8", "bf16_to_mxfp4_fp8_single_pass"])
def test_host_validation_fused(lib, entry):
    f = getattr(lib, entry)
    # x, M, K, offs, G, k, q, s, y, ys, yT, yTs, cap, status, stream
    assert f(P, 100, 96, P, 4, 0, P, P, P, P, P, P, 5, None, None) == SHAPE    # K % 128
    assert f(P, -1, 128, P, 4, 0, P, P, P, P, P, P, 5, None, None) == SHAPE
    assert f(P, 100, 128, P, 0, 0, P, P, P, P, P, P, 5, None, None) == ARG     # G < 1
    assert f(P, 100, 128, P, 4, 7, P, P, P, P, P, P, 5, None, None) == ARG     # k > 6
    assert f(P, 100, 128, P, 4, 0, P, P, P, P, P, P, 4, None, None) == ARG     # cap too small
    assert f(P, 0, 128, P, 4, 0, P, P, P, P, P, P, 4, None, None) == OK        # empty
    assert f(P, 100, 128, P, 4, 0, P, P, None, P, P, P, 5, None, None) == NULL
    assert f(P, 100, 128, None, 4, 0, P, P, P, P, P, P, 5, None, None) == NULL
    assert f(PM, 100, 128, P, 4, 0, P, P, P, P, P, P, 5, None, None) == ALIGN


def test_host_validation_mma_layout(lib):
    n = lib.mxfp4_scales_mma_bytes
    assert n(0, 128) == 0 and n(1, 128) == 512 and n(128, 128) == 512 and n(129, 256) == 2048
    assert n(100, 7168) == 56 * 512
    assert n(-1, 128) == -1 and n(4, 96) == -1 and n(4, 0) == -1 and n(4, 64) == -1
    f = lib.mxfp4_scales_mma_layout
    assert f(P, 4, 96, P, None) == SHAPE
    assert f(P, -1, 128, P, None) == SHAPE
    assert f(None, 0, 128, None, None) == OK          # empty: no-op
    assert f(None, 4, 128, P, None) == NULL
    assert f(P, 4, 128, PM, None) == ALIGN


def test_host_validation_rht(lib):
    a = lib.nvfp4_amax_rht
    assert a(P, 40, 0x1234, P, None) == SHAPE      # n % 16
    assert a(P, -16, 0, P, None) == SHAPE
    assert a(P, 32, 0, None, None) == NULL
    assert a(PM, 32, 0, P, None) == ALIGN
    f = lib.nvfp4_quantize_rht
    # x, M, K, amax, mask, sr, seed, offset, q, sb, g, stream
    assert f(P, 4, 24, P, 0, 0, 0, 0, P, P, P, None) == SHAPE
    assert f(P, 4, 32, P, 0, 2, 0, 0, P, P, P, None) == ARG
    assert f(P, 4, 32, P, 0, 1, 0, 8, P, P, P, None) == ARG       # offset % 16
    assert f(P, 0, 32, P, 0, 0, 0, 0, None, None, None, None) == OK
    assert f(P, 4, 32, None, 0, 0, 0, 0, P, P, P, None) == NULL
    assert f(P, 4, 32, P, 0, 0, 0, 0, PM, P, P, None) == ALIGN


def test_host_validation_fp8_and_dequant(lib):
    a = lib.fp8_quantize_1x128
    assert a(P, 4, 96, P, P, None) == SHAPE
    assert a(P, 0, 128, None, None, None) == OK
    assert a(P, 4, 128, None, P, None) == NULL
    assert a(PM, 4, 128, P, P, None) == ALIGN
    b = lib.fp8_quantize_128x128
    assert b(P, 100, 128, P, P, None) == SHAPE     # N % 128
    assert b(P, 128, 64, P, P, None) == SHAPE
    assert b(P, 128, 128, P, None, None) == NULL
    d = lib.mxfp4_dequantize_rows
    assert d(P, P, 4, 48, P, None) == SHAPE
    assert d(P, P, 0, 64, None, None) == OK
    assert d(P, None, 4, 64, P, None) == NULL
    assert d(P, P, 4, 64, PM, None) == ALIGN


def test_host_validation_delayed(lib):
    f = lib.nvfp4_quantize_delayed
    # x, M, K, hist, W, step, sr, seed, offset, q, sb, g, stream
    assert f(P, 4, 24, P, 64, 0, 0, 0, 0, P, P, P, None) == SHAPE
    assert f(P, 4, 32, P, 0, 0, 0, 0, 0, P, P, P, None) == ARG          # window < 1
    assert f(P, 4, 32, P, 4097, 0, 0, 0, 0, P, P, P, None) == ARG       # window too large
    assert f(P, 4, 32, P, 64, 0, 0, 0, 8, P, P, P, None) == ARG         # offset % 16
    assert f(P, 0, 32, None, 64, 0, 0, 0, 0, None, None, None, None) == OK
    assert f(P, 4, 32, None, 64, 0, 0, 0, 0, P, P, P, None) == NULL
    assert f(P, 4, 32, PM, 64, 0, 0, 0, 0, P, P, P, None) == ALIGN


def test_host_validation_nvfp4(lib):
    q = lib.nvfp4_quantize
    assert q(P, 4, 24, P, 0, 0, 0, P, P, P, None) == SHAPE
    assert q(P, 4, 32, P, 0, 0, 8, P, P, P, None) == ARG                    # offset % 16
    assert q(P, 4, 32, P, 2, 0, 0, P, P, P, None) == ARG                    # use_sr not 0/1
    assert q(P, 4, 32, None, 0, 0, 0, P, P, P, None) == NULL
    assert q(P, 4, 32, P, 0, 0, 0, P, PM, P, None) == ALIGN
    assert q(P, 0, 32, P, 1, 0, 0, P, P, P, None) == OK
    q2 = lib.nvfp4_quantize_2d
    assert q2(P, 8, 32, P, P, P, P, None) == SHAPE
    assert q2(P, 16, 24, P, P, P, P, None) == SHAPE
    assert q2(P, 16, 32, P, P, None, P, None) == NULL
    assert q2(P, 0, 32, P, P, P, P, None) == OK
    t2 = lib.nvfp4_quantize_2d_t
    # w, N, K, amax, q, sb, qT, sbT, g, stream
    assert t2(P, 8, 32, P, P, P, P, P, P, None) == SHAPE                    # N % 16
    assert t2(P, 16, 24, P, P, P, P, P, P, None) == SHAPE                   # K % 16
    assert t2(P, 16, 0, P, P, P, P, P, P, None) == SHAPE
    assert t2(P, 16, 32, P, P, P, None, P, P, None) == NULL                  # qT
    assert t2(P, 16, 32, P, P, P, P, None, P, None) == NULL                  # sbT
    assert t2(P, 16, 32, P, P, P, PM, P, P, None) == ALIGN
    assert t2(P, 0, 32, P, P, P, None, None, P, None) == OK
    a = lib.nvfp4_amax
    assert a(P, -1, P, None) == SHAPE
    assert a(P, 4, None, None) == NULL
    assert a(PM, 4, P, None) == ALIGN


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    import fp8_quantization_gb300 as fq
    monkeypatch.setattr(fq, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(fq, "_lib", None)
    with pytest.raises(RuntimeError, match="libfq.so not found"):
        fq.abi()
