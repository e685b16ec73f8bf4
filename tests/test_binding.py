"""The Python binding rejects bad tensors before anything reaches the library:
wrong dtype, layout or size of every input and output buffer (a buffer that
is too small would let a kernel read or write past its end), and tensors that
are not on the current CUDA device.  Runs on the CPU: size checks come first,
so CPU tensors of the wrong size raise ValueError without a GPU."""
import types

import pytest
import torch


@pytest.fixture(scope="module")
def fq():
    from fp8_quantization_gb300 import build
    build.build()
    import fp8_quantization_gb300 as m
    m.abi()
    return m


def u8(*shape):
    return torch.zeros(shape, dtype=torch.uint8)


def f32(*shape):
    return torch.zeros(shape, dtype=torch.float32)


def bf(*shape):
    return torch.zeros(shape, dtype=torch.bfloat16)


def raises(fn, match):
    with pytest.raises(ValueError, match=match):
        fn()


def test_mxfp4_and_rows(fq):
    x = bf(4, 64)
    raises(lambda: fq.mxfp4_quantize_rows(x, q=u8(4, 31), s=u8(4, 2)), "q must have")
    raises(lambda: fq.mxfp4_quantize_rows(x, q=u8(4, 32), s=u8(4, 1)), "s must have")
    raises(lambda: fq.mxfp4_quantize_rows(x.float()), "bfloat16")
    raises(lambda: fq.mxfp4_quantize_rows(bf(8, 64)[::2]), "contiguous")
    raises(lambda: fq.mxfp4_quantize_rows(x), "CUDA tensor")          # sizes fine, on the CPU
    q, s = u8(4, 64), u8(4, 4)
    raises(lambda: fq.fp4_to_fp8_rows(q, u8(4, 3)), "s must have shape")
    raises(lambda: fq.fp4_to_fp8_rows(q, s, y=u8(4, 127)), "y must have")
    raises(lambda: fq.fp4_to_fp8_rows(q, s, ys=f32(4, 2)), "ys must have")
    raises(lambda: fq.fp4_to_fp8_rows(q, s, ys=u8(4, 1)), "float32")
    raises(lambda: fq.mxfp4_dequantize_rows(q, u8(4, 5)), "s must have shape")
    raises(lambda: fq.mxfp4_dequantize_rows(q, s, out=bf(4, 64)), "out must have")


def test_cols_and_fused(fq):
    q, s = u8(300, 64), u8(300, 4)
    offs = torch.tensor([0, 100, 300], dtype=torch.int64)
    cap = fq.fp4_to_fp8_cols_scale_capacity(300, 2)
    raises(lambda: fq.fp4_to_fp8_cols(q, u8(300, 3), offs), "s must have shape")
    raises(lambda: fq.fp4_to_fp8_cols(q, u8(299, 4), offs), "s must have shape")
    raises(lambda: fq.fp4_to_fp8_cols(q, s, torch.tensor([0], dtype=torch.int64)), "G >= 1")
    raises(lambda: fq.fp4_to_fp8_cols(q, s, offs.int()), "int64")
    raises(lambda: fq.fp4_to_fp8_cols(q, s, offs, yT=u8(128, 299)), "yT must have")
    raises(lambda: fq.fp4_to_fp8_cols(q, s, offs, yT_scale=f32(cap - 1, 128)), "yT_scale must be")
    raises(lambda: fq.fp4_to_fp8_cols(q, s, offs, yT_scale=f32(cap, 64)), "yT_scale must be")
    raises(lambda: fq.fp4_to_fp8_cols(q, s, offs, dev_status=torch.zeros(0, dtype=torch.int32)),
           "dev_status")
    raises(lambda: fq.fp4_to_fp8_cols(q, s, offs), "CUDA tensor")
    x = bf(300, 128)
    for name, bad in (("q", u8(300, 63)), ("s", u8(300, 3)), ("y", u8(300, 127)),
                      ("ys", f32(299, 1)), ("yT", u8(128, 299))):
        raises(lambda: fq.bf16_to_mxfp4_fp8(x, offs, **{name: bad}), f"{name} must have")
    raises(lambda: fq.bf16_to_mxfp4_fp8(x, offs, yT_scale=f32(cap - 1, 128)), "yT_scale must be")
    raises(lambda: fq.bf16_to_mxfp4_fp8(x, offs), "CUDA tensor")


def test_nvfp4(fq):
    x, amax = bf(32, 64), f32(1)
    raises(lambda: fq.nvfp4_quantize(x, amax, q=u8(32, 31)), "q must have")
    raises(lambda: fq.nvfp4_quantize(x, amax, sb=u8(32, 3)), "sb must have")
    raises(lambda: fq.nvfp4_quantize(x, amax, g=f32(0)), "g must hold")
    raises(lambda: fq.nvfp4_quantize(x, f32(0)), "amax must hold")
    raises(lambda: fq.nvfp4_quantize(x, amax), "CUDA tensor")
    raises(lambda: fq.nvfp4_quantize_2d(x, amax, q=u8(32, 33)), "q must have")
    raises(lambda: fq.nvfp4_quantize_2d(x, amax, sb=u8(2, 3)), "sb must have")
    raises(lambda: fq.nvfp4_quantize_2d(x, amax), "CUDA tensor")
    raises(lambda: fq.nvfp4_quantize_2d_t(x, amax, qT=u8(64, 15)), "qT must have")
    raises(lambda: fq.nvfp4_quantize_2d_t(x, amax, sbT=u8(3, 2)), "sbT must have")
    raises(lambda: fq.nvfp4_quantize_2d_t(x, amax), "CUDA tensor")
    raises(lambda: fq.nvfp4_quantize_rht(x, amax, 0x1234, sb=u8(32, 5)), "sb must have")
    raises(lambda: fq.nvfp4_quantize_rht(x, amax, 0x1234), "CUDA tensor")
    raises(lambda: fq.nvfp4_amax(x, out=f32(0)), "out must hold")
    raises(lambda: fq.nvfp4_amax_rht(x, 1, out=f32(0)), "out must hold")
    h = torch.zeros(65, dtype=torch.int64)
    raises(lambda: fq.nvfp4_quantize_delayed(x, torch.zeros(1, dtype=torch.int64), 0), "history")
    raises(lambda: fq.nvfp4_quantize_delayed(x, h, 0, q=u8(32, 33)), "q must have")
    raises(lambda: fq.nvfp4_quantize_delayed(x, h, 0), "CUDA tensor")


def test_fp8_blocks(fq):
    x = bf(128, 256)
    raises(lambda: fq.fp8_quantize_1x128(x, y=u8(128, 255)), "y must have")
    raises(lambda: fq.fp8_quantize_1x128(x, s=f32(128, 3)), "s must have")
    raises(lambda: fq.fp8_quantize_128x128(x, s=f32(2, 2)), "s must have")
    raises(lambda: fq.fp8_quantize_128x128(x), "CUDA tensor")


def test_tensors_on_another_device_are_rejected(fq, monkeypatch):
    # A CUDA tensor on a device other than the current one (faked: this box
    # may have no GPU) is rejected before the call.
    monkeypatch.setattr(torch.cuda, "is_available", lambda: True)
    monkeypatch.setattr(torch.cuda, "current_device", lambda: 0)
    here = types.SimpleNamespace(is_cuda=True, device=types.SimpleNamespace(index=0))
    there = types.SimpleNamespace(is_cuda=True, device=types.SimpleNamespace(index=1))
    fq._on_device(a=here, b=None)
    with pytest.raises(ValueError, match="current device"):
        fq._on_device(a=here, b=there)
