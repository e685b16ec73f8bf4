"""GPU: MXFP4 scales re-laid for a block-scaled MMA operand.

Byte-exact against the oracle (with a canary tail on the output), at small
ragged sizes and at the bench tensor's size; and fed, with the codes, to the
cuBLASLt block-scaled FP4 GEMM (where it runs), whose product
must match the product of the dequantized operands -- the consumer's own
check that the layout is the one it reads."""
import numpy as np
import pytest
import torch

import oracle
from fp8_quantization_gb300 import workloads

pytestmark = pytest.mark.gpu

CANARY = 0xA5


@pytest.fixture(scope="module")
def fq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import fp8_quantization_gb300 as m
    m.abi()
    return m


@pytest.mark.parametrize("M,K", [(1, 128), (127, 256), (128, 128), (129, 384), (1000, 7168),
                                 (3000, 2048)])
def test_mma_layout_matches_oracle(fq, M, K):
    rng = np.random.default_rng(M * 3 + K)
    s = rng.integers(0, 256, size=(M, K // 32), dtype=np.uint8)
    n = fq.mxfp4_scales_mma_bytes(M, K)
    raw = torch.full((n + 64,), CANARY, dtype=torch.uint8, device="cuda")
    out = fq.mxfp4_scales_mma_layout(torch.from_numpy(s).cuda(), raw[:n])
    ref = oracle.mxfp4_scales_mma_layout(s, M, K)
    assert np.array_equal(out.cpu().numpy(), ref)
    assert np.all(raw[n:].cpu().numpy() == CANARY), "write past the end of the output"


def test_mma_layout_bench_tensor(fq):
    """The scales of the 16384 x 7168 bench tensor (from the row quantizer)."""
    M, K = 16384, 7168
    x = torch.from_numpy(workloads.moe_dispatch(M, K, seed=0).view(np.int16)).cuda()
    q, s = fq.mxfp4_quantize_rows(x.view(torch.bfloat16))
    out = fq.mxfp4_scales_mma_layout(s)
    assert np.array_equal(out.cpu().numpy(), oracle.mxfp4_scales_mma_layout(s.cpu().numpy(), M, K))


def test_mma_layout_rejects_bad_k(fq):
    with pytest.raises(ValueError):
        fq.mxfp4_scales_mma_layout(torch.zeros((4, 3), dtype=torch.uint8, device="cuda"))


def _mx_operand(fq, rows, K, seed):
    """An MXFP4 operand with scales spread over many binades (a layout error
    moves scales between blocks and shows up as a large error)."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((rows, K)).astype(np.float32)
    x *= np.exp2(rng.integers(-6, 7, (rows, K // 32))).repeat(32, axis=1).astype(np.float32)
    bits = (x.view(np.uint32) >> 16).astype(np.uint16)          # BF16 by truncation
    xb = torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)
    q, s = fq.mxfp4_quantize_rows(xb)
    deq = fq.mxfp4_dequantize_rows(q, s).float()
    return q, s, deq


class _CublasLt:
    """The few cuBLASLt calls of one block-scaled FP4 GEMM, through ctypes
    (enum values from cublasLt.h / cublas_api.h / library_types.h)."""
    OP_N, OP_T = 0, 1
    COMPUTE_32F, R_32F, R_16BF, R_8F_E4M3, R_4F_E2M1 = 68, 0, 14, 28, 33
    TRANSA, TRANSB, A_SCALE_POINTER, B_SCALE_POINTER = 3, 4, 17, 18
    A_SCALE_MODE, B_SCALE_MODE, SCALE_VEC16_UE4M3, SCALE_VEC32_UE8M0 = 31, 32, 1, 2

    def __init__(self):
        import ctypes
        import ctypes.util
        self.c = ctypes
        lib = None
        for name in ("libcublasLt.so.13", "libcublasLt.so", ctypes.util.find_library("cublasLt")):
            if not name:
                continue
            try:
                lib = ctypes.CDLL(name)
                break
            except OSError:
                continue
        if lib is None:
            pytest.skip("cuBLASLt not found")
        self.lib = lib
        self.handle = ctypes.c_void_p()
        self.check(lib.cublasLtCreate(ctypes.byref(self.handle)), "cublasLtCreate")

    def check(self, st, what):
        if st != 0:
            raise RuntimeError(f"{what}: cuBLAS status {st}")

    def layout(self, dtype, rows, cols, ld):
        c = self.c
        h = c.c_void_p()
        self.check(self.lib.cublasLtMatrixLayoutCreate(c.byref(h), c.c_int(dtype), c.c_uint64(rows),
                                                       c.c_uint64(cols), c.c_int64(ld)),
                   "cublasLtMatrixLayoutCreate")
        return h

    def set_attr(self, desc, attr, value, ctype):
        c = self.c
        v = ctype(value)
        self.check(self.lib.cublasLtMatmulDescSetAttribute(desc, c.c_int(attr), c.byref(v),
                                                           c.c_size_t(c.sizeof(v))),
                   f"cublasLtMatmulDescSetAttribute({attr})")

    def mx_gemm(self, a8, sa_mma, b8, sb_mma, M, N, K, dtype=None, mode=None, alpha=1.0):
        """D [N, M] row-major (= M x N column-major) = A B^T with A = (a8, sa)
        [M, K] and B = (b8, sb) [N, K]: row-major E4M3 bytes, UE8M0 scales
        per 32 elements along K in the block-scaled MMA layout; fp32
        accumulation, BF16 output."""
        c = self.c
        desc = c.c_void_p()
        self.check(self.lib.cublasLtMatmulDescCreate(c.byref(desc), c.c_int(self.COMPUTE_32F),
                                                     c.c_int(self.R_32F)), "cublasLtMatmulDescCreate")
        self.set_attr(desc, self.TRANSA, self.OP_T, c.c_int32)
        self.set_attr(desc, self.TRANSB, self.OP_N, c.c_int32)
        dtype = self.R_8F_E4M3 if dtype is None else dtype
        mode = self.SCALE_VEC32_UE8M0 if mode is None else mode
        self.set_attr(desc, self.A_SCALE_MODE, mode, c.c_int32)
        self.set_attr(desc, self.B_SCALE_MODE, mode, c.c_int32)
        self.set_attr(desc, self.A_SCALE_POINTER, sa_mma.data_ptr(), c.c_void_p)
        self.set_attr(desc, self.B_SCALE_POINTER, sb_mma.data_ptr(), c.c_void_p)
        # A: K x M column-major (row-major [M, K]), op T; B: K x N column-major, op N
        la = self.layout(dtype, K, M, K)
        lb = self.layout(dtype, K, N, K)
        ld = self.layout(self.R_16BF, M, N, M)
        d = torch.zeros((N, M), dtype=torch.bfloat16, device="cuda")
        ws = torch.empty((64 << 20,), dtype=torch.uint8, device="cuda")
        alpha, beta = c.c_float(alpha), c.c_float(0.0)
        st = self.lib.cublasLtMatmul(self.handle, desc, c.byref(alpha), c.c_void_p(a8.data_ptr()), la,
                                     c.c_void_p(b8.data_ptr()), lb, c.byref(beta),
                                     c.c_void_p(d.data_ptr()), ld, c.c_void_p(d.data_ptr()), ld, None,
                                     c.c_void_p(ws.data_ptr()), c.c_size_t(ws.numel()),
                                     c.c_void_p(torch.cuda.current_stream().cuda_stream))
        torch.cuda.synchronize()
        for h in (la, lb, ld):
            self.lib.cublasLtMatrixLayoutDestroy(h)
        self.lib.cublasLtMatmulDescDestroy(desc)
        return st, d


# E4M3 bytes of the eight E2M1 magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6 (exact in E4M3)
E2M1_AS_E4M3 = [0x00, 0x30, 0x38, 0x3C, 0x40, 0x44, 0x48, 0x4C]


def _codes_as_e4m3(q):
    """MXFP4 codes [rows, K/2] (element 2i in the low nibble) as E4M3 bytes
    [rows, K] of the same values: an MXFP8 operand with the same scales."""
    lut = torch.tensor([b | (0x80 if c >= 8 else 0) for c in range(16)
                        for b in [E2M1_AS_E4M3[c & 7]]], dtype=torch.uint8, device=q.device)
    lo, hi = (q & 0xF).long(), (q >> 4).long()
    return torch.stack([lut[lo], lut[hi]], dim=-1).reshape(q.shape[0], q.shape[1] * 2).contiguous()


def test_block_scaled_gemm_reads_the_layout(fq):
    """cuBLASLt's block-scaled GEMM with 32-element blocks and UE8M0 scales
    (its MXFP8 recipe: the MXFP4 values re-expressed as E4M3 bytes, exact,
    with the same scales re-laid by this library) equals the product of the
    dequantized operands; with the row-major scales passed instead it does
    not."""
    M, N, K = 256, 384, 1024
    qa, sa, da = _mx_operand(fq, M, K, 1)
    qb, sb, db = _mx_operand(fq, N, K, 2)
    a8, b8 = _codes_as_e4m3(qa), _codes_as_e4m3(qb)
    lt = _CublasLt()
    st, got = lt.mx_gemm(a8, fq.mxfp4_scales_mma_layout(sa), b8, fq.mxfp4_scales_mma_layout(sb),
                         M, N, K)
    if st != 0:
        pytest.skip(f"cuBLASLt block-scaled GEMM unavailable here (status {st})")
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = False
    try:
        ref = (da @ db.t()).t()                      # [N, M], as D is laid out
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev
    scale = ref.abs() + 1e-3 * ref.abs().max()
    err = ((got.float() - ref).abs() / scale).max().item()
    assert err < 2 ** -6, err                        # BF16 output, fp32 accumulation
    st, wrong = lt.mx_gemm(a8, sa.reshape(-1), b8, sb.reshape(-1), M, N, K)
    assert st == 0
    werr = ((wrong.float() - ref).abs() / scale).max().item()
    assert werr > 0.1, werr


def _nvfp4_operand(fq, rows, K, seed):
    """An NVFP4 operand (round to nearest) and its decoded values: code x
    E4M3 block scale x the FP32 per-tensor decode scale g."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((rows, K)).astype(np.float32)
    x *= np.exp2(rng.integers(-4, 5, (rows, K // 16))).repeat(16, axis=1).astype(np.float32)
    bits = (x.view(np.uint32) >> 16).astype(np.uint16)
    xb = torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)
    amax = fq.nvfp4_amax(xb)
    q, sb, g = fq.nvfp4_quantize(xb, amax)
    mag = torch.tensor([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], device="cuda")
    codes = torch.stack([q & 0xF, q >> 4], dim=-1).reshape(rows, K).long()
    v = mag[codes & 7] * torch.where(codes >= 8, -1.0, 1.0)
    bscale = sb.view(torch.float8_e4m3fn).float().repeat_interleave(16, dim=1)
    return q, sb, float(g.item()), v * bscale * float(g.item())


def test_nvfp4_gemm_reads_codes_and_scales(fq):
    """cuBLASLt's NVFP4 GEMM (E2M1 data, UE4M3 scales per 16 elements in the
    same 128 x 4-tile layout, the per-tensor scales as alpha) on the 1x16
    quantizer's codes and block scales equals the product of the decoded
    operands: the nibble order, the scale bytes and the per-tensor scale mean
    what the consumer reads."""
    M, N, K = 256, 384, 1024
    qa, sa, ga, da = _nvfp4_operand(fq, M, K, 3)
    qb, sb, gb, db = _nvfp4_operand(fq, N, K, 4)
    lt = _CublasLt()
    # the layout is a byte permutation of a [rows, cols] scale matrix with
    # cols % 4 == 0: the NVFP4 scales [rows, K/16] go through the same call
    st, got = lt.mx_gemm(qa, fq.mxfp4_scales_mma_layout(sa), qb, fq.mxfp4_scales_mma_layout(sb),
                         M, N, K, dtype=lt.R_4F_E2M1, mode=lt.SCALE_VEC16_UE4M3, alpha=ga * gb)
    if st != 0:
        pytest.skip(f"cuBLASLt NVFP4 GEMM unavailable here (status {st})")
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = False
    try:
        ref = (da @ db.t()).t()
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev
    scale = ref.abs() + 1e-3 * ref.abs().max()
    err = ((got.float() - ref).abs() / scale).max().item()
    assert err < 2 ** -6, err
