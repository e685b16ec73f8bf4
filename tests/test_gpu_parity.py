"""GPU parity: every cast of libfq.so against the CPU oracle, byte for byte.

All outputs are integer codes or exact powers of two (MXFP4, FP4->FP8), or
IEEE binary32 results of the same operations in the same order (NVFP4), so
the bar is bit-exact everywhere.  Inputs are seeded synthetic tensors with the
shapes and distributions of the workloads; edge cases cover tails of every
tiling, empty and tiny groups, misaligned group starts, signed zeros,
subnormals, non-finite blocks and all exponent shifts.  Output buffers carry
canary tails that must stay untouched."""
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


def dev_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def canary_out(shape, dtype, extra=64):
    """Tensor of `shape` that is a view into a larger canary-filled buffer."""
    n = int(np.prod(shape))
    itemsize = torch.empty((), dtype=dtype).element_size()
    raw = torch.full(((n * itemsize + extra + 15) // 16 * 16,), CANARY, dtype=torch.uint8,
                     device="cuda")
    return raw, raw[: n * itemsize].view(dtype).view(shape)


def check_canary(raw, n_bytes):
    tail = raw[n_bytes:].cpu().numpy()
    assert np.all(tail == CANARY), "write past the end of an output"


def eq(gpu, ref, what=""):
    got = gpu.cpu().numpy()
    ref = np.asarray(ref)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    a, b = got.view(np.uint8), np.ascontiguousarray(ref).view(np.uint8)
    if not np.array_equal(a, b):
        idx = np.flatnonzero(a.ravel() != b.ravel())
        raise AssertionError(f"{what}: {idx.size} bytes differ, first at {idx[:8].tolist()}: "
                             f"gpu {a.ravel()[idx[:8]].tolist()} oracle {b.ravel()[idx[:8]].tolist()}")


# ------------------------------------------------------------------ MXFP4

def mx_inputs():
    rng = np.random.default_rng(21)
    out = {"pr1": workloads.pr1(), "tail": workloads.pr1(3, 96, seed=2),
           "one_row": workloads.pr1(1, 32, seed=3), "moe_small": workloads.moe_dispatch(97, 7168, 4)}
    x = rng.standard_normal((64, 256)).astype(np.float32)
    x[0, :32] = 0.0
    x[0, 32:64] = -0.0
    x[1, :32] = np.float32(2.0 ** -133) * rng.integers(0, 128, 32)
    x[2, 5] = np.nan
    x[3, 40] = np.inf
    x[4, 70] = -np.inf
    x[5, :32] = np.float32(3.3e38)
    x[6, :] *= np.float32(2.0 ** -126)
    out["special"] = workloads.bf16_bits(x)
    return out


def all_bf16_below_8_blocks():
    """Every BF16 value of magnitude < 8 (and its negative), 31 per block,
    each block led by 4.0 so that its scale is 1: the E2M1 conversion sees
    every value it can be given."""
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = workloads.bits_to_float(bits)
    keep = np.isfinite(vals) & (np.abs(vals) < 8)
    bits = bits[keep]
    nblk = (bits.size + 30) // 31
    pad = np.zeros(nblk * 31, dtype=np.uint16)
    pad[: bits.size] = bits
    blocks = np.empty((nblk, 32), dtype=np.uint16)
    blocks[:, 0] = 0x4080  # 4.0
    blocks[:, 1:] = pad.reshape(nblk, 31)
    nrow = (nblk + 7) // 8
    full = np.zeros((nrow * 8, 32), dtype=np.uint16)
    full[:nblk] = blocks
    full[nblk:, 0] = 0x4080
    return full.reshape(nrow, 256)


@pytest.mark.parametrize("name", ["pr1", "tail", "one_row", "moe_small", "special", "all_bf16"])
def test_mxfp4_quantize_rows(fq, name):
    bits = all_bf16_below_8_blocks() if name == "all_bf16" else mx_inputs()[name]
    M, K = bits.shape
    qraw, q = canary_out((M, K // 2), torch.uint8)
    sraw, s = canary_out((M, K // 32), torch.uint8)
    fq.mxfp4_quantize_rows(dev_bf16(bits), q, s)
    rq, rs = oracle.mxfp4_quantize_rows(bits)
    eq(q, rq, "q")
    eq(s, rs, "s")
    check_canary(qraw, M * K // 2)
    check_canary(sraw, M * K // 32)


def rand_mx(M, K, seed, spread=40, base=100, nan_frac=0.0):
    rng = np.random.default_rng(seed)
    q = rng.integers(0, 256, (M, K // 2), dtype=np.uint8)
    s = (base + rng.integers(0, spread, (M, K // 32))).astype(np.uint8)
    if nan_frac:
        s[rng.random(s.shape) < nan_frac] = 0xFF
    return q, s


@pytest.mark.parametrize("k", [0, 3, 6])
@pytest.mark.parametrize("shape,spread", [((256, 512), 3), ((37, 384), 40), ((5, 128), 255),
                                          ((300, 7168), 20)])
def test_fp4_to_fp8_rows(fq, k, shape, spread):
    M, K = shape
    q, s = rand_mx(M, K, seed=M + K + k, spread=spread, base=0 if spread == 255 else 100,
                   nan_frac=0.01)
    yraw, y = canary_out((M, K), torch.uint8)
    ysraw, ys = canary_out((M, K // 128), torch.float32)
    fq.fp4_to_fp8_rows(torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda(), k, y, ys)
    ry, rys = oracle.fp4_to_fp8_rows(q, s, k)
    eq(y, ry, "y")
    eq(ys, rys, "ys")
    check_canary(yraw, M * K)
    check_canary(ysraw, M * K // 128 * 4)


def test_fp4_to_fp8_rows_every_shift(fq):
    # every code against every shift d = 0..254 (scale pairs (S, e)), k = 0..6
    codes = np.arange(256, dtype=np.uint8)
    rows = []
    scales = []
    for d in range(255):
        rows.append(np.tile(codes, 1))              # 256 bytes = 512 codes = 4 FP8 blocks
        s = np.full((16,), 254 - d, dtype=np.uint8)
        s[0::4] = 254                               # first MX block of each FP8 block is the max
        scales.append(s)
    q = np.stack(rows)
    s = np.stack(scales)
    for k in range(7):
        y, ys = fq.fp4_to_fp8_rows(torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda(), k)
        ry, rys = oracle.fp4_to_fp8_rows(q, s, k)
        eq(y, ry, f"y k={k}")
        eq(ys, rys, f"ys k={k}")


# ------------------------------------------------------------------ FP4 -> FP8 cols

def run_cols(fq, q, s, offs, k, check=True):
    M, K = q.shape[0], q.shape[1] * 2
    G = offs.size - 1
    cap = oracle.fp4_to_fp8_cols_scale_capacity(M, G)
    yraw, yT = canary_out((K, M), torch.uint8)
    sraw = torch.full((K * cap * 4 + 64,), CANARY, dtype=torch.uint8, device="cuda")
    yTs = sraw[: K * cap * 4].view(torch.float32).view(cap, K)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    fq.fp4_to_fp8_cols(torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda(),
                       torch.from_numpy(offs).cuda(), k, yT, yTs, st)
    check_canary(yraw, K * M)
    check_canary(sraw, K * cap * 4)
    if check:
        ryT, ryTs = oracle.fp4_to_fp8_cols(q, s, offs, k)
        nb = int(((np.diff(offs) + 127) // 128).sum())
        eq(yT, ryT, "yT")
        eq(yTs[:nb], ryTs[:nb], "yT scales")
        # rows past the last block are never written
        tail = yTs[nb:].contiguous().view(torch.uint8).cpu().numpy()
        assert np.all(tail == CANARY)
        assert int(st.item()) == 0
    return yT, yTs, int(st.item())


COLS_CASES = {
    "g1_aligned": (512, 256, lambda M: np.array([0, M])),
    "g1_ragged_tail": (333, 128, lambda M: np.array([0, M])),
    "tiny_groups": (300, 256, lambda M: np.array([0, 0, 1, 1, 128, 129, 256, 257, 299, 300])),
    "sizes_127_128_129": (512, 128, lambda M: np.array([0, 127, 255, 384, 512])),
    "random_empty": (1000, 384, lambda M: workloads.random_group_offsets(M, 23, seed=4)),
    "zipf32": (4096, 256, lambda M: workloads.zipf_group_offsets(M, 32, 1.1, 3)),
    "m_not_mult_4": (1001, 128, lambda M: workloads.random_group_offsets(M, 9, seed=5)),
    "small_m": (3, 128, lambda M: np.array([0, 1, 3])),
    "many_groups": (2000, 128, lambda M: workloads.random_group_offsets(M, 1024, seed=6)),
    # 63 and 64 groups: the last count of the one-warp group set-up, the first of the CTA-wide one
    "groups_63": (3000, 256, lambda M: workloads.random_group_offsets(M, 63, seed=7)),
    "groups_64": (3000, 128, lambda M: workloads.random_group_offsets(M, 64, seed=8)),
    # M % 4 = 2 and 3: with K % 512 != 0 the last tokens' exponent rows are
    # patched into the four-row groups in shared memory (the last group
    # below lies wholly in those tokens)
    "tail_2": (1026, 384, lambda M: workloads.random_group_offsets(M, 7, seed=9)),
    "tail_3_last_group": (1003, 256, lambda M: np.array([0, 500, 1000, 1003])),
    "one_token_groups": (200, 128, lambda M: np.arange(M + 1)),
}


COLS_CASES["zipf32_k2048"] = (4096, 2048, lambda M: workloads.zipf_group_offsets(M, 32, 1.1, 8))
COLS_CASES["g1_m_mult_16_k1536"] = (640, 1536, lambda M: np.array([0, M]))


def cols_k(K, path):
    """K of a case on one of the exponent-row paths of the single pass:
    K % 512 == 0 (rows of K/32 bytes are a multiple of 16 bytes: tensor
    copies of rows) or not (tensor copies of four-row groups when M >= 4,
    the last M % 4 rows patched in shared memory, else 4-byte asynchronous
    copies; and a short last super-tile of fewer than four 128-feature
    blocks)."""
    if path == "k_mult_512":
        return (K + 511) // 512 * 512
    return K if K % 512 else K + 128


@pytest.mark.parametrize("case", sorted(COLS_CASES))
@pytest.mark.parametrize("k", [0, 6])
@pytest.mark.parametrize("path", ["k_mult_512", "k_not_mult_512"])
def test_fp4_to_fp8_cols(fq, case, k, path):
    M, K, mk = COLS_CASES[case]
    K = cols_k(K, path)
    assert fq.fp4_to_fp8_cols_launch_count(K) == 1
    offs = np.asarray(mk(M), dtype=np.int64)
    q, s = rand_mx(M, K, seed=M * 7 + K + k, spread=16, nan_frac=0.002)
    run_cols(fq, q, s, offs, k)


def test_fp4_to_fp8_cols_launch_count_in_a_fresh_process(fq):
    """The single pass is chosen even when the launch-count query is the
    process's first CUDA call (the tensor-map encoder lookup initialises the
    runtime itself, and a failed lookup is not kept)."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = ("import fp8_quantization_gb300 as fq; "
            "print(fq.fp4_to_fp8_cols_launch_count(512), fq.fp4_to_fp8_cols_launch_count(7168))")
    out = subprocess.run([sys.executable, "-c", code], cwd=root, capture_output=True, text=True,
                         timeout=300)
    assert out.returncode == 0, out.stderr
    assert out.stdout.split() == ["1", "1"]


@pytest.mark.parametrize("K", [128, 384, 640, 1920])
def test_fp4_to_fp8_cols_short_super_tiles(fq, K):
    """K % 512 != 0: every row's last super-tile has 1, 2 or 3 of its four
    128-feature blocks (the others are empty slots), on both sides of the
    walk-order switch (M = 70000: 547 windows), 32 Zipf groups, NaN scales;
    M % 4 != 0 patches the last rows of the four-row exponent groups."""
    for M in (3000, 3003, 70000, 70002):
        offs = np.asarray(workloads.zipf_group_offsets(M, 32, 1.1, K), dtype=np.int64)
        q, s = rand_mx(M, K, seed=M + K, spread=16, nan_frac=0.001)
        run_cols(fq, q, s, offs, 2)


@pytest.mark.parametrize("M", [65536, 66000, 66001, 66003])
@pytest.mark.parametrize("K", [1024, 1152])
def test_fp4_to_fp8_cols_walk_orders(fq, M, K):
    """Every output of the single pass on either side of the switch between
    its two configurations: up to 512 128-token windows the super-tiles
    (window x 512 features) are walked window fastest with 4 code stages,
    beyond that feature quad fastest with 2 (M % 16 != 0 included); K = 1152
    takes the four-row exponent groups (the last M % 4 rows patched in
    shared memory), with a short last super-tile.  32 Zipf groups, NaN
    scales."""
    assert fq.fp4_to_fp8_cols_launch_count(K) == 1
    offs = np.asarray(workloads.zipf_group_offsets(M, 32, 1.1, 11), dtype=np.int64)
    q, s = rand_mx(M, K, seed=M + 5, spread=16, nan_frac=0.0005)
    run_cols(fq, q, s, offs, 3)


@pytest.mark.parametrize("K", [256, 512])
def test_fp4_to_fp8_cols_malformed_offsets(fq, K):
    # malformed offsets: clamped in-kernel, status raised, nothing written
    # outside the outputs (canaries checked inside run_cols)
    M = 700
    q, s = rand_mx(M, K, seed=1)
    for offs in ([0, 800], [5, 300, 200, 700], [0, -40, 700], [0, 100, 699], [10, 20, 700]):
        _, _, st = run_cols(fq, q, s, np.array(offs, dtype=np.int64), 0, check=False)
        assert st == 1, offs
    # 40 groups (two offsets per lane of the one-warp set-up): a decrease at
    # an odd and at an even index, a negative and a too-large offset inside,
    # a last offset short of M; 80 groups for the CTA-wide set-up
    good = np.linspace(0, M, 41).astype(np.int64)
    for i, v in ((17, good[16] - 1), (18, good[17] - 1), (33, -3), (20, M + 5), (40, M - 1)):
        offs = good.copy()
        offs[i] = v
        _, _, st = run_cols(fq, q, s, offs, 0, check=False)
        assert st == 1, (i, v)
    good80 = np.linspace(0, M, 81).astype(np.int64)
    for i, v in ((41, good80[40] - 1), (80, M + 1)):
        offs = good80.copy()
        offs[i] = v
        _, _, st = run_cols(fq, q, s, offs, 0, check=False)
        assert st == 1, (i, v)
    _, _, st = run_cols(fq, q, s, good, 0)
    assert st == 0


# ------------------------------------------------------------------ fused MXFP4 forward cast

def fused_input(M, K, seed):
    """PR1-like BF16 values with special blocks: zero and negative-zero
    blocks, BF16 subnormals, NaN / Inf blocks, near-overflow values."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((M, K)).astype(np.float32)
    x *= np.exp2(rng.integers(-20, 20, (M, 1))).astype(np.float32)
    x[rng.random((M, K)) < 1e-3] *= 100.0
    if M >= 8:
        x[0, :32] = 0.0
        x[1, :32] = -0.0
        x[2, 32:64] *= np.float32(2.0 ** -130)
        x[3, 70] = np.nan
        x[4, 5] = np.inf
        x[5, 200 % K] = -np.inf
        x[6, :32] = np.float32(3.0e38)
    return workloads.bf16_bits(x)


FORWARD_CASTS = ["bf16_to_mxfp4_fp8", "bf16_to_mxfp4_fp8_single_pass"]


@pytest.mark.parametrize("entry", FORWARD_CASTS)
@pytest.mark.parametrize("case", sorted(COLS_CASES))
@pytest.mark.parametrize("kmod", ["k_mult_512", "k_not_mult_512"])
def test_bf16_to_mxfp4_fp8(fq, case, kmod, entry):
    """The one-call forward cast (two kernels, or the single-pass kernel)
    equals the oracle's MXFP4 -> FP8 rows and MXFP4 -> FP8 cols, byte for
    byte, with canaries on every output."""
    M, K, mk = COLS_CASES[case]
    K = cols_k(K, kmod)
    offs = np.asarray(mk(M), dtype=np.int64)
    check_fused(fq, M, K, offs, (M + K) % 7, fused_input(M, K, seed=M + 3 * K), entry)


@pytest.mark.parametrize("entry", FORWARD_CASTS)
def test_bf16_to_mxfp4_fp8_above_512_windows(fq, entry):
    """The one-call forward cast on 66000 tokens (516 windows: the transposed
    kernel's large-tensor configuration) x 1024 features, 32 Zipf groups."""
    M, K = 66000, 1024
    offs = np.asarray(workloads.zipf_group_offsets(M, 32, 1.1, 13), dtype=np.int64)
    check_fused(fq, M, K, offs, 2, fused_input(M, K, seed=17), entry)


@pytest.mark.parametrize("entry", FORWARD_CASTS)
def test_bf16_to_mxfp4_fp8_malformed_offsets(fq, entry):
    """Malformed group offsets are clamped in the kernel, reported through
    dev_status, and nothing is written outside the outputs."""
    M, K = 700, 384
    bits = fused_input(M, K, seed=23)
    x = dev_bf16(bits)
    for offs in ([0, 800], [5, 300, 200, 700], [0, -40, 700], [0, 100, 699], [10, 20, 700]):
        offs = np.array(offs, dtype=np.int64)
        G = offs.size - 1
        cap = oracle.fp4_to_fp8_cols_scale_capacity(M, G)
        outs = [canary_out(shape, dt) for shape, dt in (
            ((M, K // 2), torch.uint8), ((M, K // 32), torch.uint8), ((M, K), torch.uint8),
            ((M, K // 128), torch.float32), ((K, M), torch.uint8), ((cap, K), torch.float32))]
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        getattr(fq, entry)(x, torch.from_numpy(offs).cuda(), 0, *[o[1] for o in outs],
                           dev_status=st)
        for (raw, view), n in zip(outs, (M * K // 2, M * K // 32, M * K, M * K // 32, K * M,
                                         cap * K * 4)):
            check_canary(raw, n)
        assert int(st.item()) == 1, offs
        # the row outputs do not depend on the groups
        rq, rs = oracle.mxfp4_quantize_rows(bits)
        eq(outs[0][1], rq, "q")
        eq(outs[1][1], rs, "s")


def check_fused(fq, M, K, offs, k, bits, entry="bf16_to_mxfp4_fp8"):
    G = offs.size - 1
    cap = oracle.fp4_to_fp8_cols_scale_capacity(M, G)
    qraw, q = canary_out((M, K // 2), torch.uint8)
    sraw, s = canary_out((M, K // 32), torch.uint8)
    yraw, y = canary_out((M, K), torch.uint8)
    ysraw, ys = canary_out((M, K // 128), torch.float32)
    yTraw, yT = canary_out((K, M), torch.uint8)
    yTsraw = torch.full((K * cap * 4 + 64,), CANARY, dtype=torch.uint8, device="cuda")
    yTs = yTsraw[: K * cap * 4].view(torch.float32).view(cap, K)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    getattr(fq, entry)(dev_bf16(bits), torch.from_numpy(offs).cuda(), k, q, s, y, ys, yT, yTs, st)
    for raw, n in ((qraw, M * K // 2), (sraw, M * K // 32), (yraw, M * K), (ysraw, M * K // 32),
                   (yTraw, K * M), (yTsraw, K * cap * 4)):
        check_canary(raw, n)
    rq, rs = oracle.mxfp4_quantize_rows(bits)
    ry, rys = oracle.fp4_to_fp8_rows(rq, rs, k)
    ryT, ryTs = oracle.fp4_to_fp8_cols(rq, rs, offs, k)
    nb = int(((np.diff(offs) + 127) // 128).sum())
    eq(q, rq, "q")
    eq(s, rs, "s")
    eq(y, ry, "y")
    eq(ys, rys, "ys")
    eq(yT, ryT, "yT")
    eq(yTs[:nb], ryTs[:nb], "yT scales")
    assert np.all(yTs[nb:].contiguous().view(torch.uint8).cpu().numpy() == CANARY)
    assert int(st.item()) == 0


# ------------------------------------------------------------------ NVFP4

def test_nvfp4_amax(fq):
    for shape, seed in (((64, 512), 1), ((3, 7), 2), ((1, 1), 3), ((1000, 1000), 4)):
        bits = workloads.nvfp4_act(*shape, seed=seed)
        a = fq.nvfp4_amax(dev_bf16(bits))
        assert a.item() == float(oracle.nvfp4_amax(bits))
    x = workloads.bits_to_float(workloads.nvfp4_act(33, 17, seed=5)).copy()
    x[7, 3] = np.nan
    assert np.isnan(fq.nvfp4_amax(dev_bf16(workloads.bf16_bits(x))).item())
    x[7, 3] = -np.inf
    assert fq.nvfp4_amax(dev_bf16(workloads.bf16_bits(x))).item() == np.inf
    empty = torch.empty((0,), dtype=torch.bfloat16, device="cuda")
    assert fq.nvfp4_amax(empty).item() == 0.0


NV_CASES = {"act": (128, 512, workloads.nvfp4_act), "tail": (3, 48, workloads.nvfp4_act),
            "k16": (40, 16, workloads.nvfp4_act), "wide": (9, 14336, workloads.nvfp4_act),
            "weight": (64, 4096, workloads.nvfp4_weight)}


@pytest.mark.parametrize("case", sorted(NV_CASES))
@pytest.mark.parametrize("sr", [False, True])
def test_nvfp4_quantize(fq, case, sr):
    M, K, gen = NV_CASES[case]
    bits = gen(M, K, seed=M + K)
    x = dev_bf16(bits)
    amax = fq.nvfp4_amax(x)
    ramax = oracle.nvfp4_amax(bits)
    qraw, q = canary_out((M, K // 2), torch.uint8)
    sraw, sb = canary_out((M, K // 16), torch.uint8)
    g = torch.empty(1, dtype=torch.float32, device="cuda")
    for seed, offset in ((1234, 0), (2**63 + 77, 16 * 1001)):
        fq.nvfp4_quantize(x, amax, use_sr=sr, seed=seed, offset=offset, q=q, sb=sb, g=g)
        rq, rsb, rg = oracle.nvfp4_quantize(bits, ramax, use_sr=sr, seed=seed, offset=offset)
        eq(q, rq, "q")
        eq(sb, rsb, "sb")
        assert g.item() == float(rg)
        check_canary(qraw, M * K // 2)
        check_canary(sraw, M * K // 16)


def test_nvfp4_special_values(fq):
    rng = np.random.default_rng(3)
    x = rng.standard_normal((32, 64)).astype(np.float32)
    x[0, :16] = 0.0
    x[1, :16] = -0.0
    x[2, :16] = np.float32(2.0 ** -130)
    x[3, :] *= np.float32(1e-30)
    x[4, 5] = np.nan                    # NaN blocks take the NaN scale (R21)
    x[5, 20] = -np.inf
    x[6, 33] = np.inf
    bits = workloads.bf16_bits(x)
    bits[7, 50] = 0xFFC1                # a negative NaN with a payload
    finite = bits.copy()
    finite[4, 5] = finite[5, 20] = finite[6, 33] = finite[7, 50] = 0
    for A in (float(oracle.nvfp4_amax(finite)), 0.0, 1e-38, 3.0e38, float("inf"), float("nan")):
        amax = torch.tensor([A], dtype=torch.float32, device="cuda")
        for sr in (False, True):
            q, sb, g = fq.nvfp4_quantize(dev_bf16(bits), amax, use_sr=sr, seed=9)
            rq, rsb, rg = oracle.nvfp4_quantize(bits, np.float32(A), use_sr=sr, seed=9)
            eq(q, rq, f"q A={A}")
            eq(sb, rsb, f"sb A={A}")


def test_nvfp4_block_scale_every_bf16_amax(fq):
    # every positive finite BF16 value as a block maximum, under three
    # per-tensor scales: drives the E4M3 block-scale conversion over its range
    bits = np.arange(1, 0x7F80, dtype=np.uint32).astype(np.uint16)
    bits = np.concatenate([bits, np.full((-bits.size) % 16, 0x3F80, dtype=np.uint16)])
    nblk = bits.size
    x = np.zeros((nblk, 16), dtype=np.uint16)
    x[:, 0] = bits
    x[:, 1:] = (bits[:, None] >> 1).astype(np.uint16)
    x = x.reshape(-1, 256)
    for A in (1.0, 3.0e38, 1.0e-20):
        amax = torch.tensor([A], dtype=torch.float32, device="cuda")
        q, sb, g = fq.nvfp4_quantize(dev_bf16(x), amax)
        rq, rsb, rg = oracle.nvfp4_quantize(x, np.float32(A))
        eq(sb, rsb, f"sb A={A}")
        eq(q, rq, f"q A={A}")


@pytest.mark.parametrize("shape", [(16, 16), (48, 272), (64, 4096), (32, 528)])
def test_nvfp4_quantize_2d(fq, shape):
    N, K = shape
    bits = workloads.nvfp4_weight(N, K, seed=N + K)
    w = dev_bf16(bits)
    amax = fq.nvfp4_amax(w)
    qraw, q = canary_out((N, K // 2), torch.uint8)
    sraw, sb = canary_out((N // 16, K // 16), torch.uint8)
    g = torch.empty(1, dtype=torch.float32, device="cuda")
    fq.nvfp4_quantize_2d(w, amax, q, sb, g)
    rq, rsb, rg = oracle.nvfp4_quantize_2d(bits, oracle.nvfp4_amax(bits))
    eq(q, rq, "q")
    eq(sb, rsb, "sb")
    assert g.item() == float(rg)
    check_canary(qraw, N * K // 2)
    check_canary(sraw, N * K // 256)


@pytest.mark.parametrize("shape", [(16, 16), (32, 48), (48, 256), (64, 272), (256, 512),
                                   (1024, 1040), (4096, 768)])
def test_nvfp4_quantize_2d_t(fq, shape):
    """The FPROP operand and the transposed DGRAD operand in one call, against
    the oracle, with canaries on all four outputs."""
    N, K = shape
    bits = workloads.nvfp4_weight(N, K, seed=N * 3 + K)
    w = dev_bf16(bits)
    amax = fq.nvfp4_amax(w)
    qraw, q = canary_out((N, K // 2), torch.uint8)
    sraw, sb = canary_out((N // 16, K // 16), torch.uint8)
    qTraw, qT = canary_out((K, N // 2), torch.uint8)
    sTraw, sbT = canary_out((K // 16, N // 16), torch.uint8)
    g = torch.empty(1, dtype=torch.float32, device="cuda")
    fq.nvfp4_quantize_2d_t(w, amax, q, sb, qT, sbT, g)
    rq, rsb, rqT, rsbT, rg = oracle.nvfp4_quantize_2d_t(bits, oracle.nvfp4_amax(bits))
    eq(q, rq, "q")
    eq(sb, rsb, "sb")
    eq(qT, rqT, "qT")
    eq(sbT, rsbT, "sbT")
    assert g.item() == float(rg)
    for raw, n in ((qraw, N * K // 2), (sraw, N * K // 256), (qTraw, N * K // 2),
                   (sTraw, N * K // 256)):
        check_canary(raw, n)


def test_nvfp4_quantize_2d_t_special_tiles(fq):
    """Zero and negative-zero tiles, BF16 subnormals, infinities, values near
    the BF16 maximum and a tile far below the tensor maximum, through both
    operands."""
    rng = np.random.default_rng(11)
    N, K = 64, 96
    x = rng.normal(0.0, 0.02, (N, K)).astype(np.float32)
    x[:16, :16] = 0.0
    x[16:32, :16] = -0.0
    x[:16, 16:32] = np.float32(2.0 ** -130) * rng.integers(-60, 61, (16, 16))
    x[32, 40] = np.inf
    x[50, 70] = -np.inf
    x[48:64, 80:96] = np.float32(3.0e38) * rng.uniform(-1, 1, (16, 16))
    x[32:48, :16] *= np.float32(1e-20)
    x[20, 60] = np.nan
    bits = workloads.bf16_bits(x)
    bits[40, 90] = 0xFF81               # a negative NaN with a payload
    for A in (float(oracle.nvfp4_amax(bits)), 1.0, 3.0e38, float("inf"), float("nan")):
        amax = torch.tensor([A], dtype=torch.float32, device="cuda")
        q, sb, qT, sbT, g = fq.nvfp4_quantize_2d_t(dev_bf16(bits), amax)
        rq, rsb, rqT, rsbT, rg = oracle.nvfp4_quantize_2d_t(bits, np.float32(A))
        for got, ref, what in ((q, rq, "q"), (sb, rsb, "sb"), (qT, rqT, "qT"), (sbT, rsbT, "sbT")):
            eq(got, ref, f"{what} A={A}")
        assert g.item() == float(rg) or (np.isnan(g.item()) and np.isnan(rg))
        q2, sb2, _ = fq.nvfp4_quantize_2d(dev_bf16(bits), amax)
        eq(q2, rq, f"2d q A={A}")
        eq(sb2, rsb, f"2d sb A={A}")


def test_errors_are_reported(fq):
    x = torch.zeros((4, 33), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fq.FQError, match="FQ_ERR_SHAPE"):
        fq.mxfp4_quantize_rows(x)
    q = torch.zeros((4, 64), dtype=torch.uint8, device="cuda")
    s = torch.zeros((4, 4), dtype=torch.uint8, device="cuda")
    with pytest.raises(fq.FQError, match="FQ_ERR_ARG"):
        fq.fp4_to_fp8_rows(q, s, 7)
    raw = torch.zeros(4 * 128 + 1, dtype=torch.uint8, device="cuda")
    with pytest.raises(fq.FQError, match="FQ_ERR_ALIGN"):
        fq.fp4_to_fp8_rows(q, s, 0, y=raw[1:].view(4, 128))


# ------------------------------------------------------------------ NVFP4 with the Hadamard transform

RHT_CASES = {"act": (128, 512, workloads.nvfp4_act), "tail": (3, 48, workloads.nvfp4_act),
             "k16": (40, 16, workloads.nvfp4_act), "wide": (9, 14336, workloads.nvfp4_act),
             "weight": (64, 4096, workloads.nvfp4_weight)}


@pytest.mark.parametrize("case", sorted(RHT_CASES))
@pytest.mark.parametrize("sr", [False, True])
@pytest.mark.parametrize("mask", [0x0000, 0xA5C3, 0xFFFF])
def test_nvfp4_quantize_rht(fq, case, sr, mask):
    M, K, gen = RHT_CASES[case]
    bits = gen(M, K, seed=M + K + mask)
    x = dev_bf16(bits)
    amax = fq.nvfp4_amax_rht(x, mask)
    ramax = oracle.nvfp4_amax_rht(bits, mask)
    assert amax.item() == float(ramax)
    qraw, q = canary_out((M, K // 2), torch.uint8)
    sraw, sb = canary_out((M, K // 16), torch.uint8)
    g = torch.empty(1, dtype=torch.float32, device="cuda")
    for seed, offset in ((4321, 0), (2**64 - 5, 16 * 777)):
        fq.nvfp4_quantize_rht(x, amax, mask, use_sr=sr, seed=seed, offset=offset, q=q, sb=sb, g=g)
        rq, rsb, rg = oracle.nvfp4_quantize_rht(bits, ramax, mask, use_sr=sr, seed=seed,
                                                offset=offset)
        eq(q, rq, "q")
        eq(sb, rsb, "sb")
        assert g.item() == float(rg)
        check_canary(qraw, M * K // 2)
        check_canary(sraw, M * K // 16)


def test_nvfp4_rht_special_values(fq):
    """Signed zeros, BF16 subnormals (their transform reaches binary32
    subnormals), huge finite values, all-zero blocks, and a NaN propagating
    through the transformed amax."""
    rng = np.random.default_rng(9)
    x = rng.standard_normal((16, 64)).astype(np.float32)
    x[0, :16] = 0.0
    x[1, :16] = -0.0
    x[2, :16] = np.float32(2.0 ** -130) * rng.integers(-64, 65, 16)
    x[3, 16:32] = np.float32(2.0 ** 120) * rng.standard_normal(16)
    x[4, :] = np.float32(2.0 ** -120)
    bits = workloads.bf16_bits(x)
    for mask in (0, 0x1111, 0xFFFF):
        xd = dev_bf16(bits)
        amax = fq.nvfp4_amax_rht(xd, mask)
        ra = oracle.nvfp4_amax_rht(bits, mask)
        assert amax.item() == float(ra)
        for sr in (False, True):
            q, sb, g = fq.nvfp4_quantize_rht(xd, amax, mask, use_sr=sr, seed=5)
            rq, rsb, rg = oracle.nvfp4_quantize_rht(bits, ra, mask, use_sr=sr, seed=5)
            eq(q, rq, f"q mask={mask:x} sr={sr}")
            eq(sb, rsb, f"sb mask={mask:x} sr={sr}")
    bad = bits.copy()
    bad[5, 3] = 0x7FC0
    assert np.isnan(fq.nvfp4_amax_rht(dev_bf16(bad), 0x2222).item())
    # a NaN block of the transform takes the NaN scale, its NaN values code
    # 7 (R21), under a finite, an infinite and a NaN per-tensor amax
    for A in (float(oracle.nvfp4_amax_rht(bits, 0x2222)), float("inf"), float("nan")):
        amax = torch.tensor([A], dtype=torch.float32, device="cuda")
        for sr in (False, True):
            q, sb, g = fq.nvfp4_quantize_rht(dev_bf16(bad), amax, 0x2222, use_sr=sr, seed=6)
            rq, rsb, rg = oracle.nvfp4_quantize_rht(bad, np.float32(A), 0x2222, use_sr=sr, seed=6)
            eq(q, rq, f"nan block q A={A} sr={sr}")
            eq(sb, rsb, f"nan block sb A={A} sr={sr}")
    empty = torch.empty((0,), dtype=torch.bfloat16, device="cuda")
    assert fq.nvfp4_amax_rht(empty, 1).item() == 0.0


# ------------------------------------------------------------------ FP8 blocks and MXFP4 dequantization

def fp8_input(M, K, seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((M, K)).astype(np.float32)
    x *= np.exp2(rng.integers(-40, 40, (M, 1))).astype(np.float32)
    x[rng.random((M, K)) < 2e-3] *= 1000.0
    if M >= 6 and K >= 256:
        x[0, :128] = 0.0
        x[1, :128] = -0.0
        x[2, 128:256] = np.float32(2.0 ** -130) * rng.integers(-100, 101, 128)
        x[3, 5] = np.nan
        x[4, 200] = np.inf
        x[5, 130] = np.float32(3.3e38)
    return workloads.bf16_bits(x)


@pytest.mark.parametrize("shape", [(256, 512), (3, 128), (1, 7168), (130, 384), (512, 1024)])
def test_fp8_quantize_1x128(fq, shape):
    M, K = shape
    bits = fp8_input(M, K, seed=M + K)
    yraw, y = canary_out((M, K), torch.uint8)
    sraw, sc = canary_out((M, K // 128), torch.float32)
    fq.fp8_quantize_1x128(dev_bf16(bits), y, sc)
    ry, rs = oracle.fp8_quantize_blocks(bits, 1)
    eq(y, ry, "codes")
    eq(sc, rs, "scales")
    check_canary(yraw, M * K)
    check_canary(sraw, M * K // 128 * 4)


@pytest.mark.parametrize("shape", [(128, 128), (256, 512), (384, 1024), (128, 7168)])
def test_fp8_quantize_128x128(fq, shape):
    N, K = shape
    bits = fp8_input(N, K, seed=N * 3 + K)
    yraw, y = canary_out((N, K), torch.uint8)
    sraw, sc = canary_out((N // 128, K // 128), torch.float32)
    fq.fp8_quantize_128x128(dev_bf16(bits), y, sc)
    ry, rs = oracle.fp8_quantize_blocks(bits, 128)
    eq(y, ry, "codes")
    eq(sc, rs, "scales")
    check_canary(yraw, N * K)
    check_canary(sraw, N * K // 16384 * 4)


def test_mxfp4_dequantize_every_code_and_scale(fq):
    q = np.tile(np.arange(256, dtype=np.uint8), (256, 1))
    s = np.repeat(np.arange(256, dtype=np.uint8)[:, None], 16, axis=1)
    oraw, out = canary_out((256, 512), torch.bfloat16)
    fq.mxfp4_dequantize_rows(torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda(), out)
    eq(out.view(torch.uint16), oracle.mxfp4_dequantize_rows(q, s), "bf16")
    check_canary(oraw, 256 * 512 * 2)


@pytest.mark.parametrize("shape", [(3, 32), (97, 7168), (64, 96)])
def test_mxfp4_dequantize_roundtrip_shapes(fq, shape):
    M, K = shape
    bits = workloads.moe_dispatch(M, K, seed=M)
    q, s = oracle.mxfp4_quantize_rows(bits)
    out = fq.mxfp4_dequantize_rows(torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda())
    eq(out.view(torch.uint16), oracle.mxfp4_dequantize_rows(q, s), "bf16")


# ------------------------------------------------------------------ delayed scaling (Max-Window)

def spiky_tensor(rng, M, K, t):
    """Student-t rows scaled per step, with occasional spikes, so the window
    estimate both trails and exceeds the current amax."""
    x = rng.standard_t(4, (M, K)).astype(np.float32) * np.float32(np.exp2(rng.uniform(-6, 6)))
    if t % 11 == 3:
        x[0, 0] = np.float32(2.0 ** 40)
    return workloads.bf16_bits(x)


@pytest.mark.parametrize("W", [1, 8, 64])
def test_nvfp4_quantize_delayed_sequence(fq, W):
    rng = np.random.default_rng(W)
    M, K = 48, 320
    hist_d = fq.amax_history(W)
    hist = np.zeros(W + 1, dtype=np.uint64)
    for t in range(2 * W + 30):
        bits = spiky_tensor(rng, M, K, t)
        sr = t % 3 == 0
        q, sb, g = fq.nvfp4_quantize_delayed(dev_bf16(bits), hist_d, t, use_sr=sr, seed=17 + t,
                                             offset=16 * t)
        rq, rsb, rg, hist = oracle.nvfp4_quantize_delayed(bits, hist, W, t, use_sr=sr,
                                                          seed=17 + t, offset=16 * t)
        eq(q, rq, f"q t={t}")
        eq(sb, rsb, f"sb t={t}")
        assert g.item() == float(rg), t
        assert np.array_equal(hist_d.cpu().numpy().view(np.uint64), hist), f"history t={t}"


def test_nvfp4_quantize_delayed_nan_step(fq):
    """A step whose tensor holds NaN records a NaN amax; while it stays in the
    window the estimate is NaN, so g = 1 (A > 0 fails), and the NaN step's own
    blocks take the NaN scale (R21)."""
    rng = np.random.default_rng(8)
    W = 3
    hist_d = fq.amax_history(W)
    hist = np.zeros(W + 1, dtype=np.uint64)
    for t in range(9):
        bits = spiky_tensor(rng, 32, 64, t)
        if t == 2:
            bits[5, 9] = 0x7FC0
        q, sb, g = fq.nvfp4_quantize_delayed(dev_bf16(bits), hist_d, t, use_sr=t % 2 == 1,
                                             seed=3 + t)
        rq, rsb, rg, hist = oracle.nvfp4_quantize_delayed(bits, hist, W, t, use_sr=t % 2 == 1,
                                                          seed=3 + t)
        eq(q, rq, f"q t={t}")
        eq(sb, rsb, f"sb t={t}")
        assert g.item() == float(rg), t
        assert np.array_equal(hist_d.cpu().numpy().view(np.uint64), hist), f"history t={t}"
        if 3 <= t <= 2 + W:
            assert g.item() == 1.0


def test_nvfp4_quantize_delayed_tag_wrap(fq):
    rng = np.random.default_rng(5)
    W = 4
    hist_d = fq.amax_history(W)
    hist = np.zeros(W + 1, dtype=np.uint64)
    for i in range(12):
        t = (2**32 - 6 + i) % 2**32
        bits = spiky_tensor(rng, 16, 64, i)
        q, sb, g = fq.nvfp4_quantize_delayed(dev_bf16(bits), hist_d, t)
        rq, rsb, rg, hist = oracle.nvfp4_quantize_delayed(bits, hist, W, t)
        eq(q, rq, f"q i={i}")
        eq(sb, rsb, f"sb i={i}")
        assert g.item() == float(rg)
        assert np.array_equal(hist_d.cpu().numpy().view(np.uint64), hist)
