"""GPU parity at the workloads' full sizes, called the way the benchmark calls
the library (one stream, caller-allocated outputs, the same entry points and
arguments).

Where the CPU oracle finishes in seconds every output byte is compared; for
the largest bandwidth-sweep tensors the comparison runs on seeded samples the
oracle computes on their own: whole rows for the row casts (rows are
independent), whole 128-token windows for the transposed cast with one group
(its blocks are then aligned to multiples of 128, so a window's output depends
only on the window's tokens)."""
import numpy as np
import pytest
import torch

import oracle
from fp8_quantization_gb300 import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import fp8_quantization_gb300 as m
    m.abi()
    return m


def dev_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def eq(gpu, ref, what):
    got = gpu.contiguous().cpu().numpy() if isinstance(gpu, torch.Tensor) else np.asarray(gpu)
    ref = np.ascontiguousarray(ref)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    a, b = got.view(np.uint8), ref.view(np.uint8)
    if not np.array_equal(a, b):
        idx = np.flatnonzero(a.ravel() != b.ravel())
        raise AssertionError(f"{what}: {idx.size} bytes differ, first at {idx[:8].tolist()}")


def cols_full(fq, q_d, s_d, offs, k):
    M, K = q_d.shape[0], q_d.shape[1] * 2
    G = offs.size - 1
    cap = fq.fp4_to_fp8_cols_scale_capacity(M, G)
    yT = torch.empty((K, M), dtype=torch.uint8, device="cuda")
    yTs = torch.empty((cap, K), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    fq.fp4_to_fp8_cols(q_d, s_d, torch.from_numpy(offs).cuda(), k, yT, yTs, st)
    assert int(st.item()) == 0
    return yT, yTs


def test_moe_dispatch_16384x7168_all_casts(fq):
    """The benchmark's workload and call sequence, every output compared."""
    M, K, G = 16384, 7168, 32
    bits = workloads.moe_dispatch(M, K, seed=0)
    offs = workloads.zipf_group_offsets(M, G, 1.1, 0)
    x = dev_bf16(bits)
    q, s = fq.mxfp4_quantize_rows(x)
    y, ys = fq.fp4_to_fp8_rows(q, s, 0)
    yT, yTs = cols_full(fq, q, s, offs, 0)
    amax = fq.nvfp4_amax(x)
    q4, sb4, g4 = fq.nvfp4_quantize(x, amax, use_sr=True, seed=1000, offset=0)
    q2, sb2, g2 = fq.nvfp4_quantize_2d(x, amax)
    fused = fq.bf16_to_mxfp4_fp8(x, torch.from_numpy(offs).cuda(), 0)

    rq, rs = oracle.mxfp4_quantize_rows(bits)
    eq(q, rq, "mxfp4 q")
    eq(s, rs, "mxfp4 s")
    ry, rys = oracle.fp4_to_fp8_rows(rq, rs, 0)
    eq(y, ry, "fp8 rows y")
    eq(ys, rys, "fp8 rows scales")
    ryT, ryTs = oracle.fp4_to_fp8_cols(rq, rs, offs, 0)
    nb = int(((np.diff(offs) + 127) // 128).sum())
    eq(yT, ryT, "fp8 cols yT")
    eq(yTs[:nb], ryTs[:nb], "fp8 cols scales")
    for got, ref, what in zip(fused[:5], (rq, rs, ry, rys, ryT), ("q", "s", "y", "ys", "yT")):
        eq(got, ref, "fused " + what)
    eq(fused[5][:nb], ryTs[:nb], "fused yT scales")
    single = fq.bf16_to_mxfp4_fp8_single_pass(x, torch.from_numpy(offs).cuda(), 0)
    for got, want in zip(single[:5], fused[:5]):
        assert torch.equal(got, want), "single-pass forward cast"
    assert torch.equal(single[5][:nb], fused[5][:nb]), "single-pass forward cast yT scales"
    del single
    ra = oracle.nvfp4_amax(bits)
    assert amax.item() == float(ra)
    rq4, rsb4, rg4 = oracle.nvfp4_quantize(bits, ra, use_sr=True, seed=1000, offset=0)
    eq(q4, rq4, "nvfp4 SR q")
    eq(sb4, rsb4, "nvfp4 SR scales")
    assert g4.item() == float(rg4)
    rq2, rsb2, rg2 = oracle.nvfp4_quantize_2d(bits, ra)
    eq(q2, rq2, "nvfp4 2d q")
    eq(sb2, rsb2, "nvfp4 2d scales")
    assert g2.item() == float(rg2)


def test_chained_steps_alternating_inputs(fq):
    """The bench step's six calls repeated 24 times on one stream with no host
    synchronisation, the input alternating between two tensors (and the
    ragged offsets between two splits), so that every kernel overlaps the
    launch of the next.  The outputs must be exactly those of the last step's
    input computed alone (a kernel that read a buffer before the previous
    kernel finished writing it would mix the two inputs)."""
    M, K, G = 16384, 7168, 32
    xs = [dev_bf16(workloads.moe_dispatch(M, K, seed=sd)) for sd in (0, 5)]
    offs = [torch.from_numpy(workloads.zipf_group_offsets(M, G, 1.1, sd)).cuda() for sd in (0, 5)]
    cap = fq.fp4_to_fp8_cols_scale_capacity(M, G)
    dev = torch.device("cuda")

    def outputs():
        u8 = dict(dtype=torch.uint8, device=dev)
        f32 = dict(dtype=torch.float32, device=dev)
        return dict(q=torch.zeros((M, K // 2), **u8), s=torch.zeros((M, K // 32), **u8),
                    y=torch.zeros((M, K), **u8), ys=torch.zeros((M, K // 128), **f32),
                    yT=torch.zeros((K, M), **u8), yTs=torch.zeros((cap, K), **f32),
                    amax=torch.zeros((1,), **f32), q4=torch.zeros((M, K // 2), **u8),
                    sb4=torch.zeros((M, K // 16), **u8), g4=torch.zeros((1,), **f32),
                    q2=torch.zeros((M, K // 2), **u8), sb2=torch.zeros((M // 16, K // 16), **u8),
                    g2=torch.zeros((1,), **f32))

    def step(o, x, off, seed):
        fq.mxfp4_quantize_rows(x, o["q"], o["s"])
        fq.fp4_to_fp8_rows(o["q"], o["s"], 0, o["y"], o["ys"])
        fq.fp4_to_fp8_cols(o["q"], o["s"], off, 0, o["yT"], o["yTs"])
        fq.nvfp4_amax(x, o["amax"])
        fq.nvfp4_quantize(x, o["amax"], True, seed, 0, o["q4"], o["sb4"], o["g4"])
        fq.nvfp4_quantize_2d(x, o["amax"], o["q2"], o["sb2"], o["g2"])

    chained = outputs()
    torch.cuda.synchronize()
    for i in range(24):
        step(chained, xs[i % 2], offs[i % 2], 77)
    torch.cuda.synchronize()
    alone = outputs()
    step(alone, xs[1], offs[1], 77)
    torch.cuda.synchronize()
    nb = int(((np.diff(offs[1].cpu().numpy()) + 127) // 128).sum())
    for k in alone:
        a, c = alone[k], chained[k]
        if k == "yTs":
            a, c = a[:nb], c[:nb]
        assert torch.equal(a.view(torch.uint8), c.view(torch.uint8)), k


@pytest.mark.parametrize("k", [0, 6])
def test_ragged_experts_65536x2048(fq, k):
    """Routed rows over 32 Zipf-sized experts: MXFP4 rows, then the
    transposed conversion on the ragged groups, and the one-call forward cast,
    every output compared."""
    bits, offs = workloads.ragged_experts(65536, 2048, 32, seed=0)
    x = dev_bf16(bits)
    q, s = fq.mxfp4_quantize_rows(x)
    yT, yTs = cols_full(fq, q, s, offs, k)
    fused = fq.bf16_to_mxfp4_fp8(x, torch.from_numpy(offs).cuda(), k)
    rq, rs = oracle.mxfp4_quantize_rows(bits)
    eq(q, rq, "mxfp4 q")
    eq(s, rs, "mxfp4 s")
    ryT, ryTs = oracle.fp4_to_fp8_cols(rq, rs, offs, k)
    nb = int(((np.diff(offs) + 127) // 128).sum())
    eq(yT, ryT, "fp8 cols yT")
    eq(yTs[:nb], ryTs[:nb], "fp8 cols scales")
    ry, rys = oracle.fp4_to_fp8_rows(rq, rs, k)
    for got, ref, what in zip(fused[:5], (rq, rs, ry, rys, ryT), ("q", "s", "y", "ys", "yT")):
        eq(got, ref, "fused " + what)
    eq(fused[5][:nb], ryTs[:nb], "fused yT scales")
    single = fq.bf16_to_mxfp4_fp8_single_pass(x, torch.from_numpy(offs).cuda(), k)
    for got, want in zip(single[:5], fused[:5]):
        assert torch.equal(got, want), "single-pass forward cast"
    assert torch.equal(single[5][:nb], fused[5][:nb]), "single-pass forward cast yT scales"


def test_nvfp4_activations_16384x14336(fq):
    """Student-t(4) activations: amax, SR and RNE quantization, all compared."""
    bits = workloads.nvfp4_act(16384, 14336, seed=0)
    x = dev_bf16(bits)
    amax = fq.nvfp4_amax(x)
    ra = oracle.nvfp4_amax(bits)
    assert amax.item() == float(ra)
    for sr in (True, False):
        q, sb, g = fq.nvfp4_quantize(x, amax, use_sr=sr, seed=20250, offset=0)
        rq, rsb, rg = oracle.nvfp4_quantize(bits, ra, use_sr=sr, seed=20250, offset=0)
        eq(q, rq, f"nvfp4 q sr={sr}")
        eq(sb, rsb, f"nvfp4 scales sr={sr}")
        assert g.item() == float(rg)


def test_nvfp4_rht_wgrad_inputs_16384x14336(fq):
    """The transformed WGRAD operands at the activation size: RNE (the
    activation operand) and SR (the gradient operand), every output compared."""
    bits = workloads.nvfp4_act(16384, 14336, seed=1)
    x = dev_bf16(bits)
    mask = 0x9E37
    amax = fq.nvfp4_amax_rht(x, mask)
    ra = oracle.nvfp4_amax_rht(bits, mask)
    assert amax.item() == float(ra)
    for sr in (False, True):
        q, sb, g = fq.nvfp4_quantize_rht(x, amax, mask, use_sr=sr, seed=777, offset=0)
        rq, rsb, rg = oracle.nvfp4_quantize_rht(bits, ra, mask, use_sr=sr, seed=777, offset=0)
        eq(q, rq, f"rht q sr={sr}")
        eq(sb, rsb, f"rht scales sr={sr}")
        assert g.item() == float(rg)


def test_fp8_backward_and_dequant_full_size(fq):
    """The FP8 backward-flow quantizers on the bench tensor (1x128) and the
    NVFP4 weight shape (128x128), and the MXFP4 -> BF16 dequantizer on the
    bench tensor's codes, every output compared."""
    bits = workloads.moe_dispatch(16384, 7168, seed=0)
    x = dev_bf16(bits)
    y, sc = fq.fp8_quantize_1x128(x)
    ry, rs = oracle.fp8_quantize_blocks(bits, 1)
    eq(y, ry, "1x128 codes")
    eq(sc, rs, "1x128 scales")
    q, s = fq.mxfp4_quantize_rows(x)
    rq, rsx = oracle.mxfp4_quantize_rows(bits)
    out = fq.mxfp4_dequantize_rows(q, s)
    eq(out.view(torch.uint16), oracle.mxfp4_dequantize_rows(rq, rsx), "dequant")
    wbits = workloads.nvfp4_weight(14336, 4096, seed=2)
    y2, s2 = fq.fp8_quantize_128x128(dev_bf16(wbits))
    ry2, rs2 = oracle.fp8_quantize_blocks(wbits, 128)
    eq(y2, ry2, "128x128 codes")
    eq(s2, rs2, "128x128 scales")


def test_nvfp4_delayed_activations_16384x14336(fq):
    """Three delayed-scaling steps at the activation size (RNE, SR, RNE):
    outputs and history compared at every step."""
    W = 64
    hist_d = fq.amax_history(W)
    hist = np.zeros(W + 1, dtype=np.uint64)
    for t in range(3):
        bits = workloads.nvfp4_act(16384, 14336, seed=10 + t)
        q, sb, g = fq.nvfp4_quantize_delayed(dev_bf16(bits), hist_d, t, use_sr=(t == 1), seed=3)
        rq, rsb, rg, hist = oracle.nvfp4_quantize_delayed(bits, hist, W, t, use_sr=(t == 1),
                                                          seed=3)
        eq(q, rq, f"delayed q t={t}")
        eq(sb, rsb, f"delayed sb t={t}")
        assert g.item() == float(rg)
        assert np.array_equal(hist_d.cpu().numpy().view(np.uint64), hist)


def test_nvfp4_weights_2d_14336x4096(fq):
    bits = workloads.nvfp4_weight(14336, 4096, seed=0)
    w = dev_bf16(bits)
    amax = fq.nvfp4_amax(w)
    ra = oracle.nvfp4_amax(bits)
    assert amax.item() == float(ra)
    q, sb, g = fq.nvfp4_quantize_2d(w, amax)
    rq, rsb, rqT, rsbT, rg = oracle.nvfp4_quantize_2d_t(bits, ra)
    eq(q, rq, "2d q")
    eq(sb, rsb, "2d scales")
    assert g.item() == float(rg)
    # with the transposed DGRAD operand, in one read
    q2, sb2, qT, sbT, g2 = fq.nvfp4_quantize_2d_t(w, amax)
    eq(q2, rq, "2d_t q")
    eq(sb2, rsb, "2d_t scales")
    eq(qT, rqT, "2d_t qT")
    eq(sbT, rsbT, "2d_t transposed scales")
    assert g2.item() == float(rg)


SWEEP_ROWS = [1024 << i for i in range(9)]  # 1K .. 262144 rows


def test_bandwidth_sweep_chain(fq):
    """BF16 -> MXFP4 -> FP8 rows and FP8 cols (one group) at every sweep size.
    Sizes up to 16384 rows: every output; larger: 48 seeded rows (and the
    last) and 6 seeded 128-token windows (and the last, ragged for no size
    here but still checked)."""
    K = 7168
    big = workloads.sweep(SWEEP_ROWS[-1], K, seed=0)
    x_all = dev_bf16(big)
    rng = np.random.default_rng(7)
    for M in SWEEP_ROWS:
        x = x_all[:M]
        q, s = fq.mxfp4_quantize_rows(x)
        y, ys = fq.fp4_to_fp8_rows(q, s, 0)
        offs = np.array([0, M], dtype=np.int64)
        yT, yTs = cols_full(fq, q, s, offs, 0)
        bits = big[:M]
        if M <= 16384:
            rq, rs = oracle.mxfp4_quantize_rows(bits)
            eq(q, rq, f"M={M} q")
            eq(s, rs, f"M={M} s")
            ry, rys = oracle.fp4_to_fp8_rows(rq, rs, 0)
            eq(y, ry, f"M={M} y")
            eq(ys, rys, f"M={M} ys")
            ryT, ryTs = oracle.fp4_to_fp8_cols(rq, rs, offs, 0)
            nb = (M + 127) // 128
            eq(yT, ryT, f"M={M} yT")
            eq(yTs[:nb], ryTs[:nb], f"M={M} yTs")
            continue
        rows = np.unique(np.concatenate([rng.choice(M, 48, replace=False), [M - 1]]))
        rq, rs = oracle.mxfp4_quantize_rows(bits[rows])
        idx = torch.from_numpy(rows).cuda()
        eq(q.index_select(0, idx), rq, f"M={M} sampled q")
        eq(s.index_select(0, idx), rs, f"M={M} sampled s")
        ry, rys = oracle.fp4_to_fp8_rows(rq, rs, 0)
        eq(y.index_select(0, idx), ry, f"M={M} sampled y")
        eq(ys.index_select(0, idx), rys, f"M={M} sampled ys")
        nwin = (M + 127) // 128
        wins = np.unique(np.concatenate([rng.choice(nwin, 6, replace=False), [nwin - 1]]))
        for wi in wins:
            t0, t1 = 128 * int(wi), min(M, 128 * int(wi) + 128)
            wq, ws = oracle.mxfp4_quantize_rows(bits[t0:t1])
            ryT, ryTs = oracle.fp4_to_fp8_cols(wq, ws, np.array([0, t1 - t0], dtype=np.int64), 0)
            eq(yT[:, t0:t1].contiguous(), ryT, f"M={M} window {wi} yT")
            eq(yTs[wi:wi + 1], ryTs[:1], f"M={M} window {wi} yTs")
        del q, s, y, ys, yT, yTs
        torch.cuda.empty_cache()


def test_more_than_2_31_elements(fq):
    """131200 x 16384 BF16 = 2,149,580,800 elements, past 2^31: every call on
    the whole tensor, and its outputs for rows at both ends and across element
    2^31 (row 131072) checked against the oracle, with the tensor's amax and
    the stochastic-rounding stream offsets of the sampled rows."""
    M, K = 131200, 16384
    assert M * K > 2**31 and (2**31) % K == 0
    gen = torch.Generator(device="cuda")
    gen.manual_seed(2**31 + 1)
    x = torch.randn((M, K), generator=gen, device="cuda", dtype=torch.float32).to(torch.bfloat16)
    strips = [0, 131056 // 16, 131072 // 16, M // 16 - 1]     # 16-row strips; 2^31 at row 131072
    rows = np.concatenate([np.arange(16 * s, 16 * s + 16) for s in strips])
    idx = torch.from_numpy(rows).cuda()
    bits = x.index_select(0, idx).view(torch.int16).cpu().numpy().view(np.uint16)

    def rows_of(t):
        return t.index_select(0, idx)

    # MXFP4 rows -> FP8 rows, and the one-call forward cast
    q, s = fq.mxfp4_quantize_rows(x)
    rq, rs = oracle.mxfp4_quantize_rows(bits)
    eq(rows_of(q), rq, "mxfp4 q")
    eq(rows_of(s), rs, "mxfp4 s")
    y, ys = fq.fp4_to_fp8_rows(q, s, 3)
    ry, rys = oracle.fp4_to_fp8_rows(rq, rs, 3)
    eq(rows_of(y), ry, "fp8 rows y")
    eq(rows_of(ys), rys, "fp8 rows ys")
    # transposed, one group: the 128-token windows ending at and after 2^31
    offs = np.array([0, M], dtype=np.int64)
    yT, yTs = cols_full(fq, q, s, offs, 3)
    for wi in (131072 // 128 - 1, M // 128 - 1):
        t0 = 128 * wi
        wbits = x[t0:t0 + 128].view(torch.int16).cpu().numpy().view(np.uint16)
        wq, ws = oracle.mxfp4_quantize_rows(wbits)
        ryT, ryTs = oracle.fp4_to_fp8_cols(wq, ws, np.array([0, 128], dtype=np.int64), 3)
        eq(yT[:, t0:t0 + 128].contiguous(), ryT, f"window {wi} yT")
        eq(yTs[wi:wi + 1], ryTs[:1], f"window {wi} yTs")
    fused = fq.bf16_to_mxfp4_fp8(x, torch.from_numpy(offs).cuda(), 3)
    for got, want, name in zip(fused, (q, s, y, ys, yT), ("q", "s", "y", "ys", "yT")):
        assert torch.equal(got, want), f"one-call forward cast {name}"
    nb = (M + 127) // 128
    assert torch.equal(fused[5][:nb], yTs[:nb]), "one-call forward cast yT scales"
    del fused
    single = fq.bf16_to_mxfp4_fp8_single_pass(x, torch.from_numpy(offs).cuda(), 3)
    for got, want, name in zip(single, (q, s, y, ys, yT), ("q", "s", "y", "ys", "yT")):
        assert torch.equal(got, want), f"single-pass forward cast {name}"
    assert torch.equal(single[5][:nb], yTs[:nb]), "single-pass forward cast yT scales"
    del q, s, y, ys, yT, yTs, single
    torch.cuda.empty_cache()

    # NVFP4: the amax, 1x16 with RNE and SR, 2D with the transposed operand
    amax = fq.nvfp4_amax(x)
    assert amax.item() == x.abs().max().float().item()
    A = np.float32(amax.item())
    for sr in (False, True):
        q4, sb4, g4 = fq.nvfp4_quantize(x, amax, use_sr=sr, seed=77)
        for sidx, st in enumerate(strips):
            r0 = 16 * st
            bq, bsb, bg = oracle.nvfp4_quantize(bits[16 * sidx:16 * sidx + 16], A, use_sr=sr,
                                                seed=77, offset=r0 * K)
            eq(q4[r0:r0 + 16], bq, f"nvfp4 q sr={sr} rows {r0}")
            eq(sb4[r0:r0 + 16], bsb, f"nvfp4 sb sr={sr} rows {r0}")
        assert g4.item() == float(bg)
        del q4, sb4
    q2, sb2, qT, sbT, g2 = fq.nvfp4_quantize_2d_t(x, amax)
    for sidx, st in enumerate(strips):
        r0 = 16 * st
        bq, bsb, bqT, bsbT, _ = oracle.nvfp4_quantize_2d_t(bits[16 * sidx:16 * sidx + 16], A)
        eq(q2[r0:r0 + 16], bq, f"2d q strip {st}")
        eq(sb2[st:st + 1], bsb, f"2d sb strip {st}")
        eq(qT[:, 8 * st:8 * st + 8].contiguous(), bqT, f"2d qT strip {st}")
        eq(sbT[:, st:st + 1].contiguous(), bsbT, f"2d sbT strip {st}")
    del q2, sb2, qT, sbT
    # the transform (the GPU amax of the transform is the common A)
    ar = fq.nvfp4_amax_rht(x, 0x5A5A)
    Ar = np.float32(ar.item())
    qh, sbh, gh = fq.nvfp4_quantize_rht(x, ar, 0x5A5A, use_sr=True, seed=5)
    for sidx, st in enumerate(strips):
        r0 = 16 * st
        bq, bsb, _ = oracle.nvfp4_quantize_rht(bits[16 * sidx:16 * sidx + 16], Ar, 0x5A5A,
                                               use_sr=True, seed=5, offset=r0 * K)
        eq(qh[r0:r0 + 16], bq, f"rht q rows {r0}")
        eq(sbh[r0:r0 + 16], bsb, f"rht sb rows {r0}")
    del qh, sbh
    # delayed scaling, first step of an empty history (estimate 0, g = 1)
    hist = fq.amax_history(1)
    qd, sbd, gd = fq.nvfp4_quantize_delayed(x, hist, 0, use_sr=True, seed=9)
    assert gd.item() == 1.0
    bq, bsb, _ = oracle.nvfp4_quantize(bits[-16:], np.float32(0.0), use_sr=True, seed=9,
                                       offset=(M - 16) * K)
    eq(qd[M - 16:], bq, "delayed q last rows")
    eq(sbd[M - 16:], bsb, "delayed sb last rows")
    assert int(hist.cpu().numpy().view(np.uint64)[0]) & 0xFFFFFFFF == int(
        np.float32(amax.item()).view(np.uint32))
    del qd, sbd
    torch.cuda.empty_cache()

    # FP8 1x128 rows, 128x128 tiles of the last 128 rows, MXFP4 -> BF16
    yf, sf = fq.fp8_quantize_1x128(x)
    by, bsf = oracle.fp8_quantize_blocks(bits, 1)
    eq(rows_of(yf), by, "fp8 1x128 y")
    eq(rows_of(sf), bsf, "fp8 1x128 s")
    del yf, sf
    yt, st2 = fq.fp8_quantize_128x128(x)
    tb = x[M - 128:].view(torch.int16).cpu().numpy().view(np.uint16)
    by2, bs2 = oracle.fp8_quantize_blocks(tb, 128)
    eq(yt[M - 128:], by2, "fp8 128x128 y last tiles")
    eq(st2[-1:], bs2, "fp8 128x128 s last tiles")
    del yt, st2
    q, s = fq.mxfp4_quantize_rows(x)
    d = fq.mxfp4_dequantize_rows(q, s)
    eq(rows_of(d).view(torch.int16), oracle.mxfp4_dequantize_rows(rq, rs).view(np.int16),
       "dequant rows")
