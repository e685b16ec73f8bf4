"""GPU: the library's calls inside a CUDA graph.

Every entry point only enqueues work on the caller's stream (with
programmatic dependent launch between kernels), so a chain of calls can be
captured once with stream capture and replayed.  Captured here: the bench
step's six casts and the other calls; the graph is replayed on fresh inputs
copied into the captured buffers, and every output is compared byte for byte
with the same calls made directly."""
import numpy as np
import pytest
import torch

from fp8_quantization_gb300 import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import fp8_quantization_gb300 as m
    m.abi()
    return m


def _outputs(fq, x, offs, hist, step, nb):
    """All calls on x into fresh outputs (also the capture body)."""
    q, s = fq.mxfp4_quantize_rows(x)
    y, ys = fq.fp4_to_fp8_rows(q, s, 0)
    yT, yTs = fq.fp4_to_fp8_cols(q, s, offs, 3)
    amax = fq.nvfp4_amax(x)
    q4, sb4, g4 = fq.nvfp4_quantize(x, amax, use_sr=True, seed=1234, offset=0)
    q2, sb2, g2 = fq.nvfp4_quantize_2d(x, amax)
    fused = fq.bf16_to_mxfp4_fp8(x, offs, 2)
    single = fq.bf16_to_mxfp4_fp8_single_pass(x, offs, 2)
    ar = fq.nvfp4_amax_rht(x, 0x1357)
    qr, sbr, gr = fq.nvfp4_quantize_rht(x, ar, 0x1357, True, 99, 0)
    f1 = fq.fp8_quantize_1x128(x)
    f2 = fq.fp8_quantize_128x128(x)
    deq = fq.mxfp4_dequantize_rows(q, s)
    w = fq.nvfp4_quantize_2d_t(x, amax)
    dl = fq.nvfp4_quantize_delayed(x, hist, step, True, 7, 0)
    mma = fq.mxfp4_scales_mma_layout(s)
    # rows of the transposed scales past the last (nb-th) block are not written
    fused, single = list(fused), list(single)
    fused[5], single[5] = fused[5][:nb], single[5][:nb]
    return [q, s, y, ys, yT, yTs[:nb], amax, q4, sb4, g4, q2, sb2, g2, *fused, *single, ar, qr,
            sbr, gr, *f1, *f2, deq, *w, *dl, mma]


def _blocks(offs_np):
    """128-token blocks of the groups (the rows of the transposed scales in use)."""
    counts = np.diff(offs_np)
    return int(((counts + 127) // 128).sum())


def test_calls_replay_in_a_cuda_graph(fq):
    M, K, G = 2048, 1024, 8
    offs_np = workloads.zipf_group_offsets(M, G, 1.1, 5)
    offs = torch.from_numpy(offs_np).cuda()
    nb = _blocks(offs_np)
    inputs = [workloads.moe_dispatch(M, K, seed=s) for s in (1, 2)]
    x = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    x.copy_(torch.from_numpy(inputs[0].view(np.int16)).view(torch.bfloat16))
    hist_g = fq.amax_history(8, device="cuda")
    _outputs(fq, x, offs, fq.amax_history(8, device="cuda"), 0, nb)  # lazy set-up outside capture
    torch.cuda.synchronize()

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        captured = _outputs(fq, x, offs, hist_g, 0, nb)
    torch.cuda.synchronize()

    hist_d = fq.amax_history(8, device="cuda")
    first = None
    for bits in inputs:
        x.copy_(torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16))
        graph.replay()
        torch.cuda.synchronize()
        xd = torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)
        direct = _outputs(fq, xd, offs, hist_d, 0, nb)
        torch.cuda.synchronize()
        assert len(direct) == len(captured)
        for i, (a, b) in enumerate(zip(captured, direct)):
            assert a.shape == b.shape, i
            assert torch.equal(a.reshape(-1).view(torch.uint8), b.reshape(-1).view(torch.uint8)), i
        assert torch.equal(hist_g, hist_d)
        if first is None:
            first = captured[0].clone()
    assert not torch.equal(first, captured[0]), "the replay did not recompute the codes"
