"""Device stochastic rounding pinned to its closed form, not to the oracle.

The byte-exact parity tests compare the SR kernels with the oracle under the
same Philox stream; they cannot tell whether that stream, as both sides map
it onto elements, gives each element a uniform random number.  Here the
device output is checked against the definition of unbiased stochastic
rounding alone (see sr_closed_form): over 256 seeds x 65536 blocks, the
up-rate of every (value, position in the block) is floor(2^16 frac) / 2^16
within 4 sigma, and the mean decoded value of every value equals the value
itself within 4 sigma -- for nvfp4_quantize and for nvfp4_quantize_rht, at
fractions 2^-16, 1/4, 1/2, 3/4, 7/8, 1 - 3 * 2^-16 and 1 - 2^-16."""
from fractions import Fraction

import numpy as np
import pytest
import torch

import sr_closed_form as S

pytestmark = pytest.mark.gpu

SEEDS = 256
NBLOCKS = 65536
MASK = 0xA5C3


@pytest.fixture(scope="module")
def fq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import fp8_quantization_gb300 as m
    m.abi()
    return m


@pytest.mark.parametrize("setup", ["pow2", "near1"])
@pytest.mark.parametrize("kind", ["plain", "rht"])
def test_device_sr_matches_closed_form(fq, kind, setup):
    d = S.build(setup, NBLOCKS, MASK if kind == "rht" else None)
    bits, types = d["bits"], d["types"]
    M, K = bits.shape
    nt = len(types)
    x = torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)
    amax = torch.tensor([float(d["A"])], dtype=torch.float32, device="cuda")
    tix = np.where(d["etype"] < 0, nt - 1, d["etype"])          # block maxima: last type
    lo = torch.from_numpy(np.array([t[1] for t in types], dtype=np.uint8)[tix]).cuda()
    hi = torch.from_numpy(np.array([t[2] for t in types], dtype=np.uint8)[tix]).cuda()
    neg = torch.from_numpy(bits >= 0x8000).cuda()
    q = torch.empty((M, K // 2), dtype=torch.uint8, device="cuda")
    sb = torch.empty((M, K // 16), dtype=torch.uint8, device="cuda")
    g = torch.empty((1,), dtype=torch.float32, device="cuda")
    ups = torch.zeros((M, K), dtype=torch.int32, device="cuda")
    stray = torch.zeros((), dtype=torch.int64, device="cuda")
    for seed in range(SEEDS):
        if kind == "rht":
            fq.nvfp4_quantize_rht(x, amax, MASK, use_sr=True, seed=seed, q=q, sb=sb, g=g)
        else:
            fq.nvfp4_quantize(x, amax, use_sr=True, seed=seed, q=q, sb=sb, g=g)
        c = torch.stack([q & 15, q >> 4], dim=-1).view(M, K)
        mag = c & 7
        stray += (~((mag == lo) | (mag == hi))).sum()
        ups += ((mag == hi) & (hi != lo)).int()
        if seed == 0:
            assert torch.all(sb == d["b"]), "block scale byte"
            assert g.item() == float(d["g"]), "per-tensor scale"
            if kind == "plain":        # the sign of every code is the input's
                assert torch.equal((c >> 3).bool(), neg)
    assert stray.item() == 0, "a code that is neither neighbour of its value"

    # up-rate per (value, position)
    idx = (tix * 16 + d["epos"]).ravel()
    ups_np = ups.cpu().numpy().ravel().astype(np.int64)
    up_tp = np.bincount(idx, weights=ups_np, minlength=nt * 16).reshape(nt, 16)
    trials_tp = np.bincount(idx, minlength=nt * 16).reshape(nt, 16) * SEEDS
    S.check_counts(up_tp, trials_tp, [t[3] for t in types], f"{kind}/{setup}")

    # mean decoded value per value type: every sample is lo or hi, so the
    # mean follows from the up count; it must equal the value y itself
    for ti, (y, lo_c, hi_c, p, expect) in enumerate(types):
        assert expect == Fraction(float(y))          # chosen so that E = y exactly
        n = int(trials_tp[ti].sum())
        k = int(up_tp[ti].sum())
        glo, ghi = S.GRID[lo_c], S.GRID[hi_c]
        mean = float(glo) + k / n * float(ghi - glo)
        sd = float(ghi - glo) * np.sqrt(float(p) * (1 - float(p)) / n)
        assert abs(mean - float(y)) <= 4 * sd + 1e-12 * float(y), (kind, setup, ti, mean, y, sd)
