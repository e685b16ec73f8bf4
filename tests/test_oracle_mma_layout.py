"""Pins of the oracle's block-scaled-MMA scale layout (MXFP4 scales [M, K/32]
re-laid as 512-byte atoms of 128 rows x 4 scale columns).

The layout is a permutation of the zero-padded scale matrix, so it is pinned
by the same permutation built from numpy's reshape and transpose of the
blocked matrix (rows split as (tile, 4 groups of 32), columns as (tile, 4)),
by the atoms holding exactly their tile's bytes, and by the multiset of bytes
(every scale once, plus the padding zeros)."""
import numpy as np
import pytest

import oracle

SHAPES = [(1, 128), (31, 128), (128, 128), (129, 256), (300, 384), (1000, 7168), (4096, 512)]


def blocked(s, M, K):
    nrb, ncb = (M + 127) // 128, K // 128
    pad = np.zeros((nrb * 128, K // 32), dtype=np.uint8)
    pad[:M] = s
    # rows: (tile rb, group i, row j in group); columns: (tile cb, column l)
    t = pad.reshape(nrb, 4, 32, ncb, 4)
    # stored order: tile rb, tile cb, then j, i, l
    return t.transpose(0, 3, 2, 1, 4).reshape(-1)


@pytest.mark.parametrize("M,K", SHAPES)
def test_layout_is_the_blocked_transpose(M, K):
    rng = np.random.default_rng(M * 7 + K)
    s = rng.integers(0, 256, size=(M, K // 32), dtype=np.uint8)
    out = oracle.mxfp4_scales_mma_layout(s, M, K)
    assert out.size == ((M + 127) // 128) * (K // 128) * 512
    assert np.array_equal(out, blocked(s, M, K))


@pytest.mark.parametrize("M,K", SHAPES)
def test_every_scale_once_and_zero_padding(M, K):
    rng = np.random.default_rng(M + K)
    s = rng.integers(1, 256, size=(M, K // 32), dtype=np.uint8)   # no zero scales
    out = oracle.mxfp4_scales_mma_layout(s, M, K)
    npad = out.size - s.size
    assert np.count_nonzero(out == 0) == npad
    assert np.array_equal(np.sort(out[out != 0]), np.sort(s.reshape(-1)))


def test_each_atom_holds_its_tile():
    """The 512 bytes of atom (rb, cb) are exactly the scales of rows
    128 rb .. 128 rb + 127, columns 4 cb .. 4 cb + 3: tagging every scale
    with its tile number shows one tag per atom, atoms in row-tile-major
    order."""
    M, K = 1000, 1024
    nrb, ncb = (M + 127) // 128, K // 128
    tag = np.zeros((M, K // 32), dtype=np.uint8)
    for r in range(M):
        for c in range(K // 32):
            tag[r, c] = 1 + (r // 128) * ncb + c // 4
    out = oracle.mxfp4_scales_mma_layout(tag, M, K).reshape(nrb * ncb, 512)
    for a in range(nrb * ncb):
        vals = set(out[a][out[a] != 0].tolist())
        assert vals == {1 + a}, (a, vals)


def test_row_and_column_positions_inside_an_atom():
    """A single nonzero scale at (r, c) lands at byte 16 (r mod 32) +
    4 ((r mod 128) / 32) + (c mod 4) of its atom: rows 32 apart are
    neighbouring words, consecutive rows are 16 bytes apart."""
    M, K = 256, 256
    for r, c in [(0, 0), (1, 0), (31, 3), (32, 0), (33, 1), (127, 3), (128, 4), (200, 6)]:
        s = np.zeros((M, K // 32), dtype=np.uint8)
        s[r, c] = 9
        out = oracle.mxfp4_scales_mma_layout(s, M, K)
        (pos,) = np.nonzero(out)
        atom = (r // 128) * (K // 128) + c // 4
        assert pos.tolist() == [atom * 512 + 16 * (r % 32) + 4 * ((r % 128) // 32) + c % 4]


def test_rejects_k_not_multiple_of_128():
    with pytest.raises(ValueError):
        oracle.mxfp4_scales_mma_layout(np.zeros((4, 3), np.uint8), 4, 96)
