"""The seeded input generators (CPU): the FAVOR+ projection draw."""
import numpy as np

import workloads


def test_favor_projection_orthogonal_blocks():
    """Rows within each block of d are mutually orthogonal; the last block is cut at m."""
    d, m = 16, 40
    W = workloads.favor_projection(7, m, d).astype(np.float64)
    assert W.shape == (m, d) and W.dtype == np.float64
    for b0 in range(0, m, d):
        blk = W[b0:b0 + d]
        g = blk @ blk.T
        off = g - np.diag(np.diag(g))
        assert np.max(np.abs(off)) <= 1e-5 * np.max(np.diag(g))


def test_favor_projection_gaussian_row_lengths():
    """Each row keeps the length distribution of an N(0, I) vector: E|w|^2 = d, with the
    spread of a chi-square with d degrees of freedom (variance 2d)."""
    d, m = 32, 32 * 256
    W = workloads.favor_projection(8, m, d).astype(np.float64)
    sq = (W ** 2).sum(1)
    assert abs(sq.mean() - d) < 5 * np.sqrt(2 * d / m)
    assert abs(sq.var() - 2 * d) < 0.15 * 2 * d


def test_favor_projection_seeded_and_bf16():
    a = workloads.favor_projection(9, 64, 64, "bf16")
    b = workloads.favor_projection(9, 64, 64, "bf16")
    assert a.dtype == np.uint16 and np.array_equal(a, b)
    f = workloads.favor_projection(9, 64, 64)
    assert np.max(np.abs(workloads.bf16_bits_to_f32(a) - f)) <= 2.0 ** -8 * np.max(np.abs(f))
    g = workloads.favor_projection(9, 64, 64, orthogonal=False)
    assert not np.allclose(f, g)
