"""Pins of the oracle's expert similarity ([SERE] 4.2: Frobenius similarity
of the experts' outputs on calibration tokens) by constructions whose value
is fixed by the definition."""
import numpy as np

import oracle


def _experts(rng, N, H, I):
    wg = (rng.standard_normal((N, I, H)) / np.sqrt(H)).astype(np.float32)
    wu = (rng.standard_normal((N, I, H)) / np.sqrt(H)).astype(np.float32)
    wd = (rng.standard_normal((N, H, I)) / np.sqrt(I)).astype(np.float32)
    return wg, wu, wd


def test_constructed_pairs():
    rng = np.random.default_rng(0)
    N, H, I, n = 6, 32, 24, 5
    wg, wu, wd = _experts(rng, N, H, I)
    wg[1], wu[1], wd[1] = wg[0], wu[0], wd[0]          # duplicate of expert 0
    wg[2], wu[2], wd[2] = wg[0], wu[0], -wd[0]         # negated output
    wg[3], wu[3], wd[3] = wg[0], wu[0], 2.5 * wd[0]    # scaled output
    x = rng.standard_normal((n, H)).astype(np.float32)
    s = oracle.similarity(x, wg, wu, wd)
    assert abs(s[0, 1] - 1.0) < 1e-12
    assert abs(s[0, 2] + 1.0) < 1e-12
    assert abs(s[0, 3] - 1.0) < 1e-12
    assert abs(s[1, 3] - 1.0) < 1e-12 and abs(s[2, 3] + 1.0) < 1e-12
    assert np.array_equal(s, s.T) and np.all(np.diag(s) == 1.0)
    assert np.all(np.abs(s) <= 1.0 + 1e-12)


def test_disjoint_output_coordinates_are_orthogonal():
    """Experts whose down projections write disjoint coordinates of H have
    orthogonal outputs: similarity exactly 0; a zero expert gets 0 too."""
    rng = np.random.default_rng(1)
    N, H, I, n = 4, 24, 16, 3
    wg, wu, wd = _experts(rng, N, H, I)
    wd[0, 12:] = 0.0
    wd[1, :12] = 0.0
    wd[3] = 0.0
    x = rng.standard_normal((n, H)).astype(np.float32)
    s = oracle.similarity(x, wg, wu, wd)
    assert s[0, 1] == 0.0 and s[1, 0] == 0.0
    assert np.all(s[3, :3] == 0.0) and s[3, 3] == 1.0


def test_random_experts_are_bounded_and_not_degenerate():
    rng = np.random.default_rng(2)
    wg, wu, wd = _experts(rng, 5, 40, 20)
    x = rng.standard_normal((7, 40)).astype(np.float32)
    s = oracle.similarity(x, wg, wu, wd)
    off = s[~np.eye(5, dtype=bool)]
    assert np.all(np.abs(off) < 0.99)
    assert np.array_equal(s, s.T)
