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


def test_swiglu_orientation_closed_form():
    """With one intermediate row, an expert's output on token t is
    s_t * w_d with s_t = silu(g_t) * u_t.  Expert 0 gates on x[0] and takes
    u from x[1]; expert 1 uses x[0] for both; both share w_d.  On the tokens
    (c, -c) and (-c, c), with s = sigmoid(c): expert 0 gives
    s_t = -c^2 (s, 1 - s) and expert 1 gives c^2 (s, 1 - s), so the similarity
    is exactly -1 for every c.  Gate and up swapped would give
    -2 s (1 - s) / (s^2 + (1 - s)^2); dropping u would give +1."""
    for c in (0.7, 1.9, 3.2):
        x = np.array([[c, -c], [-c, c]], np.float32)
        wg = np.array([[[1.0, 0.0]], [[1.0, 0.0]]], np.float32)   # [N][I][H]
        wu = np.array([[[0.0, 1.0]], [[1.0, 0.0]]], np.float32)
        wd = np.array([[[1.0], [0.5]], [[1.0], [0.5]]], np.float32)   # [N][H][I]
        s = oracle.similarity(x, wg, wu, wd)
        assert abs(s[0, 1] + 1.0) < 1e-12, (c, s[0, 1])


def test_similarity_is_frobenius_over_the_stacked_tokens():
    """The similarity is the cosine of the experts' outputs stacked over all
    calibration tokens (a Frobenius inner product), not an average of
    per-token cosines.  Tokens (c, 0) and (0, c); expert 0 has gate = up =
    (1, 0), so its second output is 0; expert 1 has gate = up = (1, 1), so
    both its outputs equal the first one of expert 0; both share w_d.  The
    stacked cosine is exactly 1 / sqrt(2) for every c; per-token cosines
    would average to 1/2 or 1."""
    for c in (0.8, 2.5):
        x = np.array([[c, 0.0], [0.0, c]], np.float32)
        wg = np.array([[[1.0, 0.0]], [[1.0, 1.0]]], np.float32)
        wu = wg.copy()
        wd = np.array([[[2.0], [-1.0]], [[2.0], [-1.0]]], np.float32)
        s = oracle.similarity(x, wg, wu, wd)
        assert abs(s[0, 1] - 1.0 / np.sqrt(2.0)) < 1e-12, (c, s[0, 1])


def test_silu_shape_through_a_sign():
    """silu(c) + silu(-c) = c * tanh(c / 2) > 0 for c > 0 (with sigmoid(-g) in
    place of sigmoid(g) the sum would be -c * tanh(c / 2)).  Expert 0 reads g
    from x[0] and u = x[2] = 1 on the tokens (c, 0, 1) and (-c, 0, 1), so its
    outputs are (silu(c), silu(-c)) along w_d; expert 1 has the constant gate
    and up x[2] = 1, so its outputs are (silu(1), silu(1)) along the same w_d,
    with silu(1) > 0.  Their similarity therefore has the sign of silu(c) +
    silu(-c): positive."""
    for c in (0.5, 2.0, 4.0):
        x = np.array([[c, 0.0, 1.0], [-c, 0.0, 1.0]], np.float32)
        wg = np.array([[[1.0, 0.0, 0.0]], [[0.0, 0.0, 1.0]]], np.float32)
        wu = np.array([[[0.0, 0.0, 1.0]], [[0.0, 0.0, 1.0]]], np.float32)
        wd = np.array([[[1.0], [1.0], [0.0]], [[1.0], [1.0], [0.0]]], np.float32)
        s = oracle.similarity(x, wg, wu, wd)
        assert 0.0 < s[0, 1] < 1.0, (c, s[0, 1])


def test_silent_expert_with_a_shared_down_projection():
    """An expert whose gate and up projections are zero outputs exactly zero,
    so its similarity with every other expert is 0, even when its down
    projection equals another expert's (I = 3, so each expert's gate/up rows are
    a block of its own)."""
    rng = np.random.default_rng(12)
    n, H, I, N = 5, 6, 3, 3
    x = rng.standard_normal((n, H)).astype(np.float32)
    wg = rng.standard_normal((N, I, H)).astype(np.float32)
    wu = rng.standard_normal((N, I, H)).astype(np.float32)
    wd = rng.standard_normal((N, H, I)).astype(np.float32)
    wg[1] = 0.0
    wu[1] = 0.0
    wd[1] = wd[0]
    s = oracle.similarity(x, wg, wu, wd)
    assert s[0, 1] == 0.0 and s[1, 0] == 0.0 and s[1, 2] == 0.0
    assert abs(s[0, 2]) < 1.0


def test_smallest_sizes():
    """One token, one feature, one intermediate unit: a single expert with a
    nonzero output has similarity 1 with itself; two such experts with outputs
    of opposite sign have -1."""
    x = np.array([[2.0]], np.float32)
    one = np.ones((1, 1, 1), np.float32)
    assert oracle.similarity(x, one, one, one).tolist() == [[1.0]]
    wd = np.array([[[1.0]], [[-3.0]]], np.float32)
    two = np.ones((2, 1, 1), np.float32)
    s = oracle.similarity(x, two, two, wd)
    assert s[0, 1] == -1.0 and s[0, 0] == 1.0 and s[1, 1] == 1.0
