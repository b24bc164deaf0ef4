"""Edge cases of the oracle: the boundary of the specified exponential's flush
to zero, rows whose features sit far from zero (where the entropy's max
subtraction matters), empty batches, and the limits of the argument checks
(an expert id equal to N, sizes of zero, the extreme visual ratios)."""
import numpy as np
import pytest
from scipy.special import softmax
from scipy.stats import entropy as scipy_entropy

import oracle


def test_exp_spec_flush_boundary():
    """The reduction's n = rint(d log2 e) keeps results normal down to n = -125,
    i.e. d = -125.5 ln 2: above that the result is within 2 ulp of exp(d), below
    it the result is flushed to 0."""
    dstar = -125.5 * np.log(2.0)
    rng = np.random.default_rng(9)
    above = (dstar + 0.005 + rng.random(20000) * (-86.0 - dstar - 0.005)).astype(np.float32)
    got = oracle.exp_spec(above).astype(np.float64)
    ref = np.exp(above.astype(np.float64))
    assert np.all(got > 0)
    assert np.max(np.abs(got - ref) / np.spacing(ref.astype(np.float32)).astype(np.float64)) <= 2.0
    below = (dstar - 0.005 - rng.random(20000) * 10.0).astype(np.float32)
    assert np.all(oracle.exp_spec(below) == 0.0)


def test_entropy_of_rows_far_from_zero():
    """Softmax and its entropy ignore a row's offset; the oracle subtracts each
    row's own maximum, so rows shifted by +-1000 (where exp itself overflows or
    underflows in double) match scipy on the unshifted rows."""
    rng = np.random.default_rng(3)
    base = rng.standard_normal((6, 200)).astype(np.float32)
    x = base.copy()
    x[1] += np.float32(1000.0)
    x[3] -= np.float32(1000.0)
    x[4] += np.float32(750.0)
    ent, _, _ = oracle.token_weights(x, np.ones(6, np.uint8))
    ref = np.array([scipy_entropy(softmax(r.astype(np.float64))) for r in x])
    assert np.all(np.isfinite(ent))
    assert np.allclose(ent, ref, rtol=1e-9, atol=1e-9)


def test_empty_batches():
    H, N, k, R = 16, 8, 2, 4
    x = np.zeros((0, H), np.float32)
    assert oracle.router(x, np.ones((N, H), np.float32)).shape == (0, N)
    ids, gates = oracle.route(np.zeros((0, N), np.float32), R)
    assert ids.shape == (0, R) and gates.shape == (0, R)
    ent, w, rv = oracle.token_weights(x, np.zeros(0, np.uint8))
    assert ent.shape == (0,) and w.shape == (0,) and rv == 0.0
    ids = np.zeros((0, R), np.int32)
    gates = np.zeros((0, R), np.float32)
    p = oracle.permute(ids, gates, N, k)
    assert np.all(p["counts"] == 0) and np.all(p["offsets"] == 0) and p["active"][0] == 0
    oi, og, st, load, C = oracle.capacity(ids, gates, N, k, R, None, 1.25)
    assert oi.shape == (0, k) and np.all(load == 0) and C == 0
    a, b, bitmap, stats = oracle.sere(ids, gates, N, k, 1, 0.5, np.eye(N, dtype=np.float32))
    assert a.shape == (0, R) and np.all(bitmap == 0) and np.all(stats == 0)
    wg = np.zeros((N, 3, H), np.float32)
    wd = np.zeros((N, H, 3), np.float32)
    y = oracle.ffn_combine(x, wg, wg, wd, ids, gates, k)
    assert y.shape == (0, H)


def test_ffn_combine_empty_token_list_and_k_limits():
    rng = np.random.default_rng(4)
    T, H, I, N, k = 3, 8, 4, 4, 2
    x = rng.standard_normal((T, H)).astype(np.float32)
    wg = rng.standard_normal((N, I, H)).astype(np.float32)
    wd = rng.standard_normal((N, H, I)).astype(np.float32)
    ids = np.array([[0, 1], [2, 3], [1, 0]], np.int32)
    gates = np.full((T, k), 0.5, np.float32)
    assert oracle.ffn_combine(x, wg, wg, wd, ids, gates, k, tokens=np.zeros(0, np.int32)).shape == (0, H)
    with pytest.raises(RuntimeError):
        oracle.ffn_combine(x, wg, wg, wd, ids, gates, 0)          # k = 0
    with pytest.raises(RuntimeError):
        oracle.ffn_combine(x, wg, wg, wd, ids, gates, 3)          # k wider than the id rows


def test_an_expert_id_equal_to_N_is_rejected():
    """Ids run over 0..N-1 (and -1 for an empty slot where the step allows it):
    an id of exactly N is out of range for every step that reads ids."""
    rng = np.random.default_rng(6)
    T, H, I, N, k = 4, 8, 4, 4, 2
    ids = np.array([[0, 1], [2, 3], [1, N], [3, 0]], np.int32)
    gates = np.full((T, k), 0.5, np.float32)
    with pytest.raises(RuntimeError):
        oracle.permute(ids, gates, N, k)
    with pytest.raises(RuntimeError):
        oracle.sere(ids, gates, N, k, 1, 0.5, np.eye(N, dtype=np.float32))
    x = rng.standard_normal((T, H)).astype(np.float32)
    wg = rng.standard_normal((N, I, H)).astype(np.float32)
    wd = rng.standard_normal((N, H, I)).astype(np.float32)
    with pytest.raises(RuntimeError):
        oracle.ffn_combine(x, wg, wg, wd, ids, gates, k)
    ok = ids.copy()
    ok[2, 1] = 0
    with pytest.raises(RuntimeError):                               # a token index equal to T
        oracle.ffn_combine(x, wg, wg, wd, ok, gates, k, tokens=np.array([0, T], np.int32))


def test_zero_sizes_are_rejected():
    with pytest.raises(RuntimeError):
        oracle.router(np.zeros((2, 0), np.float32), np.zeros((4, 0), np.float32))      # H = 0
    with pytest.raises(RuntimeError):
        oracle.router(np.zeros((2, 8), np.float32), np.zeros((0, 8), np.float32))      # N = 0
    with pytest.raises(RuntimeError):
        oracle.route(np.zeros((2, 4), np.float32), 5)                                  # R > N
    with pytest.raises(RuntimeError):
        oracle.route(np.zeros((2, 4), np.float32), 0)                                  # R = 0
    x = np.ones((2, 3), np.float32)
    wg, wd = np.ones((2, 4, 3), np.float32), np.ones((2, 3, 4), np.float32)
    for args in [(x[:, :0], wg[:, :, :0], wg[:, :, :0], wd[:, :0, :]),                  # H = 0
                 (x, wg[:, :0, :], wg[:, :0, :], wd[:, :, :0]),                          # I = 0
                 (x, wg[:0], wg[:0], wd[:0]),                                            # N = 0
                 (x[:0], wg, wg, wd)]:                                                   # no tokens
        with pytest.raises(RuntimeError):
            oracle.similarity(*args)


def test_renormalising_all_R_ranks_is_allowed():
    """renorm_k may equal R: the R ranked gates are divided by their sum."""
    rng = np.random.default_rng(8)
    ids, g = oracle.route(rng.standard_normal((5, 16)).astype(np.float32), 4, renorm_k=4)
    assert np.allclose(g.astype(np.float64).sum(axis=1), 1.0, atol=1e-6)
    with pytest.raises(RuntimeError):
        oracle.route(rng.standard_normal((5, 16)).astype(np.float32), 4, renorm_k=5)


@pytest.mark.parametrize("r_v", [0.0, 1.0])
def test_extreme_visual_ratios(r_v):
    """R_v = 0 (all text) and R_v = 1 (all visual) are valid: with m = +1 an
    expert's capacity is c (1 + (R_v - 1/2)), with m = -1 c (1 - (R_v - 1/2)),
    so half or one and a half times the static value."""
    S, k, g, N = 1000 * (1 << 24), 8, 1.25, 16
    c = S * k * g / N
    vis, txt = oracle.capacity_expert(S, k, g, N, +1, r_v), oracle.capacity_expert(S, k, g, N, -1, r_v)
    assert vis == int(np.floor(c * (0.5 + r_v))) and txt == int(np.floor(c * (1.5 - r_v)))
    rng = np.random.default_rng(10)
    ids, gates = oracle.route(rng.standard_normal((40, N)).astype(np.float32), 4)
    bias = np.array([1, -1, 0, 1] * 4, np.int8)
    oi, og, st, load, C = oracle.capacity(ids, gates, N, 2, 4, None, g, bias=bias, r_v=r_v)
    caps = [oracle.capacity_expert(40 * (1 << 24), 2, g, N, int(m), r_v) for m in bias]
    assert np.all(load <= np.array(caps))


def test_one_feature_rows_have_zero_entropy():
    """With D = 1 the softmax is the single value 1, so every entropy is 0; the
    visual tokens' entropies then have sigma = 0, Htilde = 0 and weight 1/2."""
    x = np.array([[3.0], [-7.5], [0.25]], np.float32)
    vis = np.array([1, 0, 1], np.uint8)
    ent, w, rv = oracle.token_weights(x, vis, delta=2.0)
    assert ent.tolist() == [0.0, 0.0, 0.0]
    assert w.tolist() == [0.5, 1.0, 0.5] and rv == 0.5
