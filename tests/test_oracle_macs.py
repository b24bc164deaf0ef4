"""Pins of the oracle's entropy-weighted token load ([MACS] 3.2 Eqs. (4)-(5),
3.3 Eq. (7)) against scipy, closed forms and the equations' special cases."""
import numpy as np
import pytest
from scipy.special import softmax
from scipy.stats import entropy as scipy_entropy

import oracle
from expert_routing_moe_gb300 import synthetic as syn


def test_entropy_matches_scipy():
    rng = np.random.default_rng(0)
    x = (rng.standard_normal((12, 300)) * rng.uniform(0.1, 5.0, size=(12, 1))).astype(np.float32)
    ent, _, _ = oracle.token_weights(x, np.ones(12, np.uint8))
    ref = np.array([scipy_entropy(softmax(r.astype(np.float64))) for r in x])
    assert np.allclose(ent, ref, rtol=1e-12, atol=1e-12)


def test_entropy_closed_forms():
    D = 257
    # uniform features: p uniform, H = ln D
    ent, _, _ = oracle.token_weights(np.full((1, D), 3.25, np.float32), np.ones(1, np.uint8))
    assert abs(ent[0] - np.log(D)) < 1e-12
    # one raised entry a: p0 = e^a / (e^a + D - 1), the others q = 1 / (e^a + D - 1)
    a = 4.0
    z = np.zeros((1, D), np.float32)
    z[0, 17] = a
    den = np.exp(a) + D - 1
    p0, q = np.exp(a) / den, 1.0 / den
    ent, _, _ = oracle.token_weights(z, np.ones(1, np.uint8))
    assert abs(ent[0] - (-p0 * np.log(p0) - (D - 1) * q * np.log(q))) < 1e-12
    # shift invariance
    rng = np.random.default_rng(1)
    x = rng.standard_normal((3, 64)).astype(np.float32)
    e1, _, _ = oracle.token_weights(x, np.ones(3, np.uint8))
    e2, _, _ = oracle.token_weights(x + np.float32(7.5), np.ones(3, np.uint8))
    assert np.allclose(e1, e2, atol=1e-12)


def test_two_visual_tokens_give_sigmoid_of_plus_minus_delta():
    """With two visual tokens of entropies h1 < h2 the population statistics
    are mu = (h1 + h2) / 2, sigma = (h2 - h1) / 2, so Htilde = -+1 (up to eps)
    and w = sigmoid(+-delta); the lower-entropy token weighs more."""
    D, delta, eps = 64, 1.7, 1e-6
    z = np.zeros((3, D), np.float32)
    z[1, 0] = 6.0                 # low entropy
    ent, w, rv = oracle.token_weights(z, np.array([0, 1, 1], np.uint8), delta=delta, eps=eps)
    h1, h2 = ent[1], ent[0 + 2]
    assert h1 < h2
    sig = (h2 - h1) / 2
    ht = sig / (sig + eps)
    sgm = lambda v: 1.0 / (1.0 + np.exp(-v))
    assert abs(w[1] - sgm(delta * ht)) < 1e-12
    assert abs(w[2] - sgm(-delta * ht)) < 1e-12
    assert abs(w[1] + w[2] - 1.0) < 1e-12
    assert w[0] == 1.0                            # text token
    assert abs(rv - (w[1] + w[2]) / (w.sum())) < 1e-15


def test_weight_special_cases():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((40, 128)).astype(np.float32) * rng.uniform(0.2, 3, size=(40, 1)).astype(np.float32)
    vis = (rng.random(40) < 0.6).astype(np.uint8)
    _, w0, _ = oracle.token_weights(x, vis, delta=0.0)
    assert np.all(w0[vis == 1] == 0.5) and np.all(w0[vis == 0] == 1.0)
    ent, w, rv = oracle.token_weights(x, vis, delta=2.0)
    assert np.all((w > 0) & (w <= 1))
    # monotone: among visual tokens, more entropy -> less weight
    order = np.argsort(ent[vis == 1])
    assert np.all(np.diff(w[vis == 1][order]) <= 0)
    assert 0.0 < rv < 1.0
    _, w_all_txt, rv_t = oracle.token_weights(x, np.zeros(40, np.uint8))
    assert rv_t == 0.0 and np.all(w_all_txt == 1.0)
    _, _, rv_v = oracle.token_weights(x, np.ones(40, np.uint8))
    assert rv_v == 1.0


def test_bf16_input_uses_exact_values():
    L = syn.prefill(T=64, with_weights=False)
    e_bf, _, _ = oracle.token_weights(L.x_bf16, L.is_visual.astype(np.uint8), x_dtype=oracle.DT_BF16)
    e_f, _, _ = oracle.token_weights(L.x, L.is_visual.astype(np.uint8))
    assert np.allclose(e_bf, e_f, atol=1e-12)


def test_three_visual_tokens_two_alike_closed_form():
    """Visual entropies (h, h, g): the population statistics give mu = (2h + g)/3
    and sigma = |h - g| sqrt(2)/3, so Htilde = s/sqrt(2) for the pair and
    -s sqrt(2) for the odd one (s = sign(h - g)), whatever h and g are.  A sample
    (n - 1) variance would give 1/sqrt(3) instead, and statistics taken over the
    text tokens too would move both values."""
    D, delta = 96, 1.3
    z = np.zeros((5, D), np.float32)
    z[1, 3] = 5.0                   # the odd visual token: lower entropy (g < h)
    z[3, :7] = 9.0                  # a text token far from the others
    vis = np.array([1, 1, 0, 0, 1], np.uint8)   # token 2 is a plain text token
    ent, w, _ = oracle.token_weights(z, vis, delta=delta, eps=0.0)
    h, g = ent[0], ent[1]
    assert g < h and ent[4] == h
    sgm = lambda v: 1.0 / (1.0 + np.exp(-v))
    assert abs(w[0] - sgm(-delta / np.sqrt(2))) < 1e-12
    assert abs(w[4] - sgm(-delta / np.sqrt(2))) < 1e-12
    assert abs(w[1] - sgm(delta * np.sqrt(2))) < 1e-12
    assert w[2] == 1.0 and w[3] == 1.0


def test_visual_weights_ignore_the_text_tokens():
    """Eq. (5) standardises over the visual tokens only: changing the text
    tokens' features, or adding more text tokens, leaves every visual weight as
    it was; R_v alone moves, through the text tokens' weight of 1 each."""
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((30, 80)) * rng.uniform(0.2, 4.0, size=(30, 1))).astype(np.float32)
    vis = (rng.random(30) < 0.5).astype(np.uint8)
    vis[:2] = 1
    _, w1, rv1 = oracle.token_weights(x, vis, delta=1.5)
    x2 = x.copy()
    x2[vis == 0] = (rng.standard_normal(((vis == 0).sum(), 80)) * 6.0).astype(np.float32)
    _, w2, rv2 = oracle.token_weights(x2, vis, delta=1.5)
    assert np.array_equal(w1, w2) and rv1 == rv2
    x3 = np.concatenate([x, rng.standard_normal((7, 80)).astype(np.float32)])
    vis3 = np.concatenate([vis, np.zeros(7, np.uint8)])
    _, w3, rv3 = oracle.token_weights(x3, vis3, delta=1.5)
    assert np.array_equal(w3[:30], w1) and np.all(w3[30:] == 1.0)
    wv = w1[vis == 1].sum()
    assert abs(rv3 - wv / (wv + (vis == 0).sum() + 7)) < 1e-14
