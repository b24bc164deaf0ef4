"""Pins for the oracle's router, gate and ranking (CPU only)."""
import math
from decimal import Decimal, getcontext
from fractions import Fraction

import numpy as np
import pytest

import oracle
from expert_routing_moe_gb300 import synthetic as syn


def _rn32(v: Fraction) -> float:
    """Round a positive rational to the nearest fp32, ties to even, exactly."""
    e = math.floor(math.log2(v))
    while Fraction(2) ** e > v:
        e -= 1
    while Fraction(2) ** (e + 1) <= v:
        e += 1
    m = v * Fraction(2) ** (23 - e)
    n = m.numerator // m.denominator
    rem = m - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return float(Fraction(n) * Fraction(2) ** (e - 23))


def test_exp_constants_rederived_exactly():
    getcontext().prec = 80
    ln2 = Fraction(Decimal(2).ln())
    log2e = Fraction(1 / Decimal(2).ln())
    hi = Fraction(math.floor(ln2 * 2 ** 15), 2 ** 15)
    want = [_rn32(log2e), float(hi), _rn32(ln2 - hi)] + [_rn32(Fraction(1, math.factorial(i))) for i in range(8)]
    got = [float(v) for v in oracle.exp_constants()]
    assert got == want


def test_exp_spec_accuracy_and_special_values():
    rng = np.random.default_rng(5)
    # the spec flushes results below about 2^-125 to zero, so accuracy is
    # checked where the result is a normal number with margin (d >= -86)
    d = np.concatenate([-rng.random(200000).astype(np.float32) * 86.0,
                        -rng.random(50000).astype(np.float32) * 0.5,
                        np.array([0.0, -1e-8, -0.5 * np.log(2), -np.log(2)], dtype=np.float32)])
    d = d.astype(np.float32)
    got = oracle.exp_spec(d).astype(np.float64)
    ref = np.exp(d.astype(np.float64))
    ulp = np.spacing(ref.astype(np.float32)).astype(np.float64)
    assert np.max(np.abs(got - ref) / ulp) <= 2.0
    assert oracle.exp_spec(np.float32([0.0]))[0] == 1.0
    # arguments whose result would be subnormal flush to zero
    assert oracle.exp_spec(np.float32([-88.0, -100.0, -1e30]))[:].tolist() == [0.0, 0.0, 0.0]


def test_router_matches_float64_matmul():
    L = syn.tiny()
    got = oracle.router(L.x, L.w_r)
    ref = (L.x.astype(np.float64) @ L.w_r.astype(np.float64).T).astype(np.float32)
    assert np.max(np.abs(got - ref) / np.spacing(np.abs(ref))) <= 1.0
    # bf16 input path: the bits are decoded exactly
    Lq = syn.qwen_layer(8, H=256, N=16, k=4, I=64)
    got = oracle.router(Lq.x_bf16, Lq.w_r, oracle.DT_BF16)
    ref = (Lq.x.astype(np.float64) @ Lq.w_r.astype(np.float64).T).astype(np.float32)
    assert np.max(np.abs(got - ref) / np.spacing(np.abs(ref))) <= 1.0


@pytest.mark.parametrize("N,R", [(8, 2), (8, 8), (128, 8), (128, 10), (33, 5), (256, 16)])
def test_ranking_is_lexsort_by_logit_then_id(N, R):
    rng = np.random.default_rng(N * 100 + R)
    T = 64
    logits = rng.standard_normal((T, N)).astype(np.float32)
    # plant exact ties, including ties that straddle the top-R boundary
    logits[:, N // 2] = logits[:, 0]
    logits[:, N - 1] = logits[:, 1]
    logits[::3, 2] = logits[::3, 3]
    ids, _ = oracle.route(logits, R)
    for t in range(T):
        order = np.lexsort((np.arange(N), -logits[t].astype(np.float64)))
        assert ids[t].tolist() == order[:R].tolist()


def test_gates_are_the_softmax():
    rng = np.random.default_rng(11)
    for N in (8, 64, 128, 200):
        logits = (rng.standard_normal((32, N)) * 3).astype(np.float32)
        ids, gates = oracle.route(logits, N)
        l64 = logits.astype(np.float64)
        p = np.exp(l64 - l64.max(1, keepdims=True))
        p /= p.sum(1, keepdims=True)
        ref = np.take_along_axis(p, ids.astype(np.int64), 1)
        assert np.max(np.abs(gates - ref) / ref) < 2e-6
        assert np.all(np.diff(gates, axis=1) <= 0)  # ranked gates never increase
        assert np.allclose(gates.astype(np.float64).sum(1), 1.0, atol=1e-5)


def test_gate_sum_order_is_the_fixed_tree():
    # The normaliser is the 32-lane partial sums followed by the xor butterfly;
    # recompute it independently in numpy fp32 and check the gates bit for bit.
    rng = np.random.default_rng(3)
    N = 128
    logits = (rng.standard_normal((16, N)) * 4).astype(np.float32)
    ids, gates = oracle.route(logits, N)
    for t in range(16):
        m = logits[t].max()
        e = oracle.exp_spec((logits[t] - m).astype(np.float32))
        part = np.zeros(32, dtype=np.float32)
        for ln in range(32):
            s = np.float32(0)
            for j in range(ln, N, 32):
                s = np.float32(s + e[j])
            part[ln] = s
        for off in (16, 8, 4, 2, 1):
            part = (part + part[np.arange(32) ^ off]).astype(np.float32)
        Z = part[0]
        ref = (e[ids[t]] / Z).astype(np.float32)
        assert np.array_equal(ref, gates[t])


def test_renormalised_topk_sums_to_one():
    rng = np.random.default_rng(2)
    logits = rng.standard_normal((50, 128)).astype(np.float32)
    ids, gates = oracle.route(logits, 10, renorm_k=8)
    ids0, gates0 = oracle.route(logits, 10)
    assert np.array_equal(ids, ids0)
    assert np.allclose(gates[:, :8].astype(np.float64).sum(1), 1.0, atol=1e-6)
    assert np.array_equal(gates[:, 8:], gates0[:, 8:])


def test_nonfinite_logits_are_rejected():
    logits = np.zeros((2, 8), dtype=np.float32)
    logits[1, 3] = np.nan
    with pytest.raises(RuntimeError):
        oracle.route(logits, 2)
