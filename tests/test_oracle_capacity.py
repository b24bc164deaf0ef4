"""Pins for the oracle's capacity-bounded dispatch (CPU only)."""
import json
import math
import os

import numpy as np
import pytest

import oracle
from expert_routing_moe_gb300 import synthetic as syn
from _props import capacity_check

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "capacity_worked.json")
Q = 1 << 24


@pytest.mark.parametrize("case", json.load(open(GOLDEN))["cases"], ids=lambda c: c["name"])
def test_hand_worked_cases(case):
    ids = np.array(case["ids"], dtype=np.int32)
    gates = np.array(case["gates"], dtype=np.float32)
    w = np.array(case["token_w"], dtype=np.float32)
    oi, og, st, load, C = oracle.capacity(ids, gates, case["N"], case["k"], case["R"], w, case["gamma"])
    assert oi.tolist() == case["expect_ids"]
    assert np.array_equal(og, np.array(case["expect_gates"], dtype=np.float32))
    assert st.tolist() == case["expect_status"]
    assert (load / Q).tolist() == case["expect_load_units"]
    assert C / Q == case["expect_C_units"]


def test_fixed_point_weight_and_capacity_value():
    assert oracle.fixed_weight(1.0) == Q
    assert oracle.fixed_weight(0.0) == 0
    assert oracle.fixed_weight(0.5) == Q // 2
    # Eq. (3) with w == 1: C = gamma |T| k / N tokens
    for T, k, N, g in [(8192, 8, 128, 1.25), (16, 2, 8, 1.25), (100, 3, 7, 1.0), (5, 1, 3, 2.0)]:
        C = oracle.capacity_value(T * Q, k, g, N)
        assert C // Q == math.floor(g * T * k / N)



def test_fixed_point_values_are_exact_floors():
    """The fixed-point weight is w * 2^24 rounded to nearest (ties to even), and
    both capacities are exact floors in those units: C = floor(gamma S k / N) and
    C_j = floor(gamma S k / N * (1 + m_j (R_v - 1/2))), the unfloored static
    value scaled before the floor.  Checked at arbitrary sums S against exact
    rationals, away from integers by more than the double evaluation's error
    (S up to 2^37: 8192 tokens of weight 1)."""
    from fractions import Fraction
    rng = np.random.default_rng(24)
    ws = np.concatenate([rng.random(2000).astype(np.float32),
                         np.float32([2.0 ** -25, 3 * 2.0 ** -25, 5 * 2.0 ** -26, 2.0 ** -24])])
    for w in ws:
        assert oracle.fixed_weight(float(w)) == round(Fraction(float(w)) * Q)   # round(): ties to even
    checked = 0
    while checked < 400:
        S = int(rng.integers(1, 1 << 37))
        k, N = int(rng.integers(1, 17)), int(rng.integers(2, 257))
        g = float(np.float32(rng.uniform(0.25, 2.0)))
        r_v = float(np.float32(rng.random()))
        m = int(rng.integers(-1, 2))
        c = Fraction(S) * k * Fraction(g) / N
        ce = c * (1 + m * (Fraction(r_v) - Fraction(1, 2)))
        margin = max(Fraction(1, 1000), c * Fraction(1, 1 << 48))   # a few double roundings of c
        if min(abs(c - round(c)), abs(ce - round(ce))) < margin:
            continue
        assert oracle.capacity_value(S, k, g, N) == math.floor(c)
        assert oracle.capacity_expert(S, k, g, N, m, r_v) == math.floor(ce)
        checked += 1


def _random_case(rng, T, N, k, R, gate_levels=None):
    logits = rng.standard_normal((T, N)).astype(np.float32)
    ids, gates = oracle.route(logits, R)
    if gate_levels:
        gates = (np.round(gates * gate_levels) / gate_levels).astype(np.float32)  # plant gate ties
    return ids, gates


def test_unit_weights_reduce_to_count_capacity():
    rng = np.random.default_rng(3)
    for _ in range(60):
        T, N = int(rng.integers(1, 40)), int(rng.integers(2, 12))
        k = int(rng.integers(1, min(N, 4) + 1))
        R = k  # no overflow candidates: overflow is dropped
        g = float(rng.choice([0.5, 1.0, 1.25, 2.0]))
        ids, gates = _random_case(rng, T, N, k, R, gate_levels=8)
        oi, og, st, load, C = oracle.capacity(ids, gates, N, k, R, None, g)
        cap_tokens = math.floor(np.float64(np.float32(g)) * T * k / N)
        for e in range(N):
            pairs = [(t, r) for t in range(T) for r in range(k) if ids[t, r] == e]
            pairs.sort(key=lambda p: (-float(gates[p]), p[0]))
            admitted = [p for p in pairs if st[p] == 0]
            assert admitted == pairs[: min(len(pairs), cap_tokens)]
            assert load[e] == len(admitted) * Q


def test_huge_gamma_is_plain_dispatch():
    rng = np.random.default_rng(4)
    for _ in range(30):
        T, N = int(rng.integers(1, 40)), int(rng.integers(2, 16))
        k = int(rng.integers(1, min(N, 4) + 1))
        R = int(rng.integers(k, min(N, 10) + 1))
        ids, gates = _random_case(rng, T, N, k, R)
        w = rng.random(T).astype(np.float32)
        oi, og, st, load, C = oracle.capacity(ids, gates, N, k, R, w, 1e9)
        assert np.array_equal(oi, ids[:, :k]) and np.array_equal(og, gates[:, :k]) and (st == 0).all()


def test_declarative_rules_on_random_tiny_batches():
    rng = np.random.default_rng(9)
    for it in range(250):
        T, N = int(rng.integers(1, 16)), int(rng.integers(2, 9))
        k = int(rng.integers(1, min(N, 3) + 1))
        R = int(rng.integers(k, min(N, 10) + 1))
        ids, gates = _random_case(rng, T, N, k, R, gate_levels=(6 if it % 3 == 0 else None))
        w = rng.beta(2, 5, size=T).astype(np.float32)
        w[rng.random(T) < 0.3] = 1.0
        w[rng.random(T) < 0.05] = 0.0
        g = float(rng.choice([0.5, 0.8, 1.0, 1.25]))
        oi, og, st, load, C = oracle.capacity(ids, gates, N, k, R, w, g)
        capacity_check(ids, gates, w, k, R, g, N, oi, og, st, load, C, oracle.fixed_weight)
        # every slot is admitted, rerouted or dropped exactly once; experts stay distinct per token
        assert set(np.unique(st)) <= {0, 1, 2}
        for t in range(T):
            live = [v for v in oi[t] if v >= 0]
            assert len(live) == len(set(live))
            for r in range(k):
                if st[t, r] == 1:
                    assert oi[t, r] in ids[t, k:R]


def test_prefill_workload_rules():
    L = syn.prefill(with_weights=False)
    logits = syn.skewed_logits(np.random.default_rng(0), L.T, L.N).astype(np.float32)
    ids, gates = oracle.route(logits, L.R)
    oi, og, st, load, C = oracle.capacity(ids, gates, L.N, L.k, L.R, L.token_w, L.gamma)
    S = sum(oracle.fixed_weight(float(v)) for v in L.token_w)
    assert C == oracle.capacity_value(S, L.k, L.gamma, L.N)
    assert (load <= C).all()
    assert (st == 1).sum() > 0  # the skewed popularity makes hot experts overflow
    # the load each expert reports equals the weight of what it finally holds
    wq = np.array([oracle.fixed_weight(float(v)) for v in L.token_w], dtype=np.int64)
    held = np.zeros(L.N, dtype=np.int64)
    for t, r in zip(*np.nonzero(oi >= 0)):
        held[oi[t, r]] += wq[t]
    assert np.array_equal(held, load)


def test_invalid_arguments():
    ids = np.zeros((2, 3), dtype=np.int32)
    g = np.zeros((2, 3), dtype=np.float32)
    with pytest.raises(RuntimeError):
        oracle.capacity(ids, g, 4, 3, 2, None, 1.0)        # R < k
    with pytest.raises(RuntimeError):
        oracle.capacity(ids, g, 4, 2, 3, None, 0.0)        # gamma must be > 0
    with pytest.raises(RuntimeError):
        oracle.capacity(ids, g, 4, 2, 3, np.array([1.0, -1.0], dtype=np.float32), 1.0)  # negative weight


# ---- per-expert capacity: a reading of the truncated [MACS] 3.3 ----------------
def test_expert_capacity_neutral_cases_equal_static():
    """m_j = 0 for every expert, or R_v = 1/2, must give exactly the static dispatch."""
    rng = np.random.default_rng(21)
    for _ in range(40):
        T, N = int(rng.integers(1, 30)), int(rng.integers(2, 10))
        k = int(rng.integers(1, min(N, 3) + 1))
        R = int(rng.integers(k, min(N, 8) + 1))
        ids, gates = _random_case(rng, T, N, k, R)
        w = rng.beta(2, 5, size=T).astype(np.float32)
        g = float(rng.choice([0.5, 1.0, 1.25]))
        ref = oracle.capacity(ids, gates, N, k, R, w, g)
        zero = oracle.capacity(ids, gates, N, k, R, w, g, bias=np.zeros(N, np.int8), r_v=float(rng.random()))
        half = oracle.capacity(ids, gates, N, k, R, w, g, bias=rng.integers(-1, 2, N).astype(np.int8), r_v=0.5)
        for out in (zero, half):
            for a, b in zip(ref, out):
                assert np.array_equal(np.asarray(a), np.asarray(b))


def test_expert_capacity_unit_weights_count_closed_form():
    """With w = 1 each expert admits min(n_e, floor(gamma T k / N * (1 + m (R_v - 1/2)))) of its
    (gate desc, token asc) candidates; the bound is evaluated in exact rationals at parameters
    whose product is at least 1e-3 away from an integer."""
    from fractions import Fraction
    rng = np.random.default_rng(22)
    checked = 0
    while checked < 40:
        T, N = int(rng.integers(4, 40)), int(rng.integers(2, 10))
        k = int(rng.integers(1, min(N, 3) + 1))
        g = float(np.float32(rng.choice([0.5, 0.75, 1.25])))
        r_v = float(np.float32(rng.choice([0.125, 0.25, 0.625, 0.875])))
        bias = rng.integers(-1, 2, N).astype(np.int8)
        ids, gates = _random_case(rng, T, N, k, k, gate_levels=8)
        caps = []
        ok = True
        for e in range(N):
            c = Fraction(g) * T * k / N * (1 + int(bias[e]) * (Fraction(r_v) - Fraction(1, 2)))
            if abs(c - round(c)) < Fraction(1, 1000):
                ok = False
            caps.append(math.floor(c))
        if not ok:
            continue
        oi, og, st, load, C = oracle.capacity(ids, gates, N, k, k, None, g, bias=bias, r_v=r_v)
        for e in range(N):
            pairs = [(t, r) for t in range(T) for r in range(k) if ids[t, r] == e]
            pairs.sort(key=lambda p: (-float(gates[p]), p[0]))
            admitted = [p for p in pairs if st[p] == 0]
            assert admitted == pairs[: min(len(pairs), caps[e])]
            assert oracle.capacity_expert(T * Q, k, g, N, int(bias[e]), r_v) // Q == caps[e]
        checked += 1


def test_expert_capacity_monotone_in_r_v():
    S, k, g, N = 4096 * Q, 8, 1.25, 128
    vis = [oracle.capacity_expert(S, k, g, N, +1, r) for r in (0.0, 0.25, 0.5, 0.75, 1.0)]
    txt = [oracle.capacity_expert(S, k, g, N, -1, r) for r in (0.0, 0.25, 0.5, 0.75, 1.0)]
    base = oracle.capacity_value(S, k, g, N)
    assert vis == sorted(vis) and txt == sorted(txt, reverse=True)
    assert vis[2] == txt[2] == base
    assert vis[4] == txt[0] and vis[0] == txt[4]


def test_expert_capacity_declarative_rules():
    rng = np.random.default_rng(23)
    for it in range(150):
        T, N = int(rng.integers(1, 16)), int(rng.integers(2, 9))
        k = int(rng.integers(1, min(N, 3) + 1))
        R = int(rng.integers(k, min(N, 10) + 1))
        ids, gates = _random_case(rng, T, N, k, R, gate_levels=(6 if it % 3 == 0 else None))
        w = rng.beta(2, 5, size=T).astype(np.float32)
        w[rng.random(T) < 0.3] = 1.0
        g = float(rng.choice([0.5, 0.8, 1.0, 1.25]))
        bias = rng.integers(-1, 2, N).astype(np.int8)
        r_v = float(np.float32(rng.random()))
        oi, og, st, load, C = oracle.capacity(ids, gates, N, k, R, w, g, bias=bias, r_v=r_v)
        S = sum(oracle.fixed_weight(float(v)) for v in w)
        Ce = np.array([oracle.capacity_expert(S, k, g, N, int(bias[e]), r_v) for e in range(N)])
        capacity_check(ids, gates, w, k, R, g, N, oi, og, st, load, Ce, oracle.fixed_weight)


def test_expert_capacity_rejects_bad_bias_or_ratio():
    ids = np.zeros((2, 3), dtype=np.int32)
    g = np.zeros((2, 3), dtype=np.float32)
    with pytest.raises(Exception):
        oracle.capacity(ids, g, 4, 2, 3, None, 1.0, bias=np.array([0, 2, 0, 0], np.int8), r_v=0.5)
    with pytest.raises(Exception):
        oracle.capacity(ids, g, 4, 2, 3, None, 1.0, bias=np.zeros(4, np.int8), r_v=1.5)
