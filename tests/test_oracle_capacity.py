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
