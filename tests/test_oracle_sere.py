"""Pins for the oracle's SERE batch reroute (CPU only)."""
import json
import os

import numpy as np
import pytest

import oracle
from expert_routing_moe_gb300 import synthetic as syn
from _props import check_sere

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "sere_worked.json")


def _gate(v):
    if isinstance(v, str):
        a, b = v.split("+")
        return np.float32(np.float32(float(a)) + np.float32(float(b)))
    return np.float32(v)


@pytest.mark.parametrize("case", json.load(open(GOLDEN))["cases"], ids=lambda c: c["name"])
def test_hand_worked_cases(case):
    N, k = case["N"], case["k"]
    sim = np.full((N, N), case["sim_default"], dtype=np.float32)
    np.fill_diagonal(sim, 1.0)
    for a, b, v in case["sim_entries"]:
        sim[a, b] = sim[b, a] = v
    ids = np.array(case["ids"], dtype=np.int32)
    gates = np.array(case["gates"], dtype=np.float32)
    prot = None if case["protect"] is None else np.array(case["protect"], dtype=np.uint8)
    ids1, g1, bitmap, stats = oracle.sere(ids, gates, N, k, case["k_primary"], case["rho"], sim, prot)
    assert ids1.tolist() == case["expect_ids"]
    want = np.array([[_gate(v) for v in row] for row in case["expect_gates"]], dtype=np.float32)
    assert np.array_equal(g1, want)
    assert stats.tolist() == case["expect_stats"]
    P = [p for p in range(N) if bitmap[p // 32] >> (p % 32) & 1]
    assert P == case["expect_P"]


def _random_case(rng, T, N, k):
    logits = rng.standard_normal((T, N)).astype(np.float32)
    ids, gates = oracle.route(logits, k)
    sim = rng.random((N, N), dtype=np.float32)
    sim = np.triu(sim, 1)
    sim = (sim + sim.T).astype(np.float32)
    np.fill_diagonal(sim, 1.0)
    # plant similarity ties so the lower-id rule is exercised
    sim[::2, 1] = sim[::2, 0]
    sim[1, ::2] = sim[0, ::2]
    np.fill_diagonal(sim, 1.0)
    return ids, gates, sim


def test_rho_above_one_or_all_primary_is_plain_topk():
    rng = np.random.default_rng(1)
    for _ in range(40):
        T, N = int(rng.integers(1, 20)), int(rng.integers(2, 40))
        k = int(rng.integers(1, min(N, 8) + 1))
        ids, gates, sim = _random_case(rng, T, N, k)
        kp = int(rng.integers(1, k + 1))
        a, b, _, st = oracle.sere(ids, gates, N, k, kp, 1.0001, sim)
        assert np.array_equal(a, ids) and np.array_equal(b, gates) and st[3] == st[4] == 0
        a, b, _, _ = oracle.sere(ids, gates, N, k, k, 0.0, sim)
        assert np.array_equal(a, ids) and np.array_equal(b, gates)
        # sim <= 1 everywhere and the strict threshold: rho = 1 never reroutes either
        a, b, _, _ = oracle.sere(ids, gates, N, k, kp, 1.0, sim)
        assert np.array_equal(a, ids)


def test_declarative_properties_on_random_tiny_batches():
    rng = np.random.default_rng(7)
    for it in range(300):
        T, N = int(rng.integers(1, 24)), int(rng.integers(2, 20))
        k = int(rng.integers(1, min(N, 8) + 1))
        kp = int(rng.integers(1, k + 1))
        rho = float(rng.choice([0.0, 0.3, 0.5, 0.7]))
        ids, gates, sim = _random_case(rng, T, N, k)
        prot = (rng.random(N) < 0.3).astype(np.uint8) if it % 2 else None
        a, b, bitmap, st = oracle.sere(ids, gates, N, k, kp, rho, sim, prot)
        P = check_sere(ids, gates, a, b, k, kp, rho, sim, prot, st)
        assert [p for p in range(N) if bitmap[p // 32] >> (p % 32) & 1] == P
        # per-token gate mass is preserved (fp32 adds only)
        assert np.allclose(b.astype(np.float64).sum(1), gates.astype(np.float64).sum(1), rtol=1e-6)
        # protected sources outside P never move
        if prot is not None:
            for t in range(T):
                for r in range(kp, k):
                    s = ids[t, r]
                    if prot[s] and s not in P:
                        assert a[t, r] == s and b[t, r] >= gates[t, r]
        # slot accounting: every secondary is kept, moved or merged exactly once
        nsec = sum(1 for t in range(T) for r in range(kp, k) if ids[t, r] not in P)
        assert st[3] + st[4] + st[5] + st[6] == nsec


def test_union_never_grows_on_the_decode_workload():
    L = syn.decode(32, with_weights=False)
    logits = oracle.router(L.x_bf16, L.w_r, oracle.DT_BF16)
    ids, gates = oracle.route(logits, L.k)
    a, b, _, st = oracle.sere(ids, gates, L.N, L.k, 2, 0.5, L.sim, None)
    check_sere(ids, gates, a, b, L.k, 2, 0.5, L.sim, None, st)
    assert st[2] <= st[0]
    assert st[2] < st[0]  # the clustered similarity makes SERE shrink the union here
    # protection can only keep more experts alive
    prot = syn.protect_bits(np.random.default_rng(0), L.N, 16)
    a2, b2, _, st2 = oracle.sere(ids, gates, L.N, L.k, 2, 0.5, L.sim, prot)
    check_sere(ids, gates, a2, b2, L.k, 2, 0.5, L.sim, prot, st2)
    assert st2[2] >= st[2]


def test_invalid_arguments():
    ids = np.zeros((2, 3), dtype=np.int32)
    g = np.zeros((2, 3), dtype=np.float32)
    sim = np.eye(4, dtype=np.float32)
    with pytest.raises(RuntimeError):
        oracle.sere(ids, g, 4, 3, 0, 0.5, sim)      # K' must be >= 1
    with pytest.raises(RuntimeError):
        oracle.sere(ids, g, 4, 3, 4, 0.5, sim)      # K' must be <= k
    bad = ids.copy()
    bad[0, 0] = 9
    with pytest.raises(RuntimeError):
        oracle.sere(bad, g, 4, 3, 1, 0.5, sim)      # id out of range
