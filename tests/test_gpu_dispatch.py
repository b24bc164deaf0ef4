"""GPU parity: expert-sorted permutation and capacity dispatch, bit for bit
against the oracle on the same routing."""
import json
import os

import numpy as np
import pytest

import oracle
from expert_routing_moe_gb300 import synthetic as syn
from _props import capacity_check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    import _gpu
    return _gpu


def _check_perm(d, ids, gates, N, k):
    ref = oracle.permute(ids, gates, N, k)
    assert np.array_equal(d["counts"], ref["counts"])
    assert np.array_equal(d["offsets"], ref["offsets"])
    assert np.array_equal(d["active"][:1 + ref["active"][0]], ref["active"][:1 + ref["active"][0]])
    assert np.array_equal(d["row_token"], ref["row_token"])
    assert np.array_equal(d["row_gate"].view(np.uint32), ref["row_gate"].view(np.uint32))
    # slot_row is the inverse map: every slot with an expert points at its row
    T = ids.shape[0]
    for t in range(T):
        for r in range(k):
            row = d["slot_row"][t, r]
            if ids[t, r] >= 0:
                assert d["row_token"][row] == t and ref["offsets"][ids[t, r]] <= row < ref["offsets"][ids[t, r] + 1]
            else:
                assert row == -1


@pytest.mark.parametrize("T,N,k,holes", [(0, 8, 2, 0.0), (1, 128, 8, 0.0), (16, 8, 2, 0.0), (32, 128, 8, 0.1),
                                         (1024, 128, 8, 0.0), (1025, 128, 8, 0.05), (2500, 64, 4, 0.2),
                                         (8192, 128, 8, 0.0), (300, 256, 16, 0.3)])
def test_permute_bitexact(g, T, N, k, holes):
    rng = np.random.default_rng(T * 3 + N)
    pop = rng.dirichlet(0.3 * np.ones(N))
    ids = np.stack([rng.choice(N, size=k, replace=False, p=pop) for _ in range(T)]).astype(np.int32) \
        if T else np.zeros((0, k), np.int32)
    ids[rng.random(ids.shape) < holes] = -1
    gates = rng.random(ids.shape).astype(np.float32)
    d = g.gpu_dispatch(g.dev(ids), g.dev(gates), N, k, k)
    _check_perm(d, ids, gates, N, k)
    assert np.array_equal(d["out_ids"], ids)


def _capacity_case(g, ids, gates, N, k, R, w, gamma):
    d = g.gpu_dispatch(g.dev(ids), g.dev(gates), N, k, R, None if w is None else w, gamma)
    oi, og, st, load, C = oracle.capacity(ids, gates, N, k, R, w, gamma)
    assert d["cap"] == C
    assert np.array_equal(d["status"], st)
    assert np.array_equal(d["out_ids"], oi)
    assert np.array_equal(d["out_gates"].view(np.uint32), og.view(np.uint32))
    assert np.array_equal(d["load"], load)
    _check_perm(d, oi, og, N, k)
    return d


def test_capacity_worked_cases(g):
    cases = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "capacity_worked.json")))["cases"]
    for c in cases:
        d = _capacity_case(g, np.array(c["ids"], np.int32), np.array(c["gates"], np.float32), c["N"], c["k"],
                           c["R"], np.array(c["token_w"], np.float32), c["gamma"])
        assert d["out_ids"].tolist() == c["expect_ids"]


def test_capacity_tiny_layer(g):
    L = syn.tiny(capacity=True)
    l = oracle.router(L.x, L.w_r)
    ids, gates = oracle.route(l, L.R)
    _capacity_case(g, ids, gates, L.N, L.k, L.R, L.token_w, L.gamma)


def test_capacity_random_with_ties(g):
    rng = np.random.default_rng(12)
    for it in range(40):
        T, N = int(rng.integers(1, 300)), int(rng.integers(2, 40))
        k = int(rng.integers(1, min(N, 4) + 1))
        R = int(rng.integers(k, min(N, 10) + 1))
        l = (rng.standard_normal((T, N)) * 2).astype(np.float32)
        ids, gates = oracle.route(l, R)
        if it % 2:
            gates = (np.round(gates * 8) / 8).astype(np.float32)
        w = rng.beta(2, 5, size=T).astype(np.float32)
        w[rng.random(T) < 0.3] = 1.0
        gamma = float(rng.choice([0.5, 1.0, 1.25]))
        d = _capacity_case(g, ids, gates, N, k, R, w, gamma)
        if T <= 40:
            capacity_check(ids, gates, w, k, R, gamma, N, d["out_ids"], d["out_gates"], d["status"], d["load"],
                           d["cap"], oracle.fixed_weight)


def test_capacity_prefill_full_size(g):
    L = syn.prefill(with_weights=False)
    l = oracle.router(L.x_bf16, L.w_r, oracle.DT_BF16)
    ids, gates = oracle.route(l, L.R)
    d = _capacity_case(g, ids, gates, L.N, L.k, L.R, L.token_w, L.gamma)
    assert (d["status"] == 1).sum() > 0 and (d["load"] <= d["cap"]).all()
