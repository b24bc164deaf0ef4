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


def test_capacity_large_and_small_from_two_host_threads(g):
    """A large and a small capped dispatch issued over and over from two host
    threads, each on its own stream: neither call's launch configuration may
    be undone by the other's (the admission kernel's shared-memory limit is
    raised once per device to the largest size), and each result stays
    bit-identical to the same call made alone."""
    import threading
    import torch
    from expert_routing_moe_gb300 import _abi as abi

    L = syn.prefill(with_weights=False)
    l = oracle.router(L.x_bf16, L.w_r, oracle.DT_BF16)
    ids_big, gates_big = oracle.route(l, L.R)
    tw_big = L.token_w
    small_T = 16
    ids_small, gates_small, tw_small = ids_big[:small_T].copy(), gates_big[:small_T].copy(), tw_big[:small_T].copy()

    def run(ids, gates, tw, stream, reps, results, errors):
        try:
            T = ids.shape[0]
            dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to("cuda:0")
            di, dg, dw = dev(ids), dev(gates), dev(tw)
            n = abi.workspace_size(abi.MOE_OP_DISPATCH, T, 1, 1, L.N, L.k, L.R, True, 0)
            ws = torch.empty(max(n, 256), dtype=torch.uint8, device="cuda:0")
            i32 = dict(dtype=torch.int32, device="cuda:0")
            for _ in range(reps):
                o = dict(counts=torch.full((L.N,), -7, **i32), offsets=torch.full((L.N + 1,), -7, **i32),
                         active=torch.full((L.N + 1,), -7, **i32), row_token=torch.full((T * L.k,), -7, **i32),
                         row_gate=torch.full((T * L.k,), -7.0, dtype=torch.float32, device="cuda:0"),
                         status=torch.full((T, L.k), 77, dtype=torch.uint8, device="cuda:0"))
                st = torch.zeros(2, dtype=torch.int32, device="cuda:0")
                with torch.cuda.stream(stream):
                    abi.moe_dispatch_capacity(di, dg, L.N, L.k, L.R, o["counts"], o["offsets"], o["row_token"],
                                              o["row_gate"], o["active"], ws, token_w=dw,
                                              capacity_factor=L.gamma, slot_status=o["status"], st=st,
                                              stream=stream)
                stream.synchronize()
                assert st.tolist() == [0, 0]
                results.append({name: t.cpu().numpy() for name, t in o.items()})
        except Exception as e:  # reported by the main thread
            errors.append(e)

    # each call made alone first, on the default stream
    solo = {}
    for name, (ids, gates, tw) in dict(big=(ids_big, gates_big, tw_big),
                                        small=(ids_small, gates_small, tw_small)).items():
        res, err = [], []
        run(ids, gates, tw, torch.cuda.current_stream(), 1, res, err)
        assert not err, err
        solo[name] = res[0]
    res_big, res_small, errors = [], [], []
    th = [threading.Thread(target=run, args=(ids_big, gates_big, tw_big, torch.cuda.Stream(), 6, res_big, errors)),
          threading.Thread(target=run, args=(ids_small, gates_small, tw_small, torch.cuda.Stream(), 40, res_small,
                                             errors))]
    for t in th:
        t.start()
    for t in th:
        t.join()
    assert not errors, errors
    assert len(res_big) == 6 and len(res_small) == 40
    for name, results in (("big", res_big), ("small", res_small)):
        for r in results:
            for key in r:
                assert np.array_equal(r[key].view(np.uint8), solo[name][key].view(np.uint8)), (name, key)
