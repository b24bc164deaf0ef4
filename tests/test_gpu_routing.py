"""GPU parity: ranking, gates and the SERE reroute, bit for bit against the
oracle on the same fp32 logits (the oracle's router output)."""
import numpy as np
import pytest
import torch

import oracle
from expert_routing_moe_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    import _gpu
    return _gpu


def _logits_for(L):
    xd = oracle.DT_BF16 if L.dtype == "bf16" else oracle.DT_F32
    return oracle.router(L.x_bf16 if L.dtype == "bf16" else L.x, L.w_r, xd)


def _random_logits(seed, T, N, tie=True):
    rng = np.random.default_rng(seed)
    l = (rng.standard_normal((T, N)) * 3).astype(np.float32)
    if tie and N > 3:
        l[:, N // 2] = l[:, 0]
        l[::2, 2] = l[::2, 3]
        l[1::3, N - 1] = l[1::3, 1]
    return l


@pytest.mark.parametrize("T,N,R,k", [(16, 8, 2, 2), (16, 8, 8, 2), (32, 128, 8, 8), (33, 128, 10, 8),
                                     (1, 128, 8, 8), (257, 256, 16, 8), (1000, 100, 5, 3), (0, 8, 2, 2)])
def test_rank_bitexact(g, T, N, R, k):
    l = _random_logits(T * 7 + N, T, N)
    ids, gates, st = g.gpu_route(l, R, k)
    g.assert_status_ok(st)
    rid, rg = oracle.route(l, R)
    assert np.array_equal(g.host(ids), rid)
    assert np.array_equal(g.host(gates).view(np.uint32), rg.view(np.uint32))


def test_rank_renorm_bitexact(g):
    l = _random_logits(5, 64, 128)
    ids, gates, st = g.gpu_route(l, 10, 8, renorm=True)
    rid, rg = oracle.route(l, 10, renorm_k=8)
    assert np.array_equal(g.host(ids), rid)
    assert np.array_equal(g.host(gates).view(np.uint32), rg.view(np.uint32))


def test_rank_on_workload_logits(g):
    for L in (syn.tiny(), syn.decode(32, with_weights=False), syn.prefill(with_weights=False)):
        l = _logits_for(L)
        R = L.R
        ids, gates, st = g.gpu_route(l, R, L.k)
        g.assert_status_ok(st)
        rid, rg = oracle.route(l, R)
        assert np.array_equal(g.host(ids), rid)
        assert np.array_equal(g.host(gates).view(np.uint32), rg.view(np.uint32))


def test_nonfinite_logit_sets_device_status(g):
    l = _random_logits(1, 8, 16)
    l[5, 3] = np.inf
    _, _, st = g.gpu_route(l, 4, 4)
    code, detail = (int(v) for v in st.tolist())
    assert code == 1 and detail == 5


def _sere_case(g, L, l, kp, rho, protect, fused=True):
    N, k = L.N, L.k
    sp = g.sere_params(L.sim, kp, rho, protect)
    if fused:
        ids, gates, st = g.gpu_route(l, k, k, sere=sp)
    else:
        ids, gates, st = g.gpu_route(l, k, k)
        from expert_routing_moe_gb300 import moe_reroute_sere
        moe_reroute_sere(ids, gates, N, k, sp, st)
        torch.cuda.synchronize()
    g.assert_status_ok(st)
    rid, rg = oracle.route(l, k)
    eid, eg, bm, stats = oracle.sere(rid, rg, N, k, kp, rho, L.sim, protect)
    assert np.array_equal(g.host(ids), eid)
    assert np.array_equal(g.host(gates).view(np.uint32), eg.view(np.uint32))
    assert np.array_equal(g.host(sp.union_bitmap).view(np.uint32), bm)
    assert np.array_equal(g.host(sp.stats), stats)
    return stats


def test_sere_tiny(g):
    L = syn.tiny()
    stats = _sere_case(g, L, _logits_for(L), L.k_primary, L.rho, None)
    assert stats[0] >= stats[2]


@pytest.mark.parametrize("fused", [True, False])
def test_sere_decode_batch32(g, fused):
    L = syn.decode(32, with_weights=False)
    stats = _sere_case(g, L, _logits_for(L), 2, 0.5, None, fused)
    assert stats[2] < stats[0]


@pytest.mark.parametrize("T", [1, 8, 32, 64, 128])
@pytest.mark.parametrize("kp", [1, 2])
def test_sere_sweep_with_protection(g, T, kp):
    L = syn.sweep(T, with_weights=False)
    stats = _sere_case(g, L, _logits_for(L), kp, 0.5, L.protect)
    assert stats[2] <= stats[0]


def test_sere_closed_forms_on_gpu(g):
    L = syn.decode(64, with_weights=False)
    l = _logits_for(L)
    rid, rg = oracle.route(l, L.k)
    for kp, rho in [(2, 1.5), (L.k, 0.0)]:
        sp = g.sere_params(L.sim, kp, rho)
        ids, gates, st = g.gpu_route(l, L.k, L.k, sere=sp)
        assert np.array_equal(g.host(ids), rid) and np.array_equal(g.host(gates), rg)


def test_sere_random_ties_and_large_batch(g):
    rng = np.random.default_rng(4)
    for T, N, k, kp in [(300, 64, 6, 2), (2048, 128, 8, 2), (17, 33, 5, 1)]:
        l = _random_logits(T + N, T, N)
        sim = rng.random((N, N), dtype=np.float32)
        sim = np.triu(sim, 1)
        sim = (sim + sim.T).astype(np.float32)
        sim[::2, 1] = sim[::2, 0]
        sim[1, ::2] = sim[0, ::2]
        np.fill_diagonal(sim, 1.0)
        prot = (rng.random(N) < 0.2).astype(np.uint8)
        L = syn.Layer(T=T, H=1, N=N, k=k, I=1, dtype="f32", x=None, x_bf16=None, w_r=None, w_gate=None, w_up=None,
                      w_down=None, sim=sim, protect=prot, token_w=None)
        _sere_case(g, L, l, kp, 0.5, prot)
