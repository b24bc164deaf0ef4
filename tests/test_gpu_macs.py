"""GPU parity of the MACS entropy-weighted token load (moe_token_weights)
against the oracle, and the capacity dispatch fed with those weights.

Tolerances from the fp32 arithmetic of the entropy: Z and S1 are sums of
D positive terms, so their relative error is at most D * 2^-24 (1.2e-4 at
D = 2048); the entropy is checked to 2e-4 * max(1, |H|).  The weights are a
sigmoid of the z-score with slope at most delta / (4 sigma), so they are
checked to that slope times the entropy tolerance (plus the statistics'
share), and R_v to the same bound."""
import numpy as np
import pytest
import torch

import oracle
import expert_routing_moe_gb300 as moe
from expert_routing_moe_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    import _gpu
    return _gpu


def _gpu_weights(g, x_dev, vis, delta=1.0, eps=1e-6):
    T = x_dev.shape[0]
    ent = torch.empty(T, dtype=torch.float32, device=g.DEV)
    w = torch.empty(T, dtype=torch.float32, device=g.DEV)
    rv = torch.empty(1, dtype=torch.float32, device=g.DEV)
    st = g.status_tensor()
    moe.moe_token_weights(x_dev, g.dev(vis.astype(np.uint8)), ent, w, rv, delta, eps, st)
    torch.cuda.synchronize()
    g.assert_status_ok(st)
    return g.host(ent), g.host(w), float(rv.item())


@pytest.mark.parametrize("T,H,dtype,delta", [(8192, 2048, "bf16", 1.0), (300, 256, "f32", 2.5),
                                             (37, 128, "bf16", 0.5)])
def test_token_weights_match_oracle(g, T, H, dtype, delta):
    if H == 2048:
        L = syn.prefill(T, with_weights=False)
        vis = L.is_visual.astype(np.uint8)
        xb = L.x_bf16
    else:
        rng = np.random.default_rng(T)
        x = (rng.standard_normal((T, H)) * rng.uniform(0.2, 4.0, size=(T, 1))).astype(np.float32)
        vis = (rng.random(T) < 0.7).astype(np.uint8)
        xb = syn.f32_to_bf16_bits(x) if dtype == "bf16" else x
    if dtype == "bf16":
        x_dev = g.dev(xb, torch.bfloat16)
        ent_r, w_r, rv_r = oracle.token_weights(xb, vis, delta, 1e-6, oracle.DT_BF16)
    else:
        x_dev = g.dev(xb)
        ent_r, w_r, rv_r = oracle.token_weights(xb, vis, delta, 1e-6)
    ent, w, rv = _gpu_weights(g, x_dev, vis, delta)
    tol_h = 2e-4 * np.maximum(1.0, np.abs(ent_r))
    assert np.all(np.abs(ent - ent_r) <= tol_h)
    sig = np.std(ent_r[vis == 1]) if vis.any() else 1.0
    tol_w = delta / (4 * sig) * 4 * float(tol_h.max()) + 1e-6
    assert np.all(np.abs(w - w_r) <= tol_w), float(np.max(np.abs(w - w_r)))
    assert np.all(w[vis == 0] == 1.0)
    assert abs(rv - rv_r) <= tol_w


def test_token_weights_closed_forms_on_gpu(g):
    D = 512
    x = np.zeros((4, D), np.float32)
    x[1] = 2.5                                   # uniform: ln D
    x[2, 3] = 6.0                                # one raised entry
    vis = np.array([1, 1, 1, 0], np.uint8)
    ent, w, rv = _gpu_weights(g, g.dev(x), vis, delta=0.0)
    assert abs(ent[0] - np.log(D)) < 1e-5 and abs(ent[1] - np.log(D)) < 1e-5
    den = np.exp(6.0) + D - 1
    p0, q = np.exp(6.0) / den, 1.0 / den
    assert abs(ent[2] - (-p0 * np.log(p0) - (D - 1) * q * np.log(q))) < 1e-5
    assert np.all(w[:3] == 0.5) and w[3] == 1.0      # delta = 0
    assert abs(rv - 1.5 / 2.5) < 1e-7
    _, _, rv_t = _gpu_weights(g, g.dev(x), np.zeros(4, np.uint8))
    assert rv_t == 0.0


def test_capacity_dispatch_with_entropy_weights(g):
    """The prefill batch with its load weights from the entropies (instead of
    the Beta(2,5) draw): the capacity dispatch on the GPU weights is
    bit-exact against the oracle's capacity on the same weights."""
    L = syn.prefill(with_weights=False)
    vis = L.is_visual.astype(np.uint8)
    x_dev = g.dev(L.x_bf16, torch.bfloat16)
    _, w, _ = _gpu_weights(g, x_dev, vis, 1.0)
    logits = oracle.router(L.x_bf16, L.w_r, oracle.DT_BF16)
    ids, gates = oracle.route(logits, L.R)
    d = g.gpu_dispatch(g.dev(ids), g.dev(gates), L.N, L.k, L.R, token_w=g.dev(w.astype(np.float32)),
                       gamma=L.gamma)
    ref = oracle.capacity(ids, gates, L.N, L.k, L.R, w.astype(np.float32), L.gamma)
    assert np.array_equal(d["out_ids"], ref[0])
    assert np.array_equal(d["status"], ref[2])
    assert np.array_equal(d["load"], ref[3])
