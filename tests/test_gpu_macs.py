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
from expert_routing_moe_gb300 import _abi as abi

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
                                             (37, 128, "bf16", 0.5), (20000, 256, "bf16", 1.5)])
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


def test_token_weights_reproducible_and_without_rv(g):
    """Bit-identical results on a repeat (fixed-order sums; the last-CTA
    reduction of R_v does not depend on which CTA finishes last), and the
    same weights when R_v is not requested."""
    rng = np.random.default_rng(7)
    T, H = 2000, 512
    x = (rng.standard_normal((T, H)) * rng.uniform(0.2, 4.0, size=(T, 1))).astype(np.float32)
    vis = (rng.random(T) < 0.6).astype(np.uint8)
    x_dev = g.dev(syn.f32_to_bf16_bits(x), torch.bfloat16)
    runs = [_gpu_weights(g, x_dev, vis, 1.5) for _ in range(3)]
    for ent, w, rv in runs[1:]:
        assert np.array_equal(ent, runs[0][0]) and np.array_equal(w, runs[0][1]) and rv == runs[0][2]
    ent = torch.empty(T, dtype=torch.float32, device=g.DEV)
    w = torch.empty(T, dtype=torch.float32, device=g.DEV)
    st = g.status_tensor()
    moe.moe_token_weights(x_dev, g.dev(vis), ent, w, None, 1.5, 1e-6, st)
    torch.cuda.synchronize()
    g.assert_status_ok(st)
    assert np.array_equal(g.host(w), runs[0][1])


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


def test_per_expert_capacity_from_visual_ratio(g):
    """Modality-scaled capacity: weights and R_v from the entropies on the
    GPU, a seeded modality bias per expert; the dispatch is bit-exact against
    the oracle's per-expert capacity on the same weights and ratio, and every
    expert's load stays within its own capacity."""
    import expert_routing_moe_gb300._abi as abi
    L = syn.prefill(with_weights=False)
    vis = L.is_visual.astype(np.uint8)
    x_dev = g.dev(L.x_bf16, torch.bfloat16)
    T = L.T
    ent = torch.empty(T, dtype=torch.float32, device=g.DEV)
    w = torch.empty(T, dtype=torch.float32, device=g.DEV)
    rv = torch.empty(1, dtype=torch.float32, device=g.DEV)
    st = g.status_tensor()
    moe.moe_token_weights(x_dev, g.dev(vis), ent, w, rv, 1.0, 1e-6, st)
    bias = np.random.default_rng(5).integers(-1, 2, L.N).astype(np.int8)
    logits = oracle.router(L.x_bf16, L.w_r, oracle.DT_BF16)
    ids, gates = oracle.route(logits, L.R)
    k, R, N = L.k, L.R, L.N
    i32 = dict(dtype=torch.int32, device=g.DEV)
    ws = torch.empty(abi.workspace_size(abi.MOE_OP_DISPATCH, T, 1, 1, N, k, R, True, 0), dtype=torch.uint8,
                     device=g.DEV)
    counts, offsets, active = torch.empty(N, **i32), torch.empty(N + 1, **i32), torch.empty(N + 1, **i32)
    row_token, row_gate = torch.empty(T * k, **i32), torch.empty(T * k, dtype=torch.float32, device=g.DEV)
    out_ids, out_gates = torch.empty(T, k, **i32), torch.empty(T, k, dtype=torch.float32, device=g.DEV)
    status = torch.empty(T, k, dtype=torch.uint8, device=g.DEV)
    load_q, cap_q = torch.empty(N, dtype=torch.int64, device=g.DEV), torch.empty(1, dtype=torch.int64, device=g.DEV)
    moe.moe_dispatch_capacity(g.dev(ids), g.dev(gates), N, k, R, counts, offsets, row_token, row_gate, active, ws,
                              w, L.gamma, out_ids, out_gates, None, status, load_q, cap_q, st,
                              modality_bias=g.dev(bias), r_v=rv)
    torch.cuda.synchronize()
    g.assert_status_ok(st)
    w_h, r_h = g.host(w), float(rv.item())
    ref = oracle.capacity(ids, gates, N, k, R, w_h, L.gamma, bias=bias, r_v=r_h)
    assert np.array_equal(g.host(out_ids), ref[0])
    assert np.array_equal(g.host(status), ref[2])
    assert np.array_equal(g.host(load_q), ref[3])
    assert int(cap_q.item()) == ref[4]
    S = sum(oracle.fixed_weight(float(v)) for v in w_h)
    Ce = np.array([oracle.capacity_expert(S, k, L.gamma, N, int(bias[e]), r_h) for e in range(N)])
    assert (g.host(load_q) <= Ce).all()
    # a visual-leaning batch (R_v > 1/2) gives visual experts more room than text experts
    assert (r_h > 0.5) == (Ce[bias == 1].min() > Ce[bias == -1].max())


def test_token_weights_empty_batch_clears_rv(g):
    """An empty batch launches nothing but still reports R_v = 0."""
    rv = torch.full((1,), 7.0, dtype=torch.float32, device=g.DEV)
    e = torch.empty(0, dtype=torch.float32, device=g.DEV)
    st = g.status_tensor()
    moe.moe_token_weights(torch.empty(0, 64, dtype=torch.bfloat16, device=g.DEV),
                          torch.empty(0, dtype=torch.uint8, device=g.DEV), e, e, rv, 1.0, 1e-6, st)
    torch.cuda.synchronize()
    g.assert_status_ok(st)
    assert float(rv.item()) == 0.0


def test_token_weights_one_workspace_across_sizes(g):
    """One workspace serves calls of different batch sizes in any order: each
    call matches a call on a fresh workspace bit for bit (the completion
    counter is cleared by every call)."""
    from expert_routing_moe_gb300 import _abi as abi
    rng = np.random.default_rng(11)
    ws = torch.zeros(abi.workspace_size(abi.MOE_OP_TOKEN_WEIGHTS, 20000, 1, 1, 1, 1, 1, False, 0),
                     dtype=torch.uint8, device=g.DEV)
    for T in (2000, 20000, 2000, 37, 20000):
        x = syn.f32_to_bf16_bits((rng.standard_normal((T, 256)) * rng.uniform(0.2, 4.0, size=(T, 1))).astype(np.float32))
        vis = (rng.random(T) < 0.6).astype(np.uint8)
        x_dev, v_dev = g.dev(x, torch.bfloat16), g.dev(vis)
        outs = []
        for w_s in (ws, None):
            ent = torch.empty(T, dtype=torch.float32, device=g.DEV)
            w = torch.empty(T, dtype=torch.float32, device=g.DEV)
            rv = torch.empty(1, dtype=torch.float32, device=g.DEV)
            st = g.status_tensor()
            moe.moe_token_weights(x_dev, v_dev, ent, w, rv, 1.0, 1e-6, st, workspace=w_s)
            torch.cuda.synchronize()
            g.assert_status_ok(st)
            outs.append((g.host(ent), g.host(w), float(rv.item())))
        assert np.array_equal(outs[0][0], outs[1][0]) and np.array_equal(outs[0][1], outs[1][1])
        assert outs[0][2] == outs[1][2]


@pytest.mark.parametrize("dtype,H,T", [("bf16", 2048, 64), ("f32", 512, 64), ("bf16", 4096, 64),
                                       ("bf16", 2048, 5000)])
@pytest.mark.parametrize("bad", ["nan", "+inf", "-inf"])
def test_token_weights_report_a_nonfinite_feature(g, dtype, H, T, bad):
    """One non-finite feature makes its token's entropy non-finite, which sets
    MOE_DEV_NONFINITE with that token as detail; the other tokens' entropies
    are those of the clean batch, bit for bit (at 5000 rows the per-token grid
    runs in more than one wave)."""
    rng = np.random.default_rng(11)
    t_bad, h_bad = 37, H - 3
    x = (rng.standard_normal((T, H)) * 2.0).astype(np.float32)
    vis = (rng.random(T) < 0.7).astype(np.uint8)
    if dtype == "bf16":
        xb = syn.f32_to_bf16_bits(x)
        clean = g.dev(xb, torch.bfloat16)
        xb = xb.copy()
        xb[t_bad, h_bad] = {"nan": 0x7FC0, "+inf": 0x7F80, "-inf": 0xFF80}[bad]
        dirty = g.dev(xb, torch.bfloat16)
    else:
        clean = g.dev(x)
        x = x.copy()
        x[t_bad, h_bad] = {"nan": np.nan, "+inf": np.inf, "-inf": -np.inf}[bad]
        dirty = g.dev(x)
    ent_c, _, _ = _gpu_weights(g, clean, vis)
    ent = torch.empty(T, dtype=torch.float32, device=g.DEV)
    w = torch.empty(T, dtype=torch.float32, device=g.DEV)
    rv = torch.empty(1, dtype=torch.float32, device=g.DEV)
    st = g.status_tensor()
    moe.moe_token_weights(dirty, g.dev(vis), ent, w, rv, 1.0, 1e-6, st)
    torch.cuda.synchronize()
    code, detail = (int(v) for v in st.tolist())
    assert code == abi.MOE_DEV_NONFINITE and detail == t_bad
    ent = g.host(ent)
    assert not np.isfinite(ent[t_bad])
    keep = np.arange(T) != t_bad
    assert np.array_equal(ent[keep], ent_c[keep])

