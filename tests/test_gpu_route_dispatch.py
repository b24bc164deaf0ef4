"""GPU parity of the single-launch decode routing + dispatch
(moe_route_dispatch): bit-identical to moe_route (with and without SERE)
followed by the uncapped moe_dispatch_capacity, and -- given its own fp32
logits -- to the oracle's ranking, SERE reroute and permutation, over batch
sizes from 1 to the 256-token maximum, ragged tails, expert counts that are
not multiples of the router tile, protection, rho > 1 and renormalised
gates."""
import numpy as np
import pytest
import torch

import oracle
import expert_routing_moe_gb300 as moe
from expert_routing_moe_gb300 import _abi as abi
from expert_routing_moe_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    import _gpu
    return _gpu


@pytest.fixture(scope="module")
def ws():
    n = abi.workspace_size(abi.MOE_OP_ROUTE_DISPATCH, 1, 1, 1, 1, 1, 1, False, 0)
    return torch.zeros(max(n, 256), dtype=torch.uint8, device="cuda:0")


def _buffers(T, N, k):
    i32 = dict(dtype=torch.int32, device="cuda:0")
    f32 = dict(dtype=torch.float32, device="cuda:0")
    return dict(logits=torch.full((T, N), -7.0, **f32), ids=torch.full((T, k), -7, **i32),
                gates=torch.full((T, k), -7.0, **f32), counts=torch.full((N,), -7, **i32),
                offsets=torch.full((N + 1,), -7, **i32), row_token=torch.full((max(T * k, 1),), -7, **i32),
                row_gate=torch.full((max(T * k, 1),), -7.0, **f32), active=torch.full((N + 1,), -7, **i32))


def _sere(g, sim, kp, rho, protect, N):
    return None if sim is None else g.sere_params(sim, kp, rho, protect)


def _fused(g, x, w_r, k, ws, sim=None, kp=2, rho=0.5, protect=None, renorm=False):
    T, N = x.shape[0], w_r.shape[0]
    b = _buffers(T, N, k)
    sp = _sere(g, sim, kp, rho, protect, N)
    st = g.status_tensor()
    moe.moe_route_dispatch(x, w_r, b["logits"], b["ids"], b["gates"], b["counts"], b["offsets"], b["row_token"],
                           b["row_gate"], b["active"], ws, abi.MOE_ROUTE_RENORM_TOPK if renorm else 0, sp, st)
    torch.cuda.synchronize()
    g.assert_status_ok(st)
    out = {n: g.host(t) for n, t in b.items()}
    if sp is not None:
        out["bitmap"], out["stats"] = g.host(sp.union_bitmap), g.host(sp.stats)
    return out


def _separate(g, x, w_r, k, sim=None, kp=2, rho=0.5, protect=None, renorm=False):
    T, N = x.shape[0], w_r.shape[0]
    b = _buffers(T, N, k)
    sp = _sere(g, sim, kp, rho, protect, N)
    st = g.status_tensor()
    moe.moe_route(x, w_r, b["logits"], b["ids"], b["gates"], k, abi.MOE_ROUTE_RENORM_TOPK if renorm else 0, sp, st)
    wsd = torch.empty(max(abi.workspace_size(abi.MOE_OP_DISPATCH, T, 1, 1, N, k, k, False, 0), 256),
                      dtype=torch.uint8, device="cuda:0")
    moe.moe_dispatch_capacity(b["ids"], b["gates"], N, k, k, b["counts"], b["offsets"], b["row_token"],
                              b["row_gate"], b["active"], wsd, st=st)
    torch.cuda.synchronize()
    g.assert_status_ok(st)
    out = {n: g.host(t) for n, t in b.items()}
    if sp is not None:
        out["bitmap"], out["stats"] = g.host(sp.union_bitmap), g.host(sp.stats)
    return out


def _same_bits(a, b, name):
    assert a.shape == b.shape, name
    assert np.array_equal(a.view(np.uint32) if a.dtype == np.float32 else a,
                          b.view(np.uint32) if b.dtype == np.float32 else b), name


def _check_oracle(f, k, N, sim=None, kp=2, rho=0.5, protect=None, renorm=False):
    """The fused outputs against the oracle on the fused kernel's own logits."""
    ids, gates = oracle.route(f["logits"], k, renorm_k=k if renorm else 0)
    if sim is not None:
        ids, gates, bitmap, stats = oracle.sere(ids, gates, N, k, kp, rho, sim, protect)
        assert np.array_equal(f["bitmap"].view(np.uint32), bitmap)
        assert np.array_equal(f["stats"], stats)
    assert np.array_equal(f["ids"], ids)
    assert np.array_equal(f["gates"].view(np.uint32), gates.view(np.uint32))
    p = oracle.permute(ids, gates, N, k)
    m = int(p["offsets"][N])
    for name in ("counts", "offsets"):
        assert np.array_equal(f[name], p[name]), name
    na = int(p["active"][0])   # entries past the active count are unspecified
    assert np.array_equal(f["active"][:1 + na], p["active"][:1 + na])
    assert np.array_equal(f["row_token"][:m], p["row_token"])
    assert np.array_equal(f["row_gate"][:m].view(np.uint32), p["row_gate"].view(np.uint32))


@pytest.mark.parametrize("T", [1, 8, 32, 37, 64, 128, 256])
@pytest.mark.parametrize("sere", [False, True])
def test_decode_matches_separate_calls_and_oracle(g, ws, T, sere):
    L = syn.sweep(T, with_weights=False)
    D = g.DevLayer(L, weights=False)
    kw = dict(sim=D.sim, kp=L.k_primary, rho=L.rho, protect=D.protect) if sere else {}
    f = _fused(g, D.x, D.w_r, L.k, ws, **kw)
    s = _separate(g, D.x, D.w_r, L.k, **kw)
    for name in f:
        _same_bits(f[name], s[name], name)
    okw = dict(sim=L.sim, kp=L.k_primary, rho=L.rho, protect=L.protect) if sere else {}
    _check_oracle(f, L.k, L.N, **okw)
    # the router's fp32 logits agree with the oracle's double-accumulated ones to rounding
    ref = oracle.router(L.x_bf16, L.w_r, oracle.DT_BF16)
    xabs = np.abs(L.x.astype(np.float64)) @ np.abs(L.w_r.astype(np.float64)).T
    assert np.all(np.abs(f["logits"] - ref) <= L.H * 2.0 ** -24 * xabs + 1e-30)


def test_tiny_fp32_layer_and_degenerate_settings(g, ws):
    """N = 8 (one partial router tile), fp32 x, K' = 1; rho > 1 and K' = k
    reproduce plain top-k exactly; renormalised gates."""
    L = syn.tiny()
    D = g.DevLayer(L, weights=False)
    plain = _fused(g, D.x, D.w_r, L.k, ws)
    _check_oracle(plain, L.k, L.N)
    f = _fused(g, D.x, D.w_r, L.k, ws, sim=D.sim, kp=1, rho=0.5)
    _check_oracle(f, L.k, L.N, sim=L.sim, kp=1, rho=0.5)
    for kp, rho in ((1, 1.5), (L.k, 0.5)):
        f = _fused(g, D.x, D.w_r, L.k, ws, sim=D.sim, kp=kp, rho=rho)
        for name in ("ids", "gates", "counts", "offsets", "row_token", "row_gate", "active"):
            _same_bits(f[name], plain[name], name)
    r = _fused(g, D.x, D.w_r, L.k, ws, renorm=True)
    _check_oracle(r, L.k, L.N, renorm=True)


def test_ragged_expert_count(g, ws):
    """N = 60 experts (router tiles of 8 with a ragged last tile), T = 19."""
    rng = np.random.default_rng(5)
    T, H, N, k = 19, 256, 60, 6
    x = rng.standard_normal((T, H)).astype(np.float32)
    w_r = (rng.standard_normal((N, H)) / np.sqrt(H)).astype(np.float32)
    sim = rng.uniform(0, 1, (N, N)).astype(np.float32)
    sim = ((sim + sim.T) / 2).astype(np.float32)
    np.fill_diagonal(sim, 1.0)
    prot = (rng.random(N) < 0.2).astype(np.uint8)
    f = _fused(g, g.dev(x), g.dev(w_r), k, ws, sim=g.dev(sim), kp=2, rho=0.4, protect=g.dev(prot))
    _check_oracle(f, k, N, sim=sim, kp=2, rho=0.4, protect=prot)
    assert f["stats"][3] + f["stats"][4] > 0   # some slots moved or merged


def test_repeated_calls_leave_workspace_reusable(g, ws):
    """Every call resets the completion counter: repeated calls give
    identical results (graph replays of whole steps are covered by the
    layer tests)."""
    L = syn.decode(32, with_weights=False)
    D = g.DevLayer(L, weights=False)
    first = _fused(g, D.x, D.w_r, L.k, ws, sim=D.sim)
    for _ in range(3):
        again = _fused(g, D.x, D.w_r, L.k, ws, sim=D.sim)
        for name in first:
            _same_bits(again[name], first[name], name)
    assert int(ws.view(torch.int32)[0].item()) == 0


def test_empty_batch(g, ws):
    N, k = 16, 2
    b = _buffers(0, N, k)
    x = torch.empty(0, 64, dtype=torch.float32, device="cuda:0")
    w_r = torch.zeros(N, 64, dtype=torch.float32, device="cuda:0")
    moe.moe_route_dispatch(x, w_r, b["logits"], b["ids"], b["gates"], b["counts"], b["offsets"], b["row_token"],
                           b["row_gate"], b["active"], ws)
    torch.cuda.synchronize()
    assert g.host(b["counts"]).tolist() == [0] * N
    assert g.host(b["offsets"]).tolist() == [0] * (N + 1)
    assert g.host(b["active"])[0] == 0
    # with SERE, the union bitmap and the statistics of an empty batch are
    # zero too, not what the previous call left there
    sim = torch.eye(N, dtype=torch.float32, device="cuda:0")
    sp = g.sere_params(sim, 1, 0.5)
    sp.union_bitmap.fill_(-1)
    sp.stats.fill_(-7)
    b = _buffers(0, N, k)
    moe.moe_route_dispatch(x, w_r, b["logits"], b["ids"], b["gates"], b["counts"], b["offsets"], b["row_token"],
                           b["row_gate"], b["active"], ws, 0, sp)
    torch.cuda.synchronize()
    assert g.host(sp.union_bitmap).tolist() == [0] * ((N + 31) // 32)
    assert g.host(sp.stats).tolist() == [0] * 8
    assert g.host(b["counts"]).tolist() == [0] * N


def test_layer_forward_uses_single_launch_path(g):
    """MoELayer picks the single launch for uncapped decode batches; its
    output matches the separate calls' bit for bit."""
    L = syn.decode(32)
    D = g.DevLayer(L)
    lay = moe.MoELayer(D.w_r, D.w_gate, D.w_up, D.w_down, k=L.k, max_tokens=L.T, sim=D.sim, k_primary=2, rho=0.5)
    assert lay.fused_route_dispatch_ok(L.T)
    y1 = lay.forward(D.x, sere=True).clone()
    rows1 = g.host(lay.row_token[:int(lay.offsets[L.N].item())])
    lay.route(D.x, True)
    lay.dispatch(L.T)
    lay.ffn(D.x)
    torch.cuda.synchronize()
    rows2 = g.host(lay.row_token[:int(lay.offsets[L.N].item())])
    assert np.array_equal(rows1, rows2)
    assert torch.equal(y1, lay.y[:L.T]) or float((y1 - lay.y[:L.T]).abs().max()) <= 1e-6 * float(
        y1.abs().max())
    # the same layer into a caller's buffer (zeroed inside the FFN launch)
    buf = torch.full((L.T, L.H), float("nan"), dtype=torch.float32, device="cuda:0")
    y3 = lay.forward(D.x, sere=True, out=buf)
    torch.cuda.synchronize()
    assert y3.data_ptr() == buf.data_ptr()
    assert float((y3 - y1).abs().max()) <= 1e-6 * float(y1.abs().max())


@pytest.mark.parametrize("T,N,k,H", [(128, 256, 16, 256), (100, 200, 12, 192), (256, 96, 8, 128)])
def test_limits_and_ragged_tiles(g, ws, T, N, k, H):
    """The largest slot count (T k = 2048) with N = 256 and k = 16, an expert
    count that is not a multiple of 32 (partial last lane word) and of the
    router tile of 8, and bf16 x: bit-identical to the separate calls and
    to the oracle given the kernel's logits, with and without SERE."""
    rng = np.random.default_rng(T + N + k)
    x = syn.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    w_r = (rng.standard_normal((N, H)) / np.sqrt(H)).astype(np.float32)
    sim = rng.uniform(0, 1, (N, N)).astype(np.float32)
    sim = ((sim + sim.T) / 2).astype(np.float32)
    np.fill_diagonal(sim, 1.0)
    prot = (rng.random(N) < 0.1).astype(np.uint8)
    x_dev, w_dev = g.dev(x, torch.bfloat16), g.dev(w_r)
    for sere in (False, True):
        kw = dict(sim=g.dev(sim), kp=3, rho=0.45, protect=g.dev(prot)) if sere else {}
        f = _fused(g, x_dev, w_dev, k, ws, **kw)
        s = _separate(g, x_dev, w_dev, k, **kw)
        for name in f:
            _same_bits(f[name], s[name], name)
        _check_oracle(f, k, N, **(dict(sim=sim, kp=3, rho=0.45, protect=prot) if sere else {}))
