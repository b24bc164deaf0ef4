"""GPU parity of the one-call decode layer (moe_decode_layer): as soon as
ranking ends the routing launch publishes the experts the FFN may start on
(the union before the reroute, or SERE's primary union P) and the FFN
streams their phase 1 while routing finishes.  Its routing outputs must
be bit-identical to moe_route_dispatch, its y equal to moe_route_dispatch
followed by moe_ffn_grouped up to the fp32 order of the reductions into y,
and within the stated bar of the oracle; over batch sizes 1 to 64 (16-, 32-
and 64-column token tiles, ragged token columns), with and without SERE,
protection, renormalised gates, accumulation into y, repeated calls on one
pair of workspaces, and steps captured in one CUDA graph."""
import numpy as np
import pytest
import torch

import oracle
import expert_routing_moe_gb300 as moe
from expert_routing_moe_gb300 import _abi as abi
from expert_routing_moe_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu
ROUTE_OUT = ("ids", "gates", "counts", "offsets", "active")


@pytest.fixture(scope="module")
def g():
    import _gpu
    return _gpu


def _layer(D, L, renorm=False, protect=None):
    return moe.MoELayer(D.w_r, D.w_gate, D.w_up, D.w_down, k=L.k, max_tokens=L.T, sim=D.sim,
                        protect=protect, k_primary=L.k_primary, rho=L.rho, renorm=renorm)


def _rows(lay, N):
    M = int(lay.offsets[N].item())
    return lay.row_token[:M].cpu().numpy(), lay.row_gate[:M].cpu().numpy().view(np.uint32)


def _compare(g, L, sere, renorm=False, protect=None, oracle_check=False):
    D = g.DevLayer(L)
    a, b = _layer(D, L, renorm, protect), _layer(D, L, renorm, protect)
    assert a.decode_layer_ok(D.x)
    ya = torch.full((L.T, L.H), float("nan"), dtype=torch.float32, device="cuda:0")
    a.decode_layer(D.x, sere, ya)
    # the separate calls: routing + dispatch, then the fused FFN
    b.route_dispatch(D.x, sere and b.sim is not None)
    b.ffn(D.x)
    torch.cuda.synchronize()
    for lay in (a, b):
        code, detail = lay.device_status()
        assert code == 0, (code, detail)
    T = L.T
    for name in ROUTE_OUT:
        ta, tb = getattr(a, name), getattr(b, name)
        if name in ("ids", "gates"):
            ta, tb = ta[:T], tb[:T]
        va, vb = ta.cpu().numpy(), tb.cpu().numpy()
        if name == "active":   # the count, then that many ids; the rest is not written
            va, vb = va[:1 + va[0]], vb[:1 + vb[0]]
        assert np.array_equal(va.view(np.uint32), vb.view(np.uint32)), name
    ra, rb = _rows(a, L.N), _rows(b, L.N)
    assert np.array_equal(ra[0], rb[0]) and np.array_equal(ra[1], rb[1])
    if sere and a.sim is not None:
        assert np.array_equal(a.stats.cpu().numpy(), b.stats.cpu().numpy())
        assert np.array_equal(a.union_bitmap.cpu().numpy(), b.union_bitmap.cpu().numpy())
    y1, y2 = ya.cpu().numpy(), b.y[:T].cpu().numpy()
    assert np.all(np.isfinite(y1))
    rms = float(np.sqrt(np.mean(y2.astype(np.float64) ** 2)))
    assert float(np.max(np.abs(y1 - y2))) <= 1e-4 * rms
    if oracle_check:
        gl = a.logits[:T].cpu().numpy()
        ref = oracle.layer(L, sere_on=sere and a.sim is not None, logits=gl)
        assert np.array_equal(a.ids[:T].cpu().numpy(), ref["ids"])
        g.assert_y_close(y1, ref["y"], "decode layer")
    return a, ya


@pytest.mark.parametrize("T", [1, 2, 3, 5, 8, 16, 17, 31, 32, 33, 48, 64])
@pytest.mark.parametrize("sere", [False, True])
def test_decode_layer_matches_separate_calls(g, T, sere):
    L = syn.qwen_layer(T, H=256, N=64, k=8, I=256, token_stream_offset=T)
    _compare(g, L, sere, oracle_check=T in (3, 17, 64))


@pytest.mark.parametrize("T,sere", [(40, False), (40, True), (64, True)])
def test_decode_layer_max_experts_and_ranks(g, T, sere):
    """The library's limits in the one-call decode layer: N = 256 experts
    (an eight-word early bitmap; the 256 x 256 similarity is read from
    global memory, past the shared-memory staging limit) and k = 16 (1024
    dispatch rows at 64 tokens), against the separate calls."""
    L = syn.qwen_layer(T, H=256, N=256, k=16, I=128, token_stream_offset=T)
    _compare(g, L, sere)


def test_decode_layer_full_size_against_oracle(g):
    for sere in (False, True):
        L = syn.decode(32)
        a, _ = _compare(g, L, sere, oracle_check=True)


def test_decode_layer_protection_and_renorm(g):
    L = syn.decode(32, n_protect=16)
    D = g.DevLayer(L)
    _compare(g, L, True, protect=D.protect, oracle_check=False)
    _compare(g, L, True, renorm=True)


def test_decode_layer_accumulates_into_y(g):
    L = syn.qwen_layer(24, H=256, N=64, k=8, I=256)
    D = g.DevLayer(L)
    lay = _layer(D, L)
    base = torch.randn(L.T, L.H, device="cuda:0")
    acc = base.clone()
    lay.forward(D.x, sere=True, accumulate_into=acc)
    y = lay.forward(D.x, sere=True).clone()
    torch.cuda.synchronize()
    assert lay.device_status()[0] == 0
    rms = float(y.pow(2).mean().sqrt())
    assert float((acc - base - y).abs().max()) <= 1e-4 * rms + 1e-6


def test_decode_layer_repeated_calls_reuse_workspaces(g):
    """The early flag, the work and per-expert counters and the routing
    tickets return to their starting state after every call: alternating
    batches (and SERE on and off) on one layer give the same results as
    first calls."""
    L = syn.qwen_layer(32, H=256, N=64, k=8, I=256)
    D = g.DevLayer(L)
    lay = _layer(D, L)
    xs = [D.x] + [g.DevLayer(syn.qwen_layer(32, H=256, N=64, k=8, I=256, token_stream_offset=s), weights=False).x
                  for s in (1, 2)]
    first = {}
    for rep in range(3):
        for i, x in enumerate(xs):
            for sere in (False, True):
                y = lay.forward(x, sere=sere).clone()
                torch.cuda.synchronize()
                assert lay.device_status()[0] == 0
                ids = lay.ids[:L.T].cpu().numpy().copy()
                if rep == 0:
                    first[(i, sere)] = (ids, y)
                else:
                    ids0, y0 = first[(i, sere)]
                    assert np.array_equal(ids, ids0)
                    rms = float(y0.pow(2).mean().sqrt())
                    assert float((y - y0).abs().max()) <= 1e-4 * rms
    assert int(lay.ws_route.view(torch.int32)[0].item()) == 0


def test_decode_layer_steps_in_one_graph(g):
    """Eight steps (four batches, SERE and plain alternating, each into its
    own output) captured in one CUDA graph and replayed twice match the same
    steps issued eagerly."""
    L = syn.qwen_layer(32, H=256, N=64, k=8, I=256)
    D = g.DevLayer(L)
    lay = _layer(D, L)
    xs = [g.DevLayer(syn.qwen_layer(32, H=256, N=64, k=8, I=256, token_stream_offset=s), weights=False).x
          for s in range(4)]
    outs = [torch.zeros(L.T, L.H, dtype=torch.float32, device="cuda:0") for _ in range(8)]
    eager = []
    for i in range(8):
        eager.append(lay.forward(xs[i % 4], sere=(i % 2 == 1)).clone())
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        lay.forward(xs[0], sere=False)
    s.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        for i in range(8):
            lay.forward(xs[i % 4], sere=(i % 2 == 1), out=outs[i])
    for _ in range(2):
        for o in outs:
            o.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert lay.device_status()[0] == 0
        for i in range(8):
            rms = float(eager[i].pow(2).mean().sqrt())
            assert float((outs[i] - eager[i]).abs().max()) <= 1e-4 * rms


def test_decode_layer_exercises_the_reroute(g):
    """On the Qwen-shaped batch SERE moves and merges secondaries and the
    active set shrinks, so the early list (primaries) is a strict subset of
    the active experts and the late phase-1 path runs."""
    L = syn.decode(32)
    D = g.DevLayer(L)
    lay = _layer(D, L)
    lay.forward(D.x, sere=True)
    torch.cuda.synchronize()
    st = lay.stats.cpu().numpy()
    assert st[0] > st[2] > st[1]   # union before > union after > |P|
    assert st[3] > 0 and st[4] > 0  # moved and merged slots


EARLY_WORD = 96   # the routing workspace's early flag; the early bitmap follows it


def _bits(words, N):
    return {e for e in range(N) if int(words[e >> 5]) >> (e & 31) & 1}


def test_decode_layer_publishes_the_right_early_set(g):
    """Which experts the routing launch lets the FFN start on, at the Qwen
    shape over batches 1 to 64 and K' = 1, 2: the union before the reroute
    when its phase-1 units fit one wave of the SMs, or two waves while P's
    units would fill at most a third of one and the other experts' more than
    one (an expert that then moves costs only its phase 1), else SERE's
    primary union P, which a reroute never takes an expert from.  Both cases must be reached, P must
    lie inside the final union, and the layer must equal the separate calls
    bit for bit in its routing."""
    Lw = syn.decode(32)
    Dw = g.DevLayer(Lw)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    N, I = Lw.N, Lw.I
    seen = set()
    for T in (1, 3, 5, 8, 12, 16, 24, 32, 48, 64):
        x = g.DevLayer(syn.decode(T, with_weights=False), weights=False).x
        for kp in (1, 2):
            mk = lambda: moe.MoELayer(Dw.w_r, Dw.w_gate, Dw.w_up, Dw.w_down, k=Lw.k, max_tokens=T, sim=Dw.sim,
                                      k_primary=kp, rho=Lw.rho)
            a, b, c = mk(), mk(), mk()
            assert a.decode_layer_ok(x)
            ya = torch.zeros(T, Lw.H, dtype=torch.float32, device="cuda:0")
            a.decode_layer(x, True, ya)
            b.route_dispatch(x, True)
            b.ffn(x)
            c.route_dispatch(x, False)   # plain top-k: the union before the reroute
            torch.cuda.synchronize()
            for lay in (a, b, c):
                assert lay.device_status()[0] == 0
            for name in ROUTE_OUT:
                va, vb = getattr(a, name).cpu().numpy(), getattr(b, name).cpu().numpy()
                if name in ("ids", "gates"):
                    va, vb = va[:T], vb[:T]
                if name == "active":
                    va, vb = va[:1 + va[0]], vb[:1 + vb[0]]
                assert np.array_equal(va.view(np.uint32), vb.view(np.uint32)), (T, kp, name)
            y2 = b.y[:T].cpu().numpy()
            rms = float(np.sqrt(np.mean(y2.astype(np.float64) ** 2)))
            assert float(np.max(np.abs(ya.cpu().numpy() - y2))) <= 1e-4 * rms
            ws = a.ws_route.view(torch.int32).cpu().numpy()
            assert ws[EARLY_WORD] == 1
            early = _bits(ws[EARLY_WORD + 1:EARLY_WORD + 9].view(np.uint32), N)
            before = set(np.flatnonzero(c.counts[:N].cpu().numpy() > 0).tolist())
            after = set(np.flatnonzero(a.counts[:N].cpu().numpy() > 0).tolist())
            P = _bits(a.union_bitmap.cpu().numpy().view(np.uint32), N)
            st = a.stats.cpu().numpy()
            assert len(before) == st[0] and len(P) == st[1] and len(after) == st[2]
            assert P <= after <= before
            wave = sms // (I // 64)   # half-slice phase-1 units: I / 64 per expert
            nu, np_ = len(before), len(P)
            whole = nu <= wave or (3 * np_ <= wave and nu - np_ > wave and nu <= 2 * wave)
            case, want = ("before", before) if whole else ("primary", P)
            assert early == want, (T, kp, case, sorted(early ^ want))
            seen.add(case)
    assert seen == {"before", "primary"}, seen
