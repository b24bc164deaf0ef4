"""GPU parity of the whole layer from token activations (router GEMM on the
GPU included) against the oracle, on every workload, plus the end-to-end
properties (SERE shrinks the union, capacity is respected)."""
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


def _gap(logits, R):
    s = np.sort(logits, axis=1)[:, ::-1]
    R = min(R, logits.shape[1] - 1)
    return np.min(s[:, :R] - s[:, 1:R + 1], axis=1)


def _layer(g, L, D, capped=False):
    return moe.MoELayer(D.w_r, D.w_gate, D.w_up, D.w_down, k=L.k, max_tokens=L.T, sim=D.sim, protect=D.protect,
                        k_primary=L.k_primary, rho=L.rho, R=L.R if capped else L.k,
                        capacity_factor=L.gamma if capped else 0.0)


def _router_bound_ok(L, gl, ref_logits):
    """The GPU router's fp32 logits agree with the oracle's double-accumulated
    ones within the fp32 dot-product bound H * 2^-24 * sum_h |x_h W_jh|."""
    xabs = np.abs(L.x.astype(np.float64)) @ np.abs(L.w_r.astype(np.float64)).T
    assert np.all(np.abs(gl - ref_logits) <= L.H * 2.0 ** -24 * xabs + 1e-30)


def _run(g, L, sere, capped=False, tokens=None):
    D = g.DevLayer(L)
    layer = _layer(g, L, D, capped)
    y = layer.forward(D.x, sere=sere, token_w=D.token_w if capped else None)
    torch.cuda.synchronize()
    code, detail = layer.device_status()
    assert code == 0, (code, detail)
    ref = oracle.layer(L, sere_on=sere, capacity_on=capped, tokens=tokens)
    gl = g.host(layer.logits[:L.T])
    _router_bound_ok(L, gl, ref["logits"])
    # a token may route differently only where the fp32 router's rounding can
    # reorder its ranking: adjacent logits closer than 1e-5 (the stated exclusion)
    ok = _gap(ref["logits"], (L.R if capped else L.k)) >= 1e-5
    ids = g.host((layer.out_ids if capped else layer.ids)[:L.T])
    same = np.all(ids == ref["ids"], axis=1)
    assert np.all(same[ok]), np.nonzero(~same & ok)
    yt = g.host(y) if tokens is None else g.host(y)[tokens]
    okt = ok if tokens is None else ok[tokens]
    g.assert_y_close(yt[okt], ref["y"][okt], "layer")
    return layer, ref


def test_tiny_layer_plain_and_sere(g):
    L = syn.tiny()
    _run(g, L, sere=False)
    layer, ref = _run(g, L, sere=True)
    assert np.array_equal(g.host(layer.stats), ref["stats"])


def test_tiny_layer_capacity(g):
    L = syn.tiny(capacity=True)
    layer, ref = _run(g, L, sere=False, capped=True)
    assert int(layer.cap_q.item()) == ref["cap"]


def test_decode_layer_top8_vs_sere(g):
    L = syn.decode(32)
    l0, r0 = _run(g, L, sere=False)
    l1, r1 = _run(g, L, sere=True)
    # SERE activates fewer experts than plain top-8 on this workload
    assert int(l1.active[0].item()) < int(l0.active[0].item())
    assert int(l1.active[0].item()) == r1["perm"]["active"][0]


def test_prefill_capacity_layer_full(g):
    """The capacity prefill layer at full size (8192 tokens, R = 10, gamma =
    1.25), every token checked.  Capacity couples tokens: one token's near-tie
    can change which other tokens an expert admits, so the routing is checked
    in two parts that need no exclusion at all.  (a) The GPU router's fp32
    logits are within the fp32 dot-product bound of the oracle's.  (b) Given
    the GPU's own logits, the oracle's ranking, admission, overflow rounds and
    permutation equal the GPU's bit for bit, and every token's y is within
    2e-2 * rms(y) of the oracle's."""
    L = syn.prefill()
    D = g.DevLayer(L)
    layer = _layer(g, L, D, capped=True)
    y = layer.forward(D.x, token_w=D.token_w)
    torch.cuda.synchronize()
    code, detail = layer.device_status()
    assert code == 0, (code, detail)
    gl = g.host(layer.logits[:L.T])
    _router_bound_ok(L, gl, oracle.router(L.x_bf16, L.w_r, oracle.DT_BF16))
    ref = oracle.layer(L, sere_on=False, capacity_on=True, logits=np.ascontiguousarray(gl))
    assert np.array_equal(g.host(layer.out_ids[:L.T]), ref["ids"])
    assert np.array_equal(g.host(layer.out_gates[:L.T]).view(np.uint32), ref["gates"].view(np.uint32))
    assert np.array_equal(g.host(layer.slot_status[:L.T]), ref["status"])
    assert np.array_equal(g.host(layer.load_q), ref["load"])
    assert int(layer.cap_q.item()) == ref["cap"]
    p = ref["perm"]
    m = int(p["offsets"][L.N])
    assert np.array_equal(g.host(layer.offsets), p["offsets"])
    assert np.array_equal(g.host(layer.row_token[:m]), p["row_token"])
    assert (g.host(layer.load_q) <= ref["cap"]).all()
    assert (ref["status"] == oracle.SLOT_REROUTED).sum() > 0 and (ref["status"] == oracle.SLOT_DROPPED).sum() > 0
    g.assert_y_close(g.host(y), ref["y"], "prefill layer, all tokens")


def test_decode_steps_replayed_from_one_graph(g):
    """The bench's launch configuration: several SERE decode steps (routing
    and dispatch in one launch, then the FFN, chained by programmatic
    dependent launch) captured in one CUDA graph, each on its own batch and
    into its own output, then replayed three times.  Every step's output
    matches the oracle layer, so the kernels' counters and workspaces are
    left ready for the next step inside the graph."""
    import dataclasses
    L = syn.decode(32)
    D = g.DevLayer(L)
    layer = _layer(g, L, D)
    nb = 4
    Ls = [L] + [dataclasses.replace(L, x=Lb.x, x_bf16=Lb.x_bf16) for Lb in
                (syn.decode(32, with_weights=False, token_stream_offset=b) for b in range(1, nb))]
    xs = [g.dev(Lb.x_bf16, torch.bfloat16) for Lb in Ls]
    ys = [torch.empty(L.T, L.H, dtype=torch.float32, device=g.DEV) for _ in range(nb)]
    stream = torch.cuda.Stream(device=g.DEV)
    with torch.cuda.stream(stream):
        for b in range(nb):
            layer.forward(xs[b], sere=True, out=ys[b])
        stream.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for rep in range(2):
                for b in range(nb):
                    layer.forward(xs[b], sere=True, out=ys[b])
        for y in ys:
            y.fill_(float("nan"))
        for _ in range(3):
            graph.replay()
        stream.synchronize()
    code, detail = layer.device_status()
    assert code == 0, (code, detail)
    for b, Lb in enumerate(Ls):
        ref = oracle.layer(Lb, sere_on=True)
        ok = _gap(ref["logits"], L.k) >= 1e-5
        g.assert_y_close(g.host(ys[b])[ok], ref["y"][ok], "graph step %d" % b)
