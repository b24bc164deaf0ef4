"""Pins for the oracle's permutation, expert FFN and combine (CPU only)."""
import numpy as np

import oracle
from expert_routing_moe_gb300 import synthetic as syn


def _dense_expert_outputs(x, wg, wu, wd):
    """E_j(x) for every token and every expert, float64, by whole-matrix products."""
    x = x.astype(np.float64)
    g = np.einsum("th,nih->nti", x, wg.astype(np.float64))
    u = np.einsum("th,nih->nti", x, wu.astype(np.float64))
    a = g / (1.0 + np.exp(-g)) * u
    return np.einsum("nti,nhi->nth", a, wd.astype(np.float64))  # [N][T][H]


def test_permute_is_lexsort_by_expert_then_token():
    rng = np.random.default_rng(0)
    for _ in range(50):
        T, N = int(rng.integers(0, 30)), int(rng.integers(1, 20))
        k = int(rng.integers(1, min(N, 5) + 1))
        ids = np.stack([rng.permutation(N)[:k] for _ in range(T)]).astype(np.int32) if T else np.zeros((0, k), np.int32)
        ids[rng.random(ids.shape) < 0.2] = -1
        gates = rng.random(ids.shape).astype(np.float32)
        p = oracle.permute(ids, gates, N, k)
        tt, rr = np.nonzero(ids >= 0)
        ee = ids[tt, rr]
        order = np.lexsort((tt, ee))
        assert p["row_token"].tolist() == tt[order].tolist()
        assert np.array_equal(p["row_gate"], gates[tt, rr][order])
        cnt = np.bincount(ee, minlength=N)
        assert p["counts"].tolist() == cnt.tolist()
        assert p["offsets"].tolist() == [0] + np.cumsum(cnt).tolist()
        act = np.nonzero(cnt)[0]
        assert p["active"][0] == len(act) and p["active"][1:1 + len(act)].tolist() == act.tolist()


def test_ffn_combine_matches_dense_eq1_fp32_weights():
    L = syn.tiny()
    logits = oracle.router(L.x, L.w_r)
    ids, gates = oracle.route(logits, L.k)
    y = oracle.ffn_combine(L.x, L.w_gate, L.w_up, L.w_down, ids, gates, L.k)
    E = _dense_expert_outputs(L.x, L.w_gate, L.w_up, L.w_down)
    ref = np.zeros_like(y)
    for t in range(L.T):
        for r in range(L.k):
            ref[t] += float(gates[t, r]) * E[ids[t, r], t]
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12)
    # a token subset gives the same rows
    sub = np.array([3, 0, 15], dtype=np.int32)
    ys = oracle.ffn_combine(L.x, L.w_gate, L.w_up, L.w_down, ids, gates, L.k, tokens=sub)
    assert np.array_equal(ys, y[sub])


def test_ffn_combine_bf16_decodes_bits_exactly():
    L = syn.qwen_layer(6, H=128, N=4, k=2, I=64)
    wg = syn.bf16_bits_to_f32(L.w_gate)
    wu = syn.bf16_bits_to_f32(L.w_up)
    wd = syn.bf16_bits_to_f32(L.w_down)
    ids = np.array([[0, 1], [2, 3], [1, -1], [3, 0], [-1, -1], [2, 1]], dtype=np.int32)
    gates = np.array([[0.6, 0.4], [0.5, 0.5], [1.0, 0.0], [0.7, 0.2], [0, 0], [0.1, 0.9]], dtype=np.float32)
    y = oracle.ffn_combine(L.x_bf16, L.w_gate, L.w_up, L.w_down, ids, gates, 2,
                           x_dtype=oracle.DT_BF16, w_dtype=oracle.DT_BF16)
    E = _dense_expert_outputs(L.x, wg, wu, wd)
    ref = np.zeros_like(y)
    for t in range(6):
        for r in range(2):
            if ids[t, r] >= 0:
                ref[t] += float(gates[t, r]) * E[ids[t, r], t]
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12)
    assert np.all(y[4] == 0.0)


def test_whole_tiny_layer_is_eq1():
    """y(x) = sum over the top-k of softmax(G(x))_j E_j(x), all from numpy."""
    L = syn.tiny()
    out = oracle.layer(L, sere_on=False)
    l64 = L.x.astype(np.float64) @ L.w_r.astype(np.float64).T
    p = np.exp(l64 - l64.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    top = np.argsort(-l64, axis=1, kind="stable")[:, :L.k]
    E = _dense_expert_outputs(L.x, L.w_gate, L.w_up, L.w_down)
    ref = np.zeros((L.T, L.H))
    for t in range(L.T):
        for j in top[t]:
            ref[t] += p[t, j] * E[j, t]
    assert np.array_equal(out["ids"], top.astype(np.int32))
    assert np.max(np.abs(out["y"] - ref)) <= 1e-5 * np.sqrt(np.mean(ref ** 2))


def test_thread_count_does_not_change_results():
    """The oracle's OpenMP loops (router, FFN + combine, similarity) give the
    same bits with one thread and with every host core."""
    L = syn.qwen_layer(24, H=128, N=8, k=3, I=64)
    xb = L.x_bf16
    try:
        outs = []
        for nt in (1, 0):
            oracle.set_threads(nt)
            logits = oracle.router(xb, L.w_r, oracle.DT_BF16)
            ids, gates = oracle.route(logits, L.k)
            y = oracle.ffn_combine(xb, L.w_gate, L.w_up, L.w_down, ids, gates, L.k, x_dtype=oracle.DT_BF16,
                                   w_dtype=oracle.DT_BF16)
            sim = oracle.similarity(xb[:5], L.w_gate, L.w_up, L.w_down, x_dtype=oracle.DT_BF16,
                                    w_dtype=oracle.DT_BF16)
            outs.append((logits, y, sim))
        for a, b in zip(*outs):
            assert np.array_equal(a, b)
    finally:
        oracle.set_threads(0)
