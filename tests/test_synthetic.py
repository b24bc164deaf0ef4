"""The input recipe: shapes, value ranges and the batch-union regime (CPU only)."""
import numpy as np

from expert_routing_moe_gb300 import synthetic as syn


def test_bf16_rounding_round_trip():
    a = np.array([1.0, -2.5, 3.1415927, 1e-3, 65504.0, 0.0], dtype=np.float32)
    b = syn.bf16_bits_to_f32(syn.f32_to_bf16_bits(a))
    assert np.all(np.abs(b - a) <= np.abs(a) * 2.0 ** -8)
    # ties go to even
    x = np.array([np.float32(1.0) + np.float32(2.0 ** -8)], dtype=np.float32)
    assert syn.bf16_bits_to_f32(syn.f32_to_bf16_bits(x))[0] == 1.0


def test_clustered_similarity_structure():
    s = syn.clustered_sim(np.random.default_rng(0), 128)
    assert np.array_equal(s, s.T) and np.all(np.diag(s) == 1.0)
    off = s[~np.eye(128, dtype=bool)]
    assert ((off > 0.5) == (off >= 0.55)).all()
    assert abs(int((off > 0.5).sum()) - 128 * 7) == 0  # 16 clusters of 8: 7 partners each


def test_decode_batch_union_regime():
    unions = []
    for b in range(6):
        L = syn.decode(32, with_weights=False, token_stream_offset=b)
        l = L.x.astype(np.float64) @ L.w_r.astype(np.float64).T
        top = np.argsort(-l, axis=1)[:, :8]
        unions.append(len(np.unique(top)))
    assert 45 <= np.mean(unions) <= 75


def test_prefill_mix():
    L = syn.prefill(with_weights=False)
    assert L.T == 8192 and int(L.is_visual.sum()) == round(0.7 * 8192)
    assert np.all(L.token_w[~L.is_visual] == 1.0)
    assert 0.0 < L.token_w[L.is_visual].mean() < 0.5
