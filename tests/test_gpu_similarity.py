"""GPU parity of the expert-similarity calibration (moe_similarity_calibrate,
SERE article sec. 4.2) against the oracle.

Tolerance: the GPU path rounds the SwiGLU activations to bf16 inside the
FFN and the expert outputs to bf16 before the Gram matrix, each a relative
error of at most 2^-8 per element, so ||dE|| / ||E|| <= 2^-7 and the cosine
of two such vectors moves by at most 2 * 2 * 2^-7."""
import numpy as np
import pytest
import torch

import oracle
import expert_routing_moe_gb300 as moe
from expert_routing_moe_gb300 import _abi as abi
from expert_routing_moe_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu
TOL = 4 * 2.0 ** -7


@pytest.fixture(scope="module")
def g():
    import _gpu
    return _gpu


def _gpu_sim(g, x_bits, wg, wu, wd):
    x = g.dev(x_bits, torch.bfloat16)
    Wg, Wu, Wd = (g.dev(a, torch.bfloat16) for a in (wg, wu, wd))
    n, H = x.shape
    N, I = wg.shape[0], wg.shape[1]
    ws = torch.empty(abi.workspace_size(abi.MOE_OP_CALIBRATE, n, H, I, N, 1, 1, False, abi.MOE_DTYPE_BF16),
                     dtype=torch.uint8, device=g.DEV)
    sim = torch.full((N, N), float("nan"), dtype=torch.float32, device=g.DEV)
    st = g.status_tensor()
    moe.moe_similarity_calibrate(x, Wg, Wu, Wd, sim, ws, st)
    torch.cuda.synchronize()
    g.assert_status_ok(st)
    return g.host(sim)


def _bf16_experts(rng, N, H, I):
    f = syn.f32_to_bf16_bits
    return (f(rng.standard_normal((N, I, H)).astype(np.float32) / np.sqrt(H)),
            f(rng.standard_normal((N, I, H)).astype(np.float32) / np.sqrt(H)),
            f(rng.standard_normal((N, H, I)).astype(np.float32) / np.sqrt(I)))


def test_similarity_small_matches_oracle(g):
    rng = np.random.default_rng(0)
    N, H, I, n = 8, 256, 128, 16
    wg, wu, wd = _bf16_experts(rng, N, H, I)
    # a cluster: expert 1 shares expert 0's gate/up and a perturbed down projection
    wg[1], wu[1] = wg[0], wu[0]
    wd[1] = syn.f32_to_bf16_bits(syn.bf16_bits_to_f32(wd[0]) + 0.3 * syn.bf16_bits_to_f32(wd[1]))
    x = syn.f32_to_bf16_bits(rng.standard_normal((n, H)).astype(np.float32))
    s = _gpu_sim(g, x, wg, wu, wd)
    ref = oracle.similarity(x, wg, wu, wd, oracle.DT_BF16, oracle.DT_BF16)
    assert np.all(np.abs(s - ref) <= TOL), float(np.max(np.abs(s - ref)))
    assert np.array_equal(s, s.T) and np.all(np.diag(s) == 1.0)
    assert ref[0, 1] > 0.8 and s[0, 1] > 0.8


def test_similarity_constructed_pairs_on_gpu(g):
    rng = np.random.default_rng(1)
    N, H, I, n = 6, 256, 128, 8
    wg, wu, wd = _bf16_experts(rng, N, H, I)
    wg[1], wu[1], wd[1] = wg[0], wu[0], wd[0]                       # duplicate -> 1
    wg[2], wu[2], wd[2] = wg[0], wu[0], wd[0] ^ np.uint16(0x8000)   # negated down projection -> -1
    wd[3, 128:] = 0                                                 # disjoint output coordinates -> 0
    wd[4, :128] = 0
    x = syn.f32_to_bf16_bits(rng.standard_normal((n, H)).astype(np.float32))
    s = _gpu_sim(g, x, wg, wu, wd)
    assert abs(s[0, 1] - 1.0) < 1e-5 and abs(s[0, 2] + 1.0) < 1e-5
    assert s[3, 4] == 0.0


def test_similarity_full_shape_every_pair(g):
    """The Qwen3-30B-A3B-shaped experts (128 x 2048 x 768) on 64 calibration
    tokens, every one of the 8128 pairs against the oracle.  Sixteen experts
    are made partners of another one (shared gate and up rows, a down
    projection mixed with noise at 16 strengths), so that the true cosines
    also cover the range around rho = 0.5 where SERE decides.

    What the tolerance means for those decisions: the GPU's cosine is within
    4 * 2^-7 of the oracle's, so `sim > rho` can differ from the oracle's only
    for a pair whose exact cosine lies within that distance of rho; every
    other pair is checked to decide alike."""
    L = syn.decode(32)
    wg, wu, wd = (np.array(w) for w in (L.w_gate, L.w_up, L.w_down))
    rng = np.random.default_rng(3)
    for j in range(16):
        a, b = 2 * j, 2 * j + 1
        wg[b], wu[b] = wg[a], wu[a]
        c = 0.2 * j
        wd[b] = syn.f32_to_bf16_bits(syn.bf16_bits_to_f32(wd[a]) +
                                     c * rng.standard_normal(wd[a].shape).astype(np.float32) * 0.02)
    x = syn.f32_to_bf16_bits(rng.standard_normal((64, L.H)).astype(np.float32))
    s = _gpu_sim(g, x, wg, wu, wd)
    assert np.array_equal(s, s.T) and np.all(np.diag(s) == 1.0)
    assert np.all(np.abs(s) <= 1.0 + 1e-6) and np.all(np.isfinite(s))
    oracle.set_threads(0)
    ref = oracle.similarity(x, wg, wu, wd, oracle.DT_BF16, oracle.DT_BF16)
    iu = np.triu_indices(L.N, 1)
    err = np.abs(s[iu] - ref[iu])
    assert err.max() <= TOL, (float(err.max()), np.unravel_index(np.argmax(np.abs(s - ref) - np.eye(L.N)), s.shape))
    rho = 0.5
    far = np.abs(ref[iu] - rho) > TOL
    assert np.array_equal(s[iu][far] > rho, ref[iu][far] > rho)
    # the constructed partners span both sides of rho
    pair = np.array([ref[2 * j, 2 * j + 1] for j in range(16)])
    assert (pair > rho + TOL).sum() >= 3 and (pair < rho - TOL).sum() >= 3, pair
