"""GPU parity of the router GEMM (moe_route without FROM_LOGITS, logits out)
against the float64 oracle router, on both kernels that compute it: the
CUDA-core kernels (small batches, or shapes the tensor-core path does not
take) and the tensor-core kernel for large bf16 batches, whose fp32 weight
is split exactly into three bf16 planes."""
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


def _gpu_logits(g, x_dev, w_r, N, k=2):
    T = x_dev.shape[0]
    logits = torch.empty(T, N, dtype=torch.float32, device=g.DEV)
    ids = torch.empty(T, k, dtype=torch.int32, device=g.DEV)
    gates = torch.empty(T, k, dtype=torch.float32, device=g.DEV)
    st = g.status_tensor()
    moe.moe_route(x_dev, g.dev(w_r), logits, ids, gates, k, 0, None, st)
    torch.cuda.synchronize()
    g.assert_status_ok(st)
    return g.host(logits)


@pytest.mark.parametrize("T,H,N,dtype", [
    (32, 2048, 128, "bf16"),     # decode: CUDA cores
    (300, 2048, 128, "bf16"),    # tensor cores, ragged last 128-token tile
    (1000, 512, 64, "bf16"),     # tensor cores, one 64-expert block
    (300, 512, 96, "bf16"),      # N % 64 != 0: tiled CUDA-core kernel
    (300, 256, 64, "f32"),       # fp32 tokens: tiled CUDA-core kernel
    (8192, 2048, 128, "bf16"),   # the prefill batch
])
def test_router_within_fp32_bound(g, T, H, N, dtype):
    rng = np.random.default_rng(T + H + N)
    w = (rng.standard_normal((N, H)) * 0.02).astype(np.float32)
    x = rng.standard_normal((T, H)).astype(np.float32)
    if dtype == "bf16":
        xb = syn.f32_to_bf16_bits(x)
        x = syn.bf16_bits_to_f32(xb)
        x_dev = g.dev(xb, torch.bfloat16)
        ref = oracle.router(xb, w, oracle.DT_BF16)
    else:
        x_dev = g.dev(x)
        ref = oracle.router(x, w, oracle.DT_F32)
    lg = _gpu_logits(g, x_dev, w, N)
    xabs = np.abs(x.astype(np.float64)) @ np.abs(w.astype(np.float64)).T
    assert np.all(np.abs(lg - ref) <= H * 2.0 ** -24 * xabs + 1e-30)


def test_tensor_core_router_split_is_exact(g):
    """x_t = 2^s * e_{h(t)}: every logit is one product s * W[j][h], exact in
    fp32, so the three bf16 planes must reproduce it bit for bit.  W carries
    full 24-bit mantissas over a wide exponent range; a dropped or wrong plane
    changes the low bits."""
    T, H, N = 512, 256, 128
    rng = np.random.default_rng(11)
    mant = rng.integers(1 << 23, 1 << 24, size=(N, H)).astype(np.float64) / float(1 << 23)   # [1, 2)
    expo = rng.integers(-20, 6, size=(N, H))
    sign = np.where(rng.random((N, H)) < 0.5, -1.0, 1.0)
    w = (sign * mant * np.exp2(expo)).astype(np.float32)
    hsel = rng.integers(0, H, size=T)
    scale = np.exp2(rng.integers(-3, 4, size=T)).astype(np.float32)
    x = np.zeros((T, H), dtype=np.float32)
    x[np.arange(T), hsel] = scale
    xb = syn.f32_to_bf16_bits(x)
    lg = _gpu_logits(g, g.dev(xb, torch.bfloat16), w, N)
    expect = (scale[:, None] * w[:, hsel].T).astype(np.float32)
    assert np.array_equal(lg.view(np.uint32), expect.view(np.uint32))
