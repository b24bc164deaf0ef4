"""GPU parity: the residual stream's fp32 -> bf16 rounding between stacked
layers, bit for bit against PyTorch's CPU round-to-nearest-even."""
import numpy as np
import pytest
import torch

import expert_routing_moe_gb300 as moe

pytestmark = pytest.mark.gpu


def _special_values():
    """Ties (an fp32 exactly halfway between two bf16 values, even and odd
    below), values one ulp off a tie, signed zeros, the smallest subnormals,
    the largest finite values (which round to infinity) and infinities."""
    bits = []
    for hi in (0x3F80, 0x3F81, 0xBF80, 0xBF81, 0x0001, 0x7F7F, 0xFF7F):
        base = hi << 16
        bits += [base | 0x8000, base | 0x7FFF, base | 0x8001, base]
    bits += [0x00000000, 0x80000000, 0x00000001, 0x80000001, 0x7F7FFFFF, 0xFF7FFFFF, 0x7F800000, 0xFF800000]
    return np.array(bits, dtype=np.uint32).view(np.float32)


@pytest.mark.parametrize("n", [8, 64 * 2048, 8 * 1000 + 8])
def test_residual_to_bf16_bit_exact(n):
    rng = np.random.default_rng(n)
    x = (rng.standard_normal(n) * np.exp(rng.uniform(-20, 20, n))).astype(np.float32)
    sp = _special_values()
    x[: min(n, sp.size)] = sp[: min(n, sp.size)]
    xd = torch.from_numpy(x).to("cuda:0")
    y = torch.full((n,), 7, dtype=torch.int16, device="cuda:0").view(torch.bfloat16)
    moe.moe_residual_to_bf16(xd, y)
    torch.cuda.synchronize()
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy()
    got = y.view(torch.int16).cpu().numpy()
    assert np.array_equal(got, ref), np.nonzero(got != ref)[0][:10]


def test_residual_to_bf16_empty_and_rejects():
    x = torch.zeros(16, dtype=torch.float32, device="cuda:0")
    y = torch.zeros(16, dtype=torch.bfloat16, device="cuda:0")
    moe.moe_residual_to_bf16(x[:0], y[:0])           # n = 0: no launch
    with pytest.raises(moe.MoeError):
        moe.moe_residual_to_bf16(x[:12], y[:12])     # n % 8
    with pytest.raises(moe.MoeError):
        moe.moe_residual_to_bf16(x[1:9], y[:8])      # misaligned input
