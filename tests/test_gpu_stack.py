"""GPU parity on the 48-layer decode-stack recipe (batch 64, per-layer router,
similarity and 16 protected experts, SERE K'=2 at rho=0.5, x_{l+1} = x_l +
y_l): three chained layers, each checked against the oracle on the same x_l.
The expert weights are drawn on the device from their seeded generator, as
the stack benchmark does, and copied back for the oracle."""
import numpy as np
import pytest
import torch

import oracle
import expert_routing_moe_gb300 as moe
from expert_routing_moe_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu

N, H, I, K = 128, 2048, 768, 8


def _gap(logits, R):
    s = np.sort(logits, axis=1)[:, ::-1]
    return np.min(s[:, :R] - s[:, 1:R + 1], axis=1)


@pytest.mark.parametrize("sere", [True, False])
def test_stack_layers_chained(sere):
    import _gpu as g
    dev = torch.device(g.DEV)
    B = syn.STACK_BATCH
    x0f, x0b = syn.stack_tokens(B, H)
    xres = torch.from_numpy(x0f).to(dev)
    xb = torch.from_numpy(x0b).view(torch.bfloat16).to(dev)
    toks = np.arange(0, B, 5, dtype=np.int32)   # 13 sampled tokens
    for l in range(3):
        gen = torch.Generator(device=dev)
        gen.manual_seed(syn.stack_weight_seed(l))
        w = [(torch.randn(shape, generator=gen, device=dev) * 0.02).to(torch.bfloat16)
             for shape in ((N, I, H), (N, I, H), (N, H, I))]
        w_r = syn.stack_router(x0f, l)
        sim, prot = syn.stack_sim(l), syn.stack_protect(l)
        lay = moe.MoELayer(g.dev(w_r), *w, k=K, max_tokens=B, sim=g.dev(sim), protect=g.dev(prot), k_primary=2,
                           rho=0.5)
        before = xres.clone()
        lay.route(xb, sere)
        lay.dispatch(B)
        lay.ffn(xb, accumulate_into=xres)
        torch.cuda.synchronize()
        g.assert_status_ok(lay.status)
        y = g.host(xres - before)
        # the oracle on the same layer input
        xin_bits = g.host(xb.view(torch.int16)).view(np.uint16)
        L = syn.Layer(T=B, H=H, N=N, k=K, I=I, dtype="bf16", x=syn.bf16_bits_to_f32(xin_bits), x_bf16=xin_bits,
                      w_r=w_r, w_gate=g.host(w[0].view(torch.int16)).view(np.uint16),
                      w_up=g.host(w[1].view(torch.int16)).view(np.uint16),
                      w_down=g.host(w[2].view(torch.int16)).view(np.uint16), sim=sim, protect=prot, token_w=None,
                      k_primary=2, rho=0.5)
        ref = oracle.layer(L, sere_on=sere, tokens=toks)
        ok = _gap(ref["logits"], K) >= 1e-5
        ids = g.host(lay.out_ids[:B])
        same = np.all(ids == ref["ids"], axis=1)
        assert not np.any(~same & ok), (l, np.nonzero(~same & ok))
        assert int(lay.active[0].item()) == ref["perm"]["active"][0] or not ok.all()
        sel = (ok & same)[toks]
        g.assert_y_close(y[toks][sel], ref["y"][sel], "stack layer %d" % l)
        moe.moe_residual_to_bf16(xres, xb)
