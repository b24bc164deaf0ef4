"""The allocation-free dispatch entry point.

Some callers cannot allocate device memory -- a plugin inside a serving
engine that owns the whole device memory pool, or code that runs while a
stream is being captured into a CUDA graph under a capture mode that forbids
allocation calls.  For them moe_dispatch_capacity_static does the same work
as moe_dispatch_capacity using scratch memory that the library itself holds.
These tests call it through the C ABI twice in a row and check every output
against the workspace entry point, bit for bit (all outputs are integers or
copied gates).  This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

import oracle
from expert_routing_moe_gb300 import _abi as abi
from expert_routing_moe_gb300 import build as moe_build
from expert_routing_moe_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _outputs(T, N, k, capped):
    i32 = dict(dtype=torch.int32, device=DEV)
    o = dict(counts=torch.full((N,), -9, **i32), offsets=torch.full((N + 1,), -9, **i32),
             active=torch.full((N + 1,), -9, **i32), row_token=torch.full((T * k,), -9, **i32),
             row_gate=torch.full((T * k,), -9.0, dtype=torch.float32, device=DEV),
             out_ids=torch.full((T, k), -9, **i32),
             out_gates=torch.full((T, k), -9.0, dtype=torch.float32, device=DEV),
             slot_row=torch.full((T, k), -9, **i32))
    if capped:
        o.update(slot_status=torch.full((T, k), 99, dtype=torch.uint8, device=DEV),
                 load_q=torch.full((N,), -9, dtype=torch.int64, device=DEV),
                 cap_q=torch.full((1,), -9, dtype=torch.int64, device=DEV))
    return o


def _call(static, ids, gates, N, k, R, token_w, gamma):
    T = ids.shape[0]
    capped = gamma > 0
    o = _outputs(T, N, k, capped)
    st = torch.zeros(2, dtype=torch.int32, device=DEV)
    common = dict(token_w=token_w, capacity_factor=gamma, out_ids=o["out_ids"], out_gates=o["out_gates"],
                  slot_row=o["slot_row"], slot_status=o.get("slot_status"), load_q=o.get("load_q"),
                  cap_q=o.get("cap_q"), st=st)
    if static:
        abi.moe_dispatch_capacity_static(ids, gates, N, k, R, o["counts"], o["offsets"], o["row_token"],
                                         o["row_gate"], o["active"], **common)
    else:
        n = abi.workspace_size(abi.MOE_OP_DISPATCH, T, 1, 1, N, k, R, capped, 0)
        ws = torch.empty(max(n, 256), dtype=torch.uint8, device=DEV)
        abi.moe_dispatch_capacity(ids, gates, N, k, R, o["counts"], o["offsets"], o["row_token"], o["row_gate"],
                                  o["active"], ws, **common)
    torch.cuda.synchronize()
    assert st.tolist() == [0, 0]
    return {name: t.cpu() for name, t in o.items()}


def _same(a, b):
    for name in a:
        x, y = a[name], b[name]
        if x.dtype == torch.float32:
            x, y = x.view(torch.int32), y.view(torch.int32)
        assert torch.equal(x, y), name


def _routing(T, R, stream):
    L = syn.prefill(T=T, with_weights=False, token_stream_offset=stream)
    logits = oracle.router(L.x_bf16, L.w_r, oracle.DT_BF16)
    ids, gates = oracle.route(logits, R)
    return (torch.from_numpy(ids).to(DEV), torch.from_numpy(gates).to(DEV),
            torch.from_numpy(L.token_w).to(DEV), L)


def test_static_scratch_dispatch_matches_workspace_dispatch_twice_in_a_row():
    moe_build.build()
    abi.load()
    # largest supported batch fits the fixed scratch
    assert abi.workspace_size(abi.MOE_OP_DISPATCH, 2048, 1, 1, 256, 16, 16, True, 0) <= 4608 * 1024
    # first call: capacity mode with overflow reroute and drops (prefill-like, 2048 tokens)
    ids, gates, tw, L = _routing(2048, 10, 0)
    ref = _call(False, ids, gates, L.N, L.k, 10, tw, L.gamma)
    got = _call(True, ids, gates, L.N, L.k, 10, tw, L.gamma)
    _same(got, ref)
    assert int((got["slot_status"] == 1).sum()) > 0
    # second call on the same scratch: another batch, uncapped, several permutation blocks
    ids2, gates2, _, _ = _routing(1500, 8, 1)
    ref2 = _call(False, ids2, gates2, L.N, L.k, 8, None, 0.0)
    got2 = _call(True, ids2, gates2, L.N, L.k, 8, None, 0.0)
    _same(got2, ref2)
    # and capacity mode once more, so leftovers of the uncapped call are exercised
    got3 = _call(True, ids, gates, L.N, L.k, 10, tw, L.gamma)
    _same(got3, ref)


def test_static_scratch_dispatch_rejects_batches_beyond_its_limit():
    abi.load()
    T = 2049
    ids = torch.zeros(T, 8, dtype=torch.int32, device=DEV)
    gates = torch.zeros(T, 8, dtype=torch.float32, device=DEV)
    o = _outputs(T, 128, 8, False)
    with pytest.raises(abi.MoeError, match="unsupported"):
        abi.moe_dispatch_capacity_static(ids, gates, 128, 8, 8, o["counts"], o["offsets"], o["row_token"],
                                         o["row_gate"], o["active"])
