"""Helpers for the GPU parity tests: device copies of synthetic layers and the
GPU path's stages called through the C ABI."""
from __future__ import annotations

import numpy as np
import torch

import expert_routing_moe_gb300 as moe
from expert_routing_moe_gb300 import _abi as abi

DEV = "cuda:0"


def dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.to(DEV)


def host(t):
    return t.detach().cpu().numpy()


class DevLayer:
    """Device copies of a synthetic Layer's arrays."""

    def __init__(self, L, weights=True):
        self.L = L
        bf = L.dtype == "bf16"
        self.x = dev(L.x_bf16, torch.bfloat16) if bf else dev(L.x)
        self.w_r = dev(L.w_r)
        if weights and L.w_gate is not None:
            wdt = torch.bfloat16 if bf else None
            self.w_gate, self.w_up, self.w_down = dev(L.w_gate, wdt), dev(L.w_up, wdt), dev(L.w_down, wdt)
        self.sim = dev(L.sim)
        self.protect = None if L.protect is None else dev(L.protect)
        self.token_w = None if L.token_w is None else dev(L.token_w)


def status_tensor():
    return torch.zeros(2, dtype=torch.int32, device=DEV)


def assert_status_ok(st):
    code, detail = (int(v) for v in st.tolist())
    assert code == 0, "device status %d (%s), detail %d" % (code, abi.status_string(code, True), detail)


def gpu_route(logits_np, R, k, renorm=False, sere=None, N=None):
    """Rank (and optionally SERE-reroute) given fp32 logits on the GPU."""
    T, N = logits_np.shape
    lg = dev(logits_np.astype(np.float32))
    ids = torch.empty(T, R, dtype=torch.int32, device=DEV)
    gates = torch.empty(T, R, dtype=torch.float32, device=DEV)
    st = status_tensor()
    flags = abi.MOE_ROUTE_FROM_LOGITS | (abi.MOE_ROUTE_RENORM_TOPK if renorm else 0)
    moe.moe_route(None, None, lg, ids, gates, k, flags, sere, st)
    torch.cuda.synchronize()
    return ids, gates, st


def sere_params(sim, kp, rho, protect=None, N=None):
    N = sim.shape[0]
    return abi.SereParams(kp, rho, sim if torch.is_tensor(sim) else dev(sim),
                          None if protect is None else (protect if torch.is_tensor(protect) else dev(protect)),
                          torch.zeros((N + 31) // 32, dtype=torch.int32, device=DEV),
                          torch.zeros(8, dtype=torch.int32, device=DEV))


def gpu_dispatch(ids, gates, N, k, R, token_w=None, gamma=0.0):
    """ids/gates: CUDA tensors [T][ld].  Returns a dict of host arrays."""
    T = ids.shape[0]
    capped = gamma > 0
    ws_n = abi.workspace_size(abi.MOE_OP_DISPATCH, T, 1, 1, N, k, R, capped, 0)
    ws = torch.empty(max(ws_n, 256), dtype=torch.uint8, device=DEV)
    i32 = dict(dtype=torch.int32, device=DEV)
    counts = torch.full((N,), -7, **i32)
    offsets = torch.full((N + 1,), -7, **i32)
    active = torch.full((N + 1,), -7, **i32)
    row_token = torch.full((max(T * k, 1),), -7, **i32)
    row_gate = torch.full((max(T * k, 1),), -7.0, dtype=torch.float32, device=DEV)
    out_ids = torch.full((T, k), -7, **i32)
    out_gates = torch.full((T, k), -7.0, dtype=torch.float32, device=DEV)
    slot_row = torch.full((T, k), -7, **i32)
    status = torch.full((T, k), 77, dtype=torch.uint8, device=DEV) if capped else None
    load_q = torch.zeros(N, dtype=torch.int64, device=DEV) if capped else None
    cap_q = torch.zeros(1, dtype=torch.int64, device=DEV) if capped else None
    tw = None if token_w is None else (token_w if torch.is_tensor(token_w) else dev(np.asarray(token_w, np.float32)))
    st = status_tensor()
    moe.moe_dispatch_capacity(ids, gates, N, k, R, counts, offsets, row_token, row_gate, active, ws, tw, gamma,
                              out_ids, out_gates, slot_row, status, load_q, cap_q, st)
    torch.cuda.synchronize()
    assert_status_ok(st)
    M = int(offsets[N].item())
    out = dict(counts=host(counts), offsets=host(offsets), active=host(active), row_token=host(row_token)[:M],
               row_gate=host(row_gate)[:M], out_ids=host(out_ids), out_gates=host(out_gates),
               slot_row=host(slot_row), dev=dict(offsets=offsets, row_token=row_token, row_gate=row_gate,
                                                 active=active, slot_row=slot_row, out_gates=out_gates))
    if capped:
        out.update(status=host(status), load=host(load_q), cap=int(cap_q.item()))
    return out


def ffn_workspace(x, w_gate, k, T):
    H = x.shape[1]
    N, I = w_gate.shape[0], w_gate.shape[1]
    dt = abi.MOE_DTYPE_BF16 if x.dtype == torch.bfloat16 else abi.MOE_DTYPE_F32
    ws_n = abi.workspace_size(abi.MOE_OP_FFN, T, H, I, N, k, k, False, dt)
    return torch.zeros(max(ws_n, 256), dtype=torch.uint8, device=DEV)   # zero before the first call


def gpu_ffn(x, w_gate, w_up, w_down, k, disp_dev, T, fuse=True, ws=None):
    H = x.shape[1]
    if ws is None:
        ws = ffn_workspace(x, w_gate, k, T)
    st = status_tensor()
    if fuse:
        y = torch.full((T, H), float("nan"), dtype=torch.float32, device=DEV)
        moe.moe_ffn_grouped(x, w_gate, w_up, w_down, k, disp_dev["offsets"], disp_dev["row_token"],
                            disp_dev["row_gate"], disp_dev["active"], y, ws,
                            abi.MOE_FFN_FUSE_COMBINE | abi.MOE_FFN_ZERO_Y, st)
    else:
        rows = torch.zeros(max(T * k, 1), H, dtype=torch.float32, device=DEV)
        moe.moe_ffn_grouped(x, w_gate, w_up, w_down, k, disp_dev["offsets"], disp_dev["row_token"],
                            disp_dev["row_gate"], disp_dev["active"], rows, ws, 0, st)
        y = torch.full((T, H), float("nan"), dtype=torch.float32, device=DEV)
        moe.moe_combine(rows, disp_dev["slot_row"], disp_dev["out_gates"], y)
    torch.cuda.synchronize()
    assert_status_ok(st)
    return host(y)


def assert_y_close(y, yref, what=""):
    """The layer-output bar: max |y - y_ref| <= 2e-2 * rms(y_ref)."""
    rms = float(np.sqrt(np.mean(yref ** 2)))
    err = float(np.max(np.abs(y - yref))) if y.size else 0.0
    assert np.all(np.isfinite(y)), what + ": non-finite output"
    assert err <= 2e-2 * rms, "%s: max|dy| %.3e > 2e-2 * rms %.3e" % (what, err, rms)
    return err, rms
