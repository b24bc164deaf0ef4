"""ctypes binding of the C ABI in include/moe_gb300.h.

Argument marshalling only: each function takes PyTorch CUDA tensors, passes
their device pointers, sizes and the current CUDA stream to the library, and
raises on a non-zero status.  Every step of the layer runs in the library's
CUDA kernels.  If the library has not been built the first call raises; there
is no other implementation to fall back to.
"""
from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_gb300.so")
HEADER_PATH = os.path.join(os.path.dirname(_HERE), "include", "moe_gb300.h")

MOE_OK = 0
MOE_DTYPE_F32, MOE_DTYPE_BF16 = 0, 1
MOE_ROUTE_FROM_LOGITS, MOE_ROUTE_RENORM_TOPK = 1, 2
MOE_FFN_FUSE_COMBINE, MOE_FFN_ZERO_Y = 1, 2
MOE_OP_DISPATCH, MOE_OP_FFN, MOE_OP_CALIBRATE, MOE_OP_TOKEN_WEIGHTS, MOE_OP_ROUTE_DISPATCH = 1, 2, 3, 4, 5
ROUTE_DISPATCH_MAX_T, ROUTE_DISPATCH_MAX_SLOTS = 256, 2048
DECODE_LAYER_MAX_T = 64
MOE_SLOT_KEPT, MOE_SLOT_REROUTED, MOE_SLOT_DROPPED = 0, 1, 2
MOE_DEV_OK, MOE_DEV_NONFINITE, MOE_DEV_TIMEOUT, MOE_DEV_BAD_INDEX = 0, 1, 2, 3

_lock = threading.Lock()
_lib = None


class MoeError(RuntimeError):
    pass


class _SereParams(ctypes.Structure):
    _fields_ = [("k_primary", ctypes.c_int), ("rho", ctypes.c_float), ("sim", ctypes.c_void_p),
                ("protect", ctypes.c_void_p), ("union_bitmap", ctypes.c_void_p), ("stats", ctypes.c_void_p)]


EXPORTS = ["moe_route", "moe_route_dispatch", "moe_decode_layer", "moe_reroute_sere", "moe_dispatch_capacity", "moe_ffn_grouped", "moe_combine",
           "moe_residual_to_bf16", "moe_token_weights", "moe_similarity_calibrate", "moe_workspace_size", "moe_status_string"]


def load(path: str = LIB_PATH):
    """Load the shared library (no GPU needed to load it)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise MoeError("libmoe_gb300.so is not built; run __graft_entry__.build() "
                               "(or python expert_routing_moe_gb300/build.py)")
            L = ctypes.CDLL(path)
            i, u32, f, p, sz = ctypes.c_int, ctypes.c_uint32, ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t
            L.moe_route.argtypes = [p, i, p, i, i, i, i, i, u32, p, p, p, p, p, p]
            L.moe_route.restype = i
            L.moe_route_dispatch.argtypes = [p, i, p, i, i, i, i, u32, p, p, p, p, p, p, p, p, p, p, sz, p, p]
            L.moe_route_dispatch.restype = i
            L.moe_decode_layer.argtypes = [p, p, p, p, p, i, i, i, i, i, u32, u32, p, p, p, p, p, p, p, p, p, p,
                                           p, sz, p, sz, p, p]
            L.moe_decode_layer.restype = i
            L.moe_reroute_sere.argtypes = [p, p, i, i, i, i, p, p, p]
            L.moe_reroute_sere.restype = i
            L.moe_dispatch_capacity.argtypes = [p, p, i, i, i, i, i, p, f, p, p, p, p, p, p, p, p, p, p, p, p, p,
                                                p, sz, p, p]
            L.moe_dispatch_capacity.restype = i
            L.moe_dispatch_capacity_static.argtypes = [p, p, i, i, i, i, i, p, f, p, p, p, p, p, p, p, p, p, p,
                                                       p, p, p, p, p]
            L.moe_dispatch_capacity_static.restype = i
            L.moe_ffn_grouped.argtypes = [p, i, p, p, p, i, i, i, i, i, p, p, p, p, u32, p, p, sz, p, p]
            L.moe_ffn_grouped.restype = i
            L.moe_combine.argtypes = [p, p, p, i, i, i, p, p]
            L.moe_combine.restype = i
            L.moe_residual_to_bf16.argtypes = [p, p, ctypes.c_longlong, p]
            L.moe_residual_to_bf16.restype = i
            L.moe_token_weights.argtypes = [p, i, i, i, p, f, f, p, p, p, p, sz, p, p]
            L.moe_token_weights.restype = i
            L.moe_similarity_calibrate.argtypes = [p, i, p, p, p, i, i, i, p, p, sz, p, p]
            L.moe_similarity_calibrate.restype = i
            L.moe_workspace_size.argtypes = [i, i, i, i, i, i, i, i, i]
            L.moe_workspace_size.restype = sz
            L.moe_status_string.argtypes = [i, i]
            L.moe_status_string.restype = ctypes.c_char_p
            _lib = L
    return _lib


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise MoeError("expected a CUDA tensor")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(rc: int, what: str):
    if rc != MOE_OK:
        msg = load().moe_status_string(rc, 0).decode()
        raise MoeError("%s: %s (%d)" % (what, msg, rc))


def status_string(code: int, device: bool) -> str:
    return load().moe_status_string(int(code), 1 if device else 0).decode()


@dataclass
class SereParams:
    """SERE reroute parameters: K' primaries, threshold rho, similarity [N][N]
    fp32, optional protect [N] uint8, optional outputs union_bitmap
    [ceil(N/32)] int32 and stats [8] int32 (all CUDA tensors)."""
    k_primary: int
    rho: float
    sim: torch.Tensor
    protect: Optional[torch.Tensor] = None
    union_bitmap: Optional[torch.Tensor] = None
    stats: Optional[torch.Tensor] = None

    def _c(self) -> _SereParams:
        return _SereParams(self.k_primary, self.rho, _ptr(self.sim), _ptr(self.protect), _ptr(self.union_bitmap),
                           _ptr(self.stats))


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return MOE_DTYPE_BF16
    if t.dtype == torch.float32:
        return MOE_DTYPE_F32
    raise MoeError("unsupported dtype %s" % t.dtype)


def workspace_size(op: int, T: int, H: int, I: int, N: int, k: int, R: int, capped: bool, dtype: int) -> int:
    return int(load().moe_workspace_size(op, T, H, I, N, k, R, 1 if capped else 0, dtype))


def moe_route(x, w_router, logits, ids, gates, k: int, flags: int = 0, sere: Optional[SereParams] = None,
              st=None, stream=None):
    """Router GEMM (unless MOE_ROUTE_FROM_LOGITS), softmax gate and top-R
    ranking, optionally with the SERE reroute fused in.  ids/gates are [T][R]."""
    T, N = logits.shape
    R = ids.shape[1]
    H = 0 if x is None else x.shape[1]
    xd = MOE_DTYPE_F32 if x is None else _dtype_code(x)
    sp = None if sere is None else ctypes.byref(sere._c())
    rc = load().moe_route(_ptr(x), xd, _ptr(w_router), T, H, N, R, k, flags, _ptr(logits), _ptr(ids), _ptr(gates),
                          sp, _ptr(st), _stream(stream))
    _check(rc, "moe_route")


def moe_route_dispatch(x, w_router, logits, ids, gates, counts, offsets, row_token, row_gate, active, workspace,
                       flags: int = 0, sere: Optional[SereParams] = None, st=None, stream=None):
    """Decode batches (T <= 256): moe_route with R = k (optionally with SERE)
    and the uncapped dispatch in one launch.  ids/gates are [T][k]; workspace
    is workspace_size(MOE_OP_ROUTE_DISPATCH, ...) bytes, zero-filled before
    its first use (each call leaves it zeroed)."""
    T, N = logits.shape
    k = ids.shape[1]
    H = x.shape[1]
    sp = None if sere is None else ctypes.byref(sere._c())
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load().moe_route_dispatch(_ptr(x), _dtype_code(x), _ptr(w_router), T, H, N, k, flags, _ptr(logits),
                                   _ptr(ids), _ptr(gates), sp, _ptr(counts), _ptr(offsets), _ptr(row_token),
                                   _ptr(row_gate), _ptr(active), _ptr(workspace), ws_bytes, _ptr(st),
                                   _stream(stream))
    _check(rc, "moe_route_dispatch")


def moe_decode_layer(x, w_router, w_gate, w_up, w_down, logits, ids, gates, counts, offsets, row_token, row_gate,
                     active, y, route_ws, ffn_ws, route_flags: int = 0, zero_y: bool = True,
                     sere: Optional[SereParams] = None, st=None, stream=None):
    """One decode layer (T <= 64, bf16): routing + dispatch in one launch and
    the FFN with the combine fused in, the FFN starting on the experts known
    to be active as soon as ranking ends.  y [T][H] fp32 is zeroed first when
    zero_y, else accumulated into."""
    T, H = x.shape
    N, I = w_gate.shape[0], w_gate.shape[1]
    k = ids.shape[1]
    sp = None if sere is None else ctypes.byref(sere._c())
    nb = lambda t: t.numel() * t.element_size()
    rc = load().moe_decode_layer(_ptr(x), _ptr(w_router), _ptr(w_gate), _ptr(w_up), _ptr(w_down), T, H, I, N, k,
                                 route_flags, MOE_FFN_ZERO_Y if zero_y else 0, sp, _ptr(logits), _ptr(ids),
                                 _ptr(gates), _ptr(counts), _ptr(offsets), _ptr(row_token), _ptr(row_gate),
                                 _ptr(active), _ptr(y), _ptr(route_ws), nb(route_ws), _ptr(ffn_ws), nb(ffn_ws),
                                 _ptr(st), _stream(stream))
    _check(rc, "moe_decode_layer")


def moe_reroute_sere(ids, gates, N: int, k: int, sere: SereParams, st=None, stream=None):
    T, ld = ids.shape
    rc = load().moe_reroute_sere(_ptr(ids), _ptr(gates), ld, T, N, k, ctypes.byref(sere._c()), _ptr(st),
                                 _stream(stream))
    _check(rc, "moe_reroute_sere")


def moe_dispatch_capacity(ids, gates, N: int, k: int, R: int, counts, offsets, row_token, row_gate, active,
                          workspace, token_w=None, capacity_factor: float = 0.0, out_ids=None, out_gates=None,
                          slot_row=None, slot_status=None, load_q=None, cap_q=None, st=None, stream=None,
                          modality_bias=None, r_v=None):
    T, ld = ids.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load().moe_dispatch_capacity(_ptr(ids), _ptr(gates), ld, T, N, k, R, _ptr(token_w),
                                      float(capacity_factor), _ptr(modality_bias), _ptr(r_v), _ptr(counts),
                                      _ptr(offsets), _ptr(row_token),
                                      _ptr(row_gate), _ptr(active), _ptr(out_ids), _ptr(out_gates),
                                      _ptr(slot_row), _ptr(slot_status), _ptr(load_q), _ptr(cap_q),
                                      _ptr(workspace), ws_bytes, _ptr(st), _stream(stream))
    _check(rc, "moe_dispatch_capacity")


def moe_dispatch_capacity_static(ids, gates, N: int, k: int, R: int, counts, offsets, row_token, row_gate, active,
                                 token_w=None, capacity_factor: float = 0.0, out_ids=None, out_gates=None,
                                 slot_row=None, slot_status=None, load_q=None, cap_q=None, st=None, stream=None,
                                 modality_bias=None, r_v=None):
    """moe_dispatch_capacity without a workspace: the library's own fixed
    device scratch is used (T <= 2048; calls on one device must not overlap)."""
    T, ld = ids.shape
    rc = load().moe_dispatch_capacity_static(_ptr(ids), _ptr(gates), ld, T, N, k, R, _ptr(token_w),
                                             float(capacity_factor), _ptr(modality_bias), _ptr(r_v), _ptr(counts),
                                             _ptr(offsets), _ptr(row_token),
                                             _ptr(row_gate), _ptr(active), _ptr(out_ids), _ptr(out_gates),
                                             _ptr(slot_row), _ptr(slot_status), _ptr(load_q), _ptr(cap_q), _ptr(st),
                                             _stream(stream))
    _check(rc, "moe_dispatch_capacity_static")


def moe_ffn_grouped(x, w_gate, w_up, w_down, k: int, offsets, row_token, row_gate, active, out, workspace,
                    flags: int = MOE_FFN_FUSE_COMBINE | MOE_FFN_ZERO_Y, st=None, stream=None):
    T, H = x.shape
    N, I = w_gate.shape[0], w_gate.shape[1]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load().moe_ffn_grouped(_ptr(x), _dtype_code(x), _ptr(w_gate), _ptr(w_up), _ptr(w_down), T, H, I, N, k,
                                _ptr(offsets), _ptr(row_token), _ptr(row_gate), _ptr(active), flags, _ptr(out),
                                _ptr(workspace), ws_bytes, _ptr(st), _stream(stream))
    _check(rc, "moe_ffn_grouped")


def moe_combine(rows_out, slot_row, slot_gate, y, stream=None):
    T, k = slot_row.shape
    H = y.shape[1]
    rc = load().moe_combine(_ptr(rows_out), _ptr(slot_row), _ptr(slot_gate), T, H, k, _ptr(y), _stream(stream))
    _check(rc, "moe_combine")


def moe_residual_to_bf16(x, y, stream=None):
    """y = bf16(x), round to nearest even: x fp32 and y bf16 CUDA tensors of
    the same number of elements (a multiple of 8)."""
    if x.numel() != y.numel():
        raise MoeError("moe_residual_to_bf16: %d elements in, %d out" % (x.numel(), y.numel()))
    rc = load().moe_residual_to_bf16(_ptr(x), _ptr(y), x.numel(), _stream(stream))
    _check(rc, "moe_residual_to_bf16")


def moe_token_weights(x, is_visual, entropy, token_w, r_v=None, delta: float = 1.0, eps: float = 1e-6, st=None,
                      stream=None, workspace=None):
    """MACS entropy-weighted token load: entropy [T], token_w [T] and R_v [1]
    (fp32 CUDA tensors) from the token features x [T][H] and is_visual [T]
    uint8.  workspace: workspace_size(MOE_OP_TOKEN_WEIGHTS, T, ...) bytes; when
    omitted a buffer is allocated for this call (not graph-capturable)."""
    T, H = x.shape
    if workspace is None:
        workspace = torch.empty(max(workspace_size(MOE_OP_TOKEN_WEIGHTS, T, 1, 1, 1, 1, 1, False, 0), 256),
                                dtype=torch.uint8, device=x.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    rc = load().moe_token_weights(_ptr(x), _dtype_code(x), T, H, _ptr(is_visual), float(delta), float(eps),
                                  _ptr(entropy), _ptr(token_w), _ptr(r_v), _ptr(workspace), ws_bytes, _ptr(st),
                                  _stream(stream))
    _check(rc, "moe_token_weights")


def moe_similarity_calibrate(x, w_gate, w_up, w_down, sim, workspace, st=None, stream=None):
    """SERE similarity matrix [N][N] fp32 from the experts' outputs on the
    calibration tokens x [n][H] bf16 (workspace: workspace_size(MOE_OP_CALIBRATE, n, H, I, N, 1, 1, False,
    MOE_DTYPE_BF16) bytes)."""
    n, H = x.shape
    N, I = w_gate.shape[0], w_gate.shape[1]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load().moe_similarity_calibrate(_ptr(x), n, _ptr(w_gate), _ptr(w_up), _ptr(w_down), H, I, N, _ptr(sim),
                                         _ptr(workspace), ws_bytes, _ptr(st), _stream(stream))
    _check(rc, "moe_similarity_calibrate")
