"""A resident MoE layer: device weights, preallocated buffers and the C-ABI
calls of one forward pass in order (router + rank (+ SERE) -> dispatch
(+ capacity) -> grouped FFN with the combine fused in).  Uncapped bf16
batches of up to 64 tokens take the one-call decode layer (moe_decode_layer:
the FFN starts on the experts known to be active while routing finishes);
other uncapped batches of up to 256 tokens the single-launch routing +
dispatch entry point.
Buffers are sized once for a maximum batch, so a forward pass allocates
nothing and can be captured in a CUDA graph."""
from __future__ import annotations

from typing import Optional

import torch

from . import _abi as abi


class MoELayer:
    def __init__(self, w_router: torch.Tensor, w_gate: torch.Tensor, w_up: torch.Tensor, w_down: torch.Tensor,
                 k: int, max_tokens: int, sim: Optional[torch.Tensor] = None, protect: Optional[torch.Tensor] = None,
                 k_primary: int = 2, rho: float = 0.5, R: Optional[int] = None, capacity_factor: float = 0.0,
                 renorm: bool = False, modality_bias: Optional[torch.Tensor] = None,
                 r_v: Optional[torch.Tensor] = None):
        dev = w_gate.device
        self.w_router, self.w_gate, self.w_up, self.w_down = w_router, w_gate, w_up, w_down
        self.N, self.I, self.H = w_gate.shape
        self.k = k
        self.R = R if R is not None else k
        self.max_T = max_tokens
        self.sim, self.protect = sim, protect
        self.k_primary, self.rho = k_primary, rho
        self.capacity_factor = capacity_factor
        # per-expert capacity: m_j in {+1, -1, 0} [N] int8 and the batch's visual ratio [1] fp32
        self.modality_bias, self.r_v = modality_bias, r_v
        self.flags = abi.MOE_ROUTE_RENORM_TOPK if renorm else 0
        T, N, R, H = max_tokens, self.N, self.R, self.H
        i32, f32 = torch.int32, torch.float32
        self.logits = torch.empty(T, N, dtype=f32, device=dev)
        self.ids = torch.empty(T, R, dtype=i32, device=dev)
        self.gates = torch.empty(T, R, dtype=f32, device=dev)
        self.counts = torch.empty(N, dtype=i32, device=dev)
        self.offsets = torch.empty(N + 1, dtype=i32, device=dev)
        self.active = torch.empty(N + 1, dtype=i32, device=dev)
        self.row_token = torch.empty(max(T * k, 1), dtype=i32, device=dev)
        self.row_gate = torch.empty(max(T * k, 1), dtype=f32, device=dev)
        self.out_ids = torch.empty(T, k, dtype=i32, device=dev)
        self.out_gates = torch.empty(T, k, dtype=f32, device=dev)
        self.slot_status = torch.empty(T, k, dtype=torch.uint8, device=dev)
        self.load_q = torch.empty(N, dtype=torch.int64, device=dev)
        self.cap_q = torch.empty(1, dtype=torch.int64, device=dev)
        self.union_bitmap = torch.empty((N + 31) // 32, dtype=i32, device=dev)
        self.stats = torch.zeros(8, dtype=i32, device=dev)
        self.status = torch.zeros(2, dtype=i32, device=dev)
        dt = abi.MOE_DTYPE_BF16 if w_gate.dtype == torch.bfloat16 else abi.MOE_DTYPE_F32
        capped = capacity_factor > 0
        wsd = abi.workspace_size(abi.MOE_OP_DISPATCH, T, H, self.I, N, k, self.R, capped, dt)
        wsf = abi.workspace_size(abi.MOE_OP_FFN, T, H, self.I, N, k, self.R, capped, dt)
        self.ws_dispatch = torch.empty(max(wsd, 256), dtype=torch.uint8, device=dev)
        # the FFN keeps counters at the start of its workspace: zero before the first call
        self.ws_ffn = torch.zeros(max(wsf, 256), dtype=torch.uint8, device=dev)
        # the single-launch routing + dispatch keeps a counter here (zero between calls)
        wsr = abi.workspace_size(abi.MOE_OP_ROUTE_DISPATCH, T, H, self.I, N, k, self.R, False, dt)
        self.ws_route = torch.zeros(max(wsr, 256), dtype=torch.uint8, device=dev)
        self.y = torch.empty(T, H, dtype=f32, device=dev)

    def sere_params(self) -> abi.SereParams:
        return abi.SereParams(self.k_primary, self.rho, self.sim, self.protect, self.union_bitmap, self.stats)

    def route(self, x: torch.Tensor, sere: bool, stream=None):
        T = x.shape[0]
        sp = self.sere_params() if sere else None
        abi.moe_route(x, self.w_router, self.logits[:T], self.ids[:T], self.gates[:T], self.k, self.flags, sp,
                      self.status, stream)

    def fused_route_dispatch_ok(self, T: int) -> bool:
        return (self.capacity_factor <= 0 and self.R == self.k and T <= abi.ROUTE_DISPATCH_MAX_T
                and T * self.k <= abi.ROUTE_DISPATCH_MAX_SLOTS)

    def route_dispatch(self, x: torch.Tensor, sere: bool, stream=None):
        """Routing and the uncapped dispatch in one launch (decode batches)."""
        T = x.shape[0]
        sp = self.sere_params() if sere else None
        abi.moe_route_dispatch(x, self.w_router, self.logits[:T], self.ids[:T], self.gates[:T], self.counts,
                               self.offsets, self.row_token, self.row_gate, self.active, self.ws_route, self.flags,
                               sp, self.status, stream)

    def decode_layer_ok(self, x: torch.Tensor) -> bool:
        """Whether moe_decode_layer can run this batch: uncapped top-k,
        bf16 activations and weights, 1 <= T <= 64."""
        T = x.shape[0]
        return (self.fused_route_dispatch_ok(T) and 1 <= T <= abi.DECODE_LAYER_MAX_T
                and x.dtype == torch.bfloat16 and self.w_gate.dtype == torch.bfloat16
                and self.H % 128 == 0 and self.I % 128 == 0)

    def decode_layer(self, x: torch.Tensor, sere: bool, y: torch.Tensor, zero_y: bool = True, stream=None):
        """Routing, dispatch and the FFN of one decode batch in one call;
        y [T][H] fp32 is overwritten (zero_y) or accumulated into."""
        T = x.shape[0]
        sp = self.sere_params() if (sere and self.sim is not None) else None
        abi.moe_decode_layer(x, self.w_router, self.w_gate, self.w_up, self.w_down, self.logits[:T], self.ids[:T],
                             self.gates[:T], self.counts, self.offsets, self.row_token, self.row_gate, self.active,
                             y, self.ws_route, self.ws_ffn, self.flags, zero_y, sp, self.status, stream)

    def route_and_dispatch(self, x: torch.Tensor, sere: bool, token_w: Optional[torch.Tensor] = None, stream=None):
        """Routing (+ SERE when a similarity matrix is set) and dispatch: one
        launch for uncapped batches of up to 256 tokens, separate calls
        otherwise."""
        T = x.shape[0]
        sere = sere and self.sim is not None
        if self.fused_route_dispatch_ok(T):
            self.route_dispatch(x, sere, stream)
        else:
            self.route(x, sere, stream)
            self.dispatch(T, token_w, stream)

    def dispatch(self, T: int, token_w: Optional[torch.Tensor] = None, stream=None):
        abi.moe_dispatch_capacity(self.ids[:T], self.gates[:T], self.N, self.k, self.R, self.counts, self.offsets,
                                  self.row_token, self.row_gate, self.active, self.ws_dispatch, token_w,
                                  self.capacity_factor, self.out_ids[:T], self.out_gates[:T], None,
                                  self.slot_status[:T] if self.capacity_factor > 0 else None,
                                  self.load_q if self.capacity_factor > 0 else None,
                                  self.cap_q if self.capacity_factor > 0 else None, self.status, stream,
                                  modality_bias=self.modality_bias if self.capacity_factor > 0 else None,
                                  r_v=self.r_v if self.capacity_factor > 0 else None)

    def ffn(self, x: torch.Tensor, stream=None, accumulate_into: Optional[torch.Tensor] = None,
            out: Optional[torch.Tensor] = None):
        """y = sum_j G_j E_j(x) into `out` ([T][H] fp32) or the layer's buffer,
        or added to `accumulate_into` ([T][H] fp32, e.g. a residual stream)."""
        T = x.shape[0]
        if accumulate_into is not None:
            out, flags = accumulate_into, abi.MOE_FFN_FUSE_COMBINE
        else:
            out = self.y[:T] if out is None else out
            flags = abi.MOE_FFN_FUSE_COMBINE | abi.MOE_FFN_ZERO_Y
        abi.moe_ffn_grouped(x, self.w_gate, self.w_up, self.w_down, self.k, self.offsets, self.row_token,
                            self.row_gate, self.active, out, self.ws_ffn, flags, self.status, stream)

    def forward(self, x: torch.Tensor, sere: bool = False, token_w: Optional[torch.Tensor] = None, stream=None,
                out: Optional[torch.Tensor] = None, accumulate_into: Optional[torch.Tensor] = None):
        """y[T][H] fp32: written into `out` if given, else into (a view of)
        the layer's output buffer; or added to `accumulate_into` ([T][H]
        fp32, e.g. a residual stream), which is then returned."""
        T = x.shape[0]
        if T > self.max_T:
            raise abi.MoeError("batch %d exceeds the layer's max_tokens %d" % (T, self.max_T))
        if token_w is None and self.decode_layer_ok(x):
            if accumulate_into is not None:
                self.decode_layer(x, sere, accumulate_into, zero_y=False, stream=stream)
                return accumulate_into
            y = self.y[:T] if out is None else out
            self.decode_layer(x, sere, y, zero_y=True, stream=stream)
            return y
        self.route_and_dispatch(x, sere, token_w, stream)
        self.ffn(x, stream, out=out, accumulate_into=accumulate_into)
        if accumulate_into is not None:
            return accumulate_into
        return self.y[:T] if out is None else out

    def device_status(self):
        code, detail = (int(v) for v in self.status.tolist())
        return code, detail
