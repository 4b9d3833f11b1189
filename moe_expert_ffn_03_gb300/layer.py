"""One expert-FFN layer step on the device: buffer allocation (torch) plus the
C entry points called in order.  No arithmetic happens here.

Forward:  moe_route_permute -> grouped_mlp_fwd -> moe_unpermute_combine
Backward: grouped_mlp_bwd -> moe_unpermute_combine (dx_perm -> dx)
Weights:  mxfp8_quantize of the bf16 master weights (axis 0 for the forward,
          axis 1 for the backward copies), once per optimizer step.
"""
from __future__ import annotations

import torch

from . import binding as B

U8 = torch.uint8

# Routing: top-k and the per-expert scan of the token masks are one launch while the
# masks hold at most 16384 words (E * ceil(T/32)), else two; the permutation itself is
# finished by the launch that gathers and quantizes the x rows.
ROUTE_SCAN_FUSED_MAX_WORDS = 16384


def route_launches(T: int, E: int) -> int:
    """Launches of routing up to (not including) the row gather-quantize."""
    return 1 if E * ((T + 31) // 32) <= ROUTE_SCAN_FUSED_MAX_WORDS else 2


def launches_per_step(T: int, E: int, k: int, training: bool) -> int:
    """Kernel launches of one step (quantize_weights + forward [+ backward]).

    weights 2 (both orientations of W_gu and of W_d); routing 1 or 2; permutation with the
    x rows gathered and quantized (padding rows zeroed in the same launch) 1; forward 2
    GEMMs; combine 1.  Training adds x along tokens 1 and the backward: dY rows (with
    padding rows) 1, dY along tokens 1, down dgrad 1, dprob reduce 1, down wgrad 1,
    gate_up dgrad 1, gate_up wgrad 1, and the dx combine 1.
    """
    fwd = 2 + route_launches(T, E) + 1 + 2 + 1
    return fwd + (1 + 8 if training else 0)


class _Range:
    """An NVTX range around one call when the layer asks for it (otherwise nothing)."""

    def __init__(self, on: bool, name: str):
        self.on, self.name = on, name

    def __enter__(self):
        if self.on:
            torch.cuda.nvtx.range_push(self.name)

    def __exit__(self, *exc):
        if self.on:
            torch.cuda.nvtx.range_pop()
        return False


class ExpertFFN:
    """Buffers of one layer for fixed sizes (T, H, I, E, k) on one device."""

    def __init__(self, T, H, I, E, k, training=True, renormalize=True, device="cuda", bf16_training=False,
                 nvtx=False):
        """bf16_training: also size the workspace for backward_bf16 (the bf16 training path).
        nvtx: mark every call with an NVTX range named after it (for profilers)."""
        self.nvtx = nvtx
        self.T, self.H, self.I, self.E, self.k = T, H, I, E, k
        self.training = training
        self.bf16_training = bool(training and bf16_training)
        self.d = B.dims(T, H, I, E, k, int(renormalize))
        self.cap = B.moe_rows_capacity(self.d)
        if self.cap == 0:
            raise B.MoeError(2, f"unsupported sizes T={T} H={H} I={I} E={E} k={k}")
        cap = self.cap
        dev = torch.device(device)
        z = lambda *s, dt: torch.zeros(*s, dtype=dt, device=dev)  # noqa: E731
        e = lambda *s, dt: torch.empty(*s, dtype=dt, device=dev)  # noqa: E731
        self.ws = z(B.moe_workspace_size(self.d, 2 if self.bf16_training else int(training)), dt=U8)
        self.idx = e(T, k, dt=torch.int32)
        self.prob = e(T, k, dt=torch.float32)
        self.split_sizes = e(E, dt=torch.int32)
        self.row_of = e(T, k, dt=torch.int32)
        self.src_of = e(cap, dt=torch.int32)
        self.prob_perm = e(cap, dt=torch.float32)
        self.xq = e(cap, H, dt=U8)
        self.xq_s = e(cap * H // 32, dt=U8)
        self.y = e(cap, H, dt=torch.bfloat16)
        self.out = e(T, H, dt=torch.bfloat16)
        self.wgu_q = e(E, 2 * I, H, dt=U8)
        self.wgu_s = e(E * 2 * I * H // 32, dt=U8)
        self.wd_q = e(E, H, I, dt=U8)
        self.wd_s = e(E * H * I // 32, dt=U8)
        if training:
            self.xq_col = e(H, cap, dt=U8)
            self.xq_col_s = e(H * cap // 32, dt=U8)
            self.saved_gu = e(cap, 2 * I, dt=torch.bfloat16)
            self.aq_col = e(I, cap, dt=U8)
            self.aq_col_s = e(I * cap // 32, dt=U8)
            self.dx_perm = e(cap, H, dt=torch.bfloat16)
            self.dx = e(T, H, dt=torch.bfloat16)
            self.dwgu = e(E, 2 * I, H, dt=torch.bfloat16)
            self.dwd = e(E, H, I, dt=torch.bfloat16)
            self.dprob = e(T, k, dt=torch.float32)
            self.wguT_q = e(E, H, 2 * I, dt=U8)
            self.wguT_s = e(E * H * 2 * I // 32, dt=U8)
            self.wdT_q = e(E, I, H, dt=U8)
            self.wdT_s = e(E * I * H // 32, dt=U8)
        else:
            self.xq_col = self.xq_col_s = self.saved_gu = self.aq_col = self.aq_col_s = None

    # ---- steps -------------------------------------------------------------------
    def quantize_weights(self, w_gu, w_d, stream=None):
        """MX copies of the master weights: stacked tensors [E][2I][H] and [E][H][I], or
        lists of E per-expert tensors [2I][H] and [H][I]."""
        with _Range(self.nvtx, "moe.quantize_weights"):
            E, H, I = self.E, self.H, self.I
            if isinstance(w_gu, (list, tuple)):
                t = self.training
                B.mxfp8_quantize_experts(w_gu, 2 * I, H, self.wgu_q, self.wgu_s, self.wguT_q if t else None,
                                         self.wguT_s if t else None, stream)
                B.mxfp8_quantize_experts(w_d, H, I, self.wd_q, self.wd_s, self.wdT_q if t else None,
                                         self.wdT_s if t else None, stream)
                return
            if self.training:
                B.mxfp8_quantize_dual(w_gu, E, 2 * I, H, self.wgu_q, self.wgu_s, self.wguT_q, self.wguT_s, stream)
                B.mxfp8_quantize_dual(w_d, E, H, I, self.wd_q, self.wd_s, self.wdT_q, self.wdT_s, stream)
            else:
                B.mxfp8_quantize(w_gu, E, 2 * I, H, 0, self.wgu_q, self.wgu_s, stream)
                B.mxfp8_quantize(w_d, E, H, I, 0, self.wd_q, self.wd_s, stream)

    def route(self, logits, x, stream=None):
        with _Range(self.nvtx, "moe.route_permute"):
            B.moe_route_permute(self.d, logits, x, self.idx, self.prob, self.split_sizes, self.row_of, self.src_of,
                                self.prob_perm, self.xq, self.xq_s, self.xq_col, self.xq_col_s, self.ws, stream)

    def ffn_forward(self, stream=None):
        with _Range(self.nvtx, "moe.grouped_mlp_fwd"):
            B.grouped_mlp_fwd(self.d, self.xq, self.xq_s, self.split_sizes, self.prob_perm, self.wgu_q, self.wgu_s,
                              self.wd_q, self.wd_s, self.y, self.saved_gu, self.aq_col, self.aq_col_s, self.ws, stream)

    def combine_out(self, stream=None):
        with _Range(self.nvtx, "moe.combine"):
            B.moe_unpermute_combine(self.d, self.y, self.row_of, None, self.out, stream)

    def forward(self, logits, x, stream=None):
        self.route(logits, x, stream)
        self.ffn_forward(stream)
        self.combine_out(stream)
        return self.out

    def ffn_backward(self, dout, stream=None):
        with _Range(self.nvtx, "moe.grouped_mlp_bwd"):
            B.grouped_mlp_bwd(self.d, dout, self.split_sizes, self.row_of, self.src_of, self.prob_perm, self.saved_gu,
                              self.aq_col, self.aq_col_s, self.xq_col, self.xq_col_s, self.wguT_q, self.wguT_s,
                              self.wdT_q, self.wdT_s, self.dx_perm, self.dwgu, self.dwd, self.dprob, self.ws, stream)

    def combine_dx(self, stream=None):
        with _Range(self.nvtx, "moe.combine_dx"):
            B.moe_unpermute_combine(self.d, self.dx_perm, self.row_of, None, self.dx, stream)

    def backward(self, dout, stream=None):
        self.ffn_backward(dout, stream)
        self.combine_dx(stream)
        return self.dx

    # ---- one step as a CUDA graph (for launch-bound sizes) -------------------------------
    def step(self, w_gu, w_d, logits, x, dout=None, stream=None):
        """quantize_weights + forward (+ backward when training) on the given tensors."""
        self.quantize_weights(w_gu, w_d, stream)
        self.forward(logits, x, stream)
        if self.training:
            self.backward(dout, stream)

    def capture_step(self, w_gu, w_d, logits, x, dout=None) -> torch.cuda.CUDAGraph:
        """Record step() on these tensors as one CUDA graph.  Every launch of the step is
        replayed by graph.replay(); refill the same tensors in place between replays.
        The step runs once eagerly first (on a side stream) so that one-time setup
        (kernel attributes, driver entry points) happens outside the capture."""
        side = torch.cuda.Stream(self.ws.device)
        side.wait_stream(torch.cuda.current_stream(self.ws.device))
        with torch.cuda.stream(side):
            self.step(w_gu, w_d, logits, x, dout)
        torch.cuda.current_stream(self.ws.device).wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            self.step(w_gu, w_d, logits, x, dout)
        return graph

    # ---- bf16 forward (no quantization), on the routing of route() ----------------------
    def forward_bf16(self, x, w_gu, w_d, stream=None):
        """After route(): gather x rows, bf16 grouped gate_up + ScaledSwiGLU + down, combine.
        w_gu, w_d: stacked [E][2I][H], [E][H][I], or lists of E per-expert tensors."""
        if not hasattr(self, "x_perm"):
            dev = self.ws.device
            self.x_perm = torch.empty(self.cap, self.H, dtype=torch.bfloat16, device=dev)
            self.a_perm = torch.empty(self.cap, self.I, dtype=torch.bfloat16, device=dev)
            self.y_b16 = torch.empty(self.cap, self.H, dtype=torch.bfloat16, device=dev)
            self.out_b16 = torch.empty(self.T, self.H, dtype=torch.bfloat16, device=dev)
        B.moe_gather_rows(self.d, x, self.row_of, self.split_sizes, self.x_perm, self.ws, stream)
        saved = self.saved_gu if self.bf16_training else None
        if isinstance(w_gu, (list, tuple)):                 # one weight tensor per expert
            B.grouped_mlp_fwd_bf16_experts(self.d, self.x_perm, self.split_sizes, self.prob_perm, w_gu, w_d,
                                           self.a_perm, self.y_b16, self.ws, saved, stream)
        else:
            B.grouped_mlp_fwd_bf16(self.d, self.x_perm, self.split_sizes, self.prob_perm, w_gu, w_d, self.a_perm,
                                   self.y_b16, self.ws, saved, stream)
        B.moe_unpermute_combine(self.d, self.y_b16, self.row_of, None, self.out_b16, stream)
        return self.out_b16

    # ---- bf16 training path: transposed weights once per step, then the backward ------------
    def transpose_weights_bf16(self, w_gu, w_d, stream=None):
        """W_gu^T [E][H][2I] and W_d^T [E][I][H] for backward_bf16 (once per step); the weights
        stacked or as lists of per-expert tensors."""
        if not hasattr(self, "wguT16"):
            dev = self.ws.device
            self.wguT16 = torch.empty(self.E, self.H, 2 * self.I, dtype=torch.bfloat16, device=dev)
            self.wdT16 = torch.empty(self.E, self.I, self.H, dtype=torch.bfloat16, device=dev)
        if isinstance(w_gu, (list, tuple)):                 # one weight tensor per expert
            B.moe_transpose_bf16_experts(w_gu, 2 * self.I, self.H, self.wguT16, stream)
            B.moe_transpose_bf16_experts(w_d, self.H, self.I, self.wdT16, stream)
            return
        B.moe_transpose_bf16(w_gu, self.E, 2 * self.I, self.H, self.wguT16, stream)
        B.moe_transpose_bf16(w_d, self.E, self.H, self.I, self.wdT16, stream)

    def backward_bf16(self, dout, stream=None):
        """After forward_bf16 and transpose_weights_bf16 (layer built with bf16_training=True)."""
        if not self.bf16_training:
            raise RuntimeError("backward_bf16 needs ExpertFFN(..., bf16_training=True)")
        if not hasattr(self, "dx16"):
            dev = self.ws.device
            self.dx16 = torch.empty(self.T, self.H, dtype=torch.bfloat16, device=dev)
            self.dwgu16 = torch.empty(self.E, 2 * self.I, self.H, dtype=torch.bfloat16, device=dev)
            self.dwd16 = torch.empty(self.E, self.H, self.I, dtype=torch.bfloat16, device=dev)
            self.dprob16 = torch.empty(self.T, self.k, dtype=torch.float32, device=dev)
        B.grouped_mlp_bwd_bf16(self.d, dout, self.split_sizes, self.row_of, self.src_of, self.prob_perm,
                               self.saved_gu, self.x_perm, self.a_perm, self.wguT16, self.wdT16, self.dx_perm,
                               self.dwgu16, self.dwd16, self.dprob16, self.ws, stream)
        B.moe_unpermute_combine(self.d, self.dx_perm, self.row_of, None, self.dx16, stream)
        return self.dx16

    # ---- per-tensor FP8 forward (one scale per expert operand tensor) ------------------
    def quantize_weights_fp8_tensor(self, w_gu, w_d, stream=None):
        """E4M3 codes of W_gu and W_d with one dynamic scale per expert weight."""
        if not hasattr(self, "t8_wgu"):
            dev = self.ws.device
            self.t8_wgu = torch.empty(self.E, 2 * self.I, self.H, dtype=U8, device=dev)
            self.t8_wd = torch.empty(self.E, self.H, self.I, dtype=U8, device=dev)
            self.t8_amax_gu = torch.empty(self.E, dtype=torch.float32, device=dev)
            self.t8_amax_d = torch.empty(self.E, dtype=torch.float32, device=dev)
        if isinstance(w_gu, (list, tuple)):
            B.fp8_tensor_quantize_experts(w_gu, 2 * self.I, self.H, self.t8_wgu, self.t8_amax_gu, stream)
            B.fp8_tensor_quantize_experts(w_d, self.H, self.I, self.t8_wd, self.t8_amax_d, stream)
            return
        B.fp8_tensor_quantize(w_gu, self.E, 2 * self.I, self.H, self.t8_wgu, self.t8_amax_gu, stream)
        B.fp8_tensor_quantize(w_d, self.E, self.H, self.I, self.t8_wd, self.t8_amax_d, stream)

    def forward_fp8_tensor(self, x, stream=None):
        """After route() and quantize_weights_fp8_tensor(): per-tensor FP8 x rows, grouped
        gate_up + ScaledSwiGLU (bf16 a), per-tensor FP8 a, grouped down, combine."""
        if not hasattr(self, "t8_xq"):
            dev = self.ws.device
            self.t8_xq = torch.empty(self.cap, self.H, dtype=U8, device=dev)
            self.t8_a = torch.empty(self.cap, self.I, dtype=torch.bfloat16, device=dev)
            self.t8_aq = torch.empty(self.cap, self.I, dtype=U8, device=dev)
            self.t8_y = torch.empty(self.cap, self.H, dtype=torch.bfloat16, device=dev)
            self.t8_out = torch.empty(self.T, self.H, dtype=torch.bfloat16, device=dev)
            self.t8_amax_x = torch.empty(self.E, dtype=torch.float32, device=dev)
            self.t8_amax_a = torch.empty(self.E, dtype=torch.float32, device=dev)
        B.moe_fp8_tensor_quantize_tokens(self.d, x, self.idx, self.row_of, self.split_sizes, self.t8_xq,
                                         self.t8_amax_x, self.ws, stream)
        B.grouped_mlp_fwd_fp8_tensor(self.d, self.t8_xq, self.t8_amax_x, self.split_sizes, self.prob_perm, self.t8_wgu,
                                     self.t8_amax_gu, self.t8_wd, self.t8_amax_d, self.t8_a, self.t8_aq,
                                     self.t8_amax_a, self.t8_y, self.ws, self.saved_gu if self.training else None,
                                     stream)
        B.moe_unpermute_combine(self.d, self.t8_y, self.row_of, None, self.t8_out, stream)
        return self.t8_out

    def backward_fp8_tensor(self, dout, stream=None):
        """After forward_fp8_tensor on a training layer: the per-tensor FP8 backward
        (its own workspace, allocated on first use); results in t8_dx, t8_dwgu, t8_dwd,
        t8_dprob."""
        if not self.training:
            raise RuntimeError("backward_fp8_tensor needs a training layer")
        if not hasattr(self, "ws_t8"):
            dev = self.ws.device
            self.ws_t8 = torch.zeros(B.moe_workspace_size(self.d, 3), dtype=U8, device=dev)
            self.t8_dx = torch.empty(self.T, self.H, dtype=torch.bfloat16, device=dev)
            self.t8_dwgu = torch.empty(self.E, 2 * self.I, self.H, dtype=torch.bfloat16, device=dev)
            self.t8_dwd = torch.empty(self.E, self.H, self.I, dtype=torch.bfloat16, device=dev)
            self.t8_dprob = torch.empty(self.T, self.k, dtype=torch.float32, device=dev)
        B.grouped_mlp_bwd_fp8_tensor(self.d, dout, self.idx, self.split_sizes, self.row_of, self.prob_perm,
                                     self.saved_gu, self.t8_xq, self.t8_amax_x, self.t8_aq, self.t8_amax_a,
                                     self.t8_wgu, self.t8_amax_gu, self.t8_wd, self.t8_amax_d, self.dx_perm,
                                     self.t8_dwgu, self.t8_dwd, self.t8_dprob, self.ws_t8, stream)
        B.moe_unpermute_combine(self.d, self.dx_perm, self.row_of, None, self.t8_dx, stream)
        return self.t8_dx

    # ---- router (optional: when the logits come from x) ------------------------------
    def router_forward(self, x, w_r, stream=None):
        """logits = x W_r^T into self.logits (allocated on first use)."""
        if not hasattr(self, "logits"):
            self.logits = torch.empty(self.T, self.E, dtype=torch.float32, device=self.ws.device)
        B.moe_router_fwd(self.d, x, w_r, self.logits, self.ws, stream)
        return self.logits

    def router_backward(self, x, w_r, stream=None):
        """After backward(): dlogits, dW_r, and the router's term added into self.dx."""
        if not hasattr(self, "dlogits"):
            self.dlogits = torch.empty(self.T, self.E, dtype=torch.float32, device=self.ws.device)
            self.dw_r = torch.empty(self.E, self.H, dtype=torch.float32, device=self.ws.device)
        B.moe_router_bwd(self.d, x, w_r, self.logits, self.idx, self.prob, self.dprob, self.dlogits, self.dx,
                         self.dw_r, self.ws, stream)
        return self.dx

    def workspace_tensor(self, which: str) -> torch.Tensor:
        """A uint8 view of a named intermediate tensor in this layer's workspace (binding.WS_TENSORS:
        the MX codes and tile-layout scales of a, dY and dH; see moe_workspace_tensor)."""
        training = 2 if self.bf16_training else int(self.training)
        off, n = B.moe_workspace_tensor(self.d, training, which)
        return self.ws[off:off + n]

    def device_error(self, stream=None):
        """(code, site) of the first device error recorded in any workspace of this layer."""
        for ws in (self.ws, getattr(self, "ws_t8", None)):
            if ws is not None:
                code, site = B.moe_get_device_error(ws, stream)
                if code != 0:
                    return code, site
        return 0, 0

    def padded_rows(self) -> int:
        s = self.split_sizes.to("cpu", torch.int64)
        return int(((s + 127) // 128 * 128).sum())
