"""Thin ctypes binding of libmoeffn.so: one Python function per C entry point,
same names, argument marshalling only (torch tensors -> device pointers, the
current CUDA stream).  Every step of the computation runs in the library's
CUDA kernels; there is no fallback -- a missing library raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

c_int32, c_size_t, c_void_p = ctypes.c_int32, ctypes.c_size_t, ctypes.c_void_p

EXPORTS = (
    "moe_status_string", "moe_last_error_message", "moe_rows_capacity", "moe_workspace_size",
    "mxfp8_quantize", "mxfp8_quantize_dual", "moe_route_permute", "grouped_mlp_fwd", "grouped_mlp_bwd",
    "moe_unpermute_combine", "moe_get_device_error", "moe_clear_device_error", "moe_route_permute_noalloc",
    "moe_selftest_wait_timeout", "moe_router_fwd", "moe_router_bwd", "moe_gather_rows", "grouped_mlp_fwd_bf16",
    "fp8_tensor_quantize", "moe_fp8_tensor_quantize_tokens", "grouped_mlp_fwd_fp8_tensor",
    "mxfp8_quantize_experts", "fp8_tensor_quantize_experts", "moe_transpose_bf16", "grouped_mlp_bwd_bf16",
    "grouped_mlp_bwd_fp8_tensor", "moe_workspace_tensor", "moe_selftest_epilogue_quant", "moe_selftest_mma_issue",
    "moe_transpose_bf16_experts", "grouped_mlp_fwd_bf16_experts", "moe_route", "moe_permute", "moe_ep_pack",
    "moe_gather_f32",
)

# moe_ws_tensor ids (include/moe_ffn.h)
WS_TENSORS = {"a_codes": 0, "a_scales": 1, "dy_codes": 2, "dy_scales": 3, "dy_col_codes": 4, "dy_col_scales": 5,
              "dh_codes": 6, "dh_scales": 7, "dh_col_codes": 8, "dh_col_scales": 9}

MOE_OK = 0
STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_ALIGNMENT",
          4: "MOE_ERR_WORKSPACE", 5: "MOE_ERR_CUDA", 6: "MOE_ERR_DEVICE_TIMEOUT", 7: "MOE_ERR_DEVICE_BOUNDS"}


class MoeError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


class MoeDims(ctypes.Structure):
    _fields_ = [("T", c_int32), ("H", c_int32), ("I", c_int32), ("E", c_int32), ("k", c_int32),
                ("renormalize", c_int32)]


def dims(T, H, I, E, k, renormalize=1) -> MoeDims:
    return MoeDims(T, H, I, E, k, renormalize)


_lib = None


def lib_path() -> str:
    return _build.LIB_PATH


def lib() -> ctypes.CDLL:
    """Load libmoeffn.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        path = lib_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with moe_expert_ffn_03_gb300.build.build()")
        L = ctypes.CDLL(path)
        D = ctypes.POINTER(MoeDims)
        P = c_void_p
        sig = {
            "moe_status_string": ([c_int32], ctypes.c_char_p),
            "moe_last_error_message": ([], ctypes.c_char_p),
            "moe_rows_capacity": ([D], c_size_t),
            "moe_workspace_size": ([D, c_int32], c_size_t),
            "mxfp8_quantize": ([P, c_int32, c_int32, c_int32, c_int32, P, P, P], c_int32),
            "mxfp8_quantize_dual": ([P, c_int32, c_int32, c_int32, P, P, P, P, P], c_int32),
            "moe_route_permute": ([D, P, P, P, P, P, P, P, P, P, P, P, P, P, c_size_t, P], c_int32),
            "grouped_mlp_fwd": ([D, P, P, P, P, P, P, P, P, P, P, P, P, P, c_size_t, P], c_int32),
            "grouped_mlp_bwd": ([D] + [P] * 19 + [c_size_t, P], c_int32),
            "moe_unpermute_combine": ([D, P, P, P, P, P], c_int32),
            "moe_get_device_error": ([P, ctypes.POINTER(c_int32), ctypes.POINTER(c_int32), P], c_int32),
            "moe_clear_device_error": ([P, P], c_int32),
            "moe_route_permute_noalloc": ([D, P, P, P, P, P, P, P, P, P, P, P, P, P], c_int32),
            "moe_router_fwd": ([D, P, P, P, P, c_size_t, P], c_int32),
            "moe_gather_rows": ([D, P, P, P, P, P, c_size_t, P], c_int32),
            "grouped_mlp_fwd_bf16": ([D, P, P, P, P, P, P, P, P, P, c_size_t, P], c_int32),
            "moe_transpose_bf16": ([P, c_int32, c_int32, c_int32, P, P], c_int32),
            "grouped_mlp_bwd_bf16": ([D] + [P] * 15 + [c_size_t, P], c_int32),
            "moe_router_bwd": ([D, P, P, P, P, P, P, P, P, P, P, c_size_t, P], c_int32),
            "fp8_tensor_quantize": ([P, c_int32, c_int32, c_int32, P, P, P], c_int32),
            "moe_fp8_tensor_quantize_tokens": ([D, P, P, P, P, P, P, P, c_size_t, P], c_int32),
            "grouped_mlp_fwd_fp8_tensor": ([D] + [P] * 14 + [c_size_t, P], c_int32),
            "grouped_mlp_bwd_fp8_tensor": ([D] + [P] * 19 + [c_size_t, P], c_int32),
            "mxfp8_quantize_experts": ([ctypes.POINTER(P), c_int32, c_int32, c_int32, P, P, P, P, P], c_int32),
            "fp8_tensor_quantize_experts": ([ctypes.POINTER(P), c_int32, c_int32, c_int32, P, P, P], c_int32),
            "moe_selftest_wait_timeout": ([P, c_size_t, ctypes.c_int64, ctypes.POINTER(c_int32),
                                           ctypes.POINTER(c_int32), P], c_int32),
            "moe_workspace_tensor": ([D, c_int32, c_int32, ctypes.POINTER(c_size_t), ctypes.POINTER(c_size_t)],
                                     c_int32),
            "moe_selftest_epilogue_quant": ([P, c_int32, c_int32, P, P, P, P, P], c_int32),
            "moe_selftest_mma_issue": ([c_int32, P, c_size_t, ctypes.POINTER(c_int32), P], c_int32),
            "moe_transpose_bf16_experts": ([ctypes.POINTER(P), c_int32, c_int32, c_int32, P, P], c_int32),
            "moe_route": ([D, P, P, P, P, P, P, P, P, c_size_t, P], c_int32),
            "moe_permute": ([D] + [P] * 12 + [c_size_t, P], c_int32),
            "moe_ep_pack": ([D, c_int32] + [P] * 11 + [c_size_t, P], c_int32),
            "moe_gather_f32": ([P, ctypes.c_int64, P, ctypes.c_int64, P, P, P], c_int32),
            "grouped_mlp_fwd_bf16_experts": ([D, P, P, P, ctypes.POINTER(P), ctypes.POINTER(P), P, P, P, P, c_size_t,
                                              P], c_int32),
        }
        for name, (args, res) in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _lib = L
    return _lib


def _p(t):
    if t is None:
        return None
    return c_void_p(t.data_ptr())


def _st(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return c_void_p(stream.cuda_stream)


def _check(status: int):
    if status != MOE_OK:
        msg = lib().moe_last_error_message().decode()
        raise MoeError(status, msg)


def moe_rows_capacity(d: MoeDims) -> int:
    return int(lib().moe_rows_capacity(ctypes.byref(d)))


def moe_workspace_size(d: MoeDims, training: bool) -> int:
    return int(lib().moe_workspace_size(ctypes.byref(d), int(training)))


def mxfp8_quantize(src, batch, rows, cols, axis, codes, scales, stream=None):
    _check(lib().mxfp8_quantize(_p(src), batch, rows, cols, axis, _p(codes), _p(scales), _st(stream)))


def mxfp8_quantize_dual(src, batch, rows, cols, codes, scales, codes_t, scales_t, stream=None):
    _check(lib().mxfp8_quantize_dual(_p(src), batch, rows, cols, _p(codes), _p(scales), _p(codes_t), _p(scales_t),
                                     _st(stream)))


def moe_route_permute(d, logits, x, idx, prob, split_sizes, row_of, src_of, prob_perm, xq, xq_scale,
                      xq_col, xq_col_scale, workspace, stream=None):
    _check(lib().moe_route_permute(ctypes.byref(d), _p(logits), _p(x), _p(idx), _p(prob), _p(split_sizes),
                                   _p(row_of), _p(src_of), _p(prob_perm), _p(xq), _p(xq_scale), _p(xq_col),
                                   _p(xq_col_scale), _p(workspace), workspace.numel() * workspace.element_size(),
                                   _st(stream)))


def moe_route_permute_noalloc(d, logits, x, idx, prob, split_sizes, row_of, src_of, prob_perm, xq, xq_scale,
                              xq_col, xq_col_scale, stream=None):
    _check(lib().moe_route_permute_noalloc(ctypes.byref(d), _p(logits), _p(x), _p(idx), _p(prob), _p(split_sizes),
                                           _p(row_of), _p(src_of), _p(prob_perm), _p(xq), _p(xq_scale), _p(xq_col),
                                           _p(xq_col_scale), _st(stream)))


def grouped_mlp_fwd(d, xq, xq_scale, split_sizes, prob_perm, wgu_q, wgu_s, wd_q, wd_s, y, saved_gu, aq_col,
                    aq_col_scale, workspace, stream=None):
    _check(lib().grouped_mlp_fwd(ctypes.byref(d), _p(xq), _p(xq_scale), _p(split_sizes), _p(prob_perm), _p(wgu_q),
                                 _p(wgu_s), _p(wd_q), _p(wd_s), _p(y), _p(saved_gu), _p(aq_col), _p(aq_col_scale),
                                 _p(workspace), workspace.numel() * workspace.element_size(), _st(stream)))


def grouped_mlp_bwd(d, dout, split_sizes, row_of, src_of, prob_perm, saved_gu, aq_col, aq_col_scale, xq_col,
                    xq_col_scale, wguT_q, wguT_s, wdT_q, wdT_s, dx_perm, dwgu, dwd, dprob, workspace, stream=None):
    _check(lib().grouped_mlp_bwd(ctypes.byref(d), _p(dout), _p(split_sizes), _p(row_of), _p(src_of), _p(prob_perm),
                                 _p(saved_gu), _p(aq_col), _p(aq_col_scale), _p(xq_col), _p(xq_col_scale),
                                 _p(wguT_q), _p(wguT_s), _p(wdT_q), _p(wdT_s), _p(dx_perm), _p(dwgu), _p(dwd),
                                 _p(dprob), _p(workspace), workspace.numel() * workspace.element_size(),
                                 _st(stream)))


def moe_unpermute_combine(d, y_perm, row_of, prob, out, stream=None):
    _check(lib().moe_unpermute_combine(ctypes.byref(d), _p(y_perm), _p(row_of), _p(prob), _p(out), _st(stream)))


def moe_get_device_error(workspace, stream=None):
    code, site = c_int32(0), c_int32(0)
    _check(lib().moe_get_device_error(_p(workspace), ctypes.byref(code), ctypes.byref(site), _st(stream)))
    return int(code.value), int(site.value)


def moe_gather_rows(d, x, row_of, split_sizes, x_perm, workspace, stream=None):
    _check(lib().moe_gather_rows(ctypes.byref(d), _p(x), _p(row_of), _p(split_sizes), _p(x_perm), _p(workspace),
                                 workspace.numel() * workspace.element_size(), _st(stream)))


def grouped_mlp_fwd_bf16(d, x_perm, split_sizes, prob_perm, w_gu, w_d, a_perm, y, workspace, saved_gu=None,
                         stream=None):
    _check(lib().grouped_mlp_fwd_bf16(ctypes.byref(d), _p(x_perm), _p(split_sizes), _p(prob_perm), _p(w_gu),
                                      _p(w_d), _p(a_perm), _p(y), _p(saved_gu), _p(workspace),
                                      workspace.numel() * workspace.element_size(), _st(stream)))


def moe_transpose_bf16(src, batch, rows, cols, dst, stream=None):
    _check(lib().moe_transpose_bf16(_p(src), batch, rows, cols, _p(dst), _st(stream)))


def grouped_mlp_bwd_bf16(d, dout, split_sizes, row_of, src_of, prob_perm, saved_gu, x_perm, a_perm, w_guT, w_dT,
                         dx_perm, dwgu, dwd, dprob, workspace, stream=None):
    _check(lib().grouped_mlp_bwd_bf16(ctypes.byref(d), _p(dout), _p(split_sizes), _p(row_of), _p(src_of),
                                      _p(prob_perm), _p(saved_gu), _p(x_perm), _p(a_perm), _p(w_guT), _p(w_dT),
                                      _p(dx_perm), _p(dwgu), _p(dwd), _p(dprob), _p(workspace),
                                      workspace.numel() * workspace.element_size(), _st(stream)))


def moe_router_fwd(d, x, w_r, logits, workspace, stream=None):
    _check(lib().moe_router_fwd(ctypes.byref(d), _p(x), _p(w_r), _p(logits), _p(workspace),
                                workspace.numel() * workspace.element_size(), _st(stream)))


def moe_router_bwd(d, x, w_r, logits, idx, prob, dprob, dlogits, dx, dw_r, workspace, stream=None):
    _check(lib().moe_router_bwd(ctypes.byref(d), _p(x), _p(w_r), _p(logits), _p(idx), _p(prob), _p(dprob),
                                _p(dlogits), _p(dx), _p(dw_r), _p(workspace),
                                workspace.numel() * workspace.element_size(), _st(stream)))


def moe_selftest_wait_timeout(scratch, limit_ns, stream=None):
    code, site = c_int32(0), c_int32(0)
    _check(lib().moe_selftest_wait_timeout(_p(scratch), scratch.numel() * scratch.element_size(), int(limit_ns),
                                           ctypes.byref(code), ctypes.byref(site), _st(stream)))
    return int(code.value), int(site.value)


def moe_workspace_tensor(d, training, which):
    """(byte offset, bytes) of a named intermediate tensor inside a workspace."""
    off, n = c_size_t(0), c_size_t(0)
    _check(lib().moe_workspace_tensor(ctypes.byref(d), int(training), WS_TENSORS[which], ctypes.byref(off),
                                      ctypes.byref(n)))
    return int(off.value), int(n.value)


def moe_selftest_epilogue_quant(src, rows, cols, codes, scales, codes_t, scales_t, stream=None):
    _check(lib().moe_selftest_epilogue_quant(_p(src), rows, cols, _p(codes), _p(scales), _p(codes_t), _p(scales_t),
                                             _st(stream)))


def moe_selftest_mma_issue(k_steps, scratch, stream=None):
    """Launches the MMA issue-rate self-test; returns the number of CTA pairs it used."""
    pairs = c_int32(0)
    _check(lib().moe_selftest_mma_issue(int(k_steps), _p(scratch), scratch.numel() * scratch.element_size(),
                                        ctypes.byref(pairs), _st(stream)))
    return int(pairs.value)


def moe_clear_device_error(workspace, stream=None):
    _check(lib().moe_clear_device_error(_p(workspace), _st(stream)))


def fp8_tensor_quantize(src, batch, rows, cols, codes, amax, stream=None):
    _check(lib().fp8_tensor_quantize(_p(src), batch, rows, cols, _p(codes), _p(amax), _st(stream)))


def moe_fp8_tensor_quantize_tokens(d, x, idx, row_of, split_sizes, xq, amax_x, workspace, stream=None):
    _check(lib().moe_fp8_tensor_quantize_tokens(ctypes.byref(d), _p(x), _p(idx), _p(row_of), _p(split_sizes), _p(xq),
                                                _p(amax_x), _p(workspace),
                                                workspace.numel() * workspace.element_size(), _st(stream)))


def grouped_mlp_fwd_fp8_tensor(d, xq, amax_x, split_sizes, prob_perm, wgu_q, amax_gu, wd_q, amax_d, a_perm, aq,
                               amax_a, y, workspace, saved_gu=None, stream=None):
    _check(lib().grouped_mlp_fwd_fp8_tensor(ctypes.byref(d), _p(xq), _p(amax_x), _p(split_sizes), _p(prob_perm),
                                            _p(wgu_q), _p(amax_gu), _p(wd_q), _p(amax_d), _p(a_perm), _p(aq),
                                            _p(amax_a), _p(y), _p(saved_gu), _p(workspace),
                                            workspace.numel() * workspace.element_size(), _st(stream)))


def grouped_mlp_bwd_fp8_tensor(d, dout, idx, split_sizes, row_of, prob_perm, saved_gu, xq, amax_x, aq, amax_a,
                               wgu_q, amax_gu, wd_q, amax_d, dx_perm, dwgu, dwd, dprob, workspace, stream=None):
    _check(lib().grouped_mlp_bwd_fp8_tensor(ctypes.byref(d), _p(dout), _p(idx), _p(split_sizes), _p(row_of),
                                            _p(prob_perm), _p(saved_gu), _p(xq), _p(amax_x), _p(aq), _p(amax_a),
                                            _p(wgu_q), _p(amax_gu), _p(wd_q), _p(amax_d), _p(dx_perm), _p(dwgu),
                                            _p(dwd), _p(dprob), _p(workspace),
                                            workspace.numel() * workspace.element_size(), _st(stream)))


def _ptr_array(tensors):
    """Host array of the device pointers of a list of tensors (one per expert)."""
    return (c_void_p * len(tensors))(*[t.data_ptr() for t in tensors])


def mxfp8_quantize_experts(w_list, rows, cols, codes, scales, codes_t=None, scales_t=None, stream=None):
    _check(lib().mxfp8_quantize_experts(_ptr_array(w_list), len(w_list), rows, cols, _p(codes), _p(scales),
                                        _p(codes_t), _p(scales_t), _st(stream)))


def _wsb(workspace):
    return workspace.numel() * workspace.element_size()


def moe_route(d, logits, idx, prob, split_sizes, row_of, src_of, prob_perm, workspace, stream=None):
    _check(lib().moe_route(ctypes.byref(d), _p(logits), _p(idx), _p(prob), _p(split_sizes), _p(row_of), _p(src_of),
                           _p(prob_perm), _p(workspace), _wsb(workspace), _st(stream)))


def moe_permute(d, idx, prob, x, split_sizes, row_of, src_of, prob_perm, xq, xq_scale, xq_col, xq_col_scale,
                workspace, stream=None):
    _check(lib().moe_permute(ctypes.byref(d), _p(idx), _p(prob), _p(x), _p(split_sizes), _p(row_of), _p(src_of),
                             _p(prob_perm), _p(xq), _p(xq_scale), _p(xq_col), _p(xq_col_scale), _p(workspace),
                             _wsb(workspace), _st(stream)))


def moe_ep_pack(d, world, x, idx, prob, row_of, split_sizes, send_x, send_prob, send_eid, pos_of, rank_counts,
                workspace, stream=None):
    _check(lib().moe_ep_pack(ctypes.byref(d), int(world), _p(x), _p(idx), _p(prob), _p(row_of), _p(split_sizes),
                             _p(send_x), _p(send_prob), _p(send_eid), _p(pos_of), _p(rank_counts), _p(workspace),
                             _wsb(workspace), _st(stream)))


def moe_gather_f32(src, map_, n, out, workspace, stream=None):
    _check(lib().moe_gather_f32(_p(src), src.numel(), _p(map_), int(n), _p(out), _p(workspace), _st(stream)))


def moe_transpose_bf16_experts(w_list, rows, cols, dst, stream=None):
    _check(lib().moe_transpose_bf16_experts(_ptr_array(w_list), len(w_list), rows, cols, _p(dst), _st(stream)))


def grouped_mlp_fwd_bf16_experts(d, x_perm, split_sizes, prob_perm, w_gu_list, w_d_list, a_perm, y, workspace,
                                 saved_gu=None, stream=None):
    _check(lib().grouped_mlp_fwd_bf16_experts(ctypes.byref(d), _p(x_perm), _p(split_sizes), _p(prob_perm),
                                              _ptr_array(w_gu_list), _ptr_array(w_d_list), _p(a_perm), _p(y),
                                              _p(saved_gu), _p(workspace), workspace.numel() * workspace.element_size(),
                                              _st(stream)))


def fp8_tensor_quantize_experts(w_list, rows, cols, codes, amax, stream=None):
    _check(lib().fp8_tensor_quantize_experts(_ptr_array(w_list), len(w_list), rows, cols, _p(codes), _p(amax),
                                             _st(stream)))
