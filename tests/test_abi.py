"""The C-ABI library loads and exports every entry point the header declares;
host-side argument checks answer without touching a GPU."""
import ctypes
import os
import re

import pytest

from moe_expert_ffn_03_gb300 import binding as B
from moe_expert_ffn_03_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_ffn.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(\w+)\s*\(", text, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return B.lib()


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("mxfp8_quantize", "moe_route_permute", "grouped_mlp_fwd", "grouped_mlp_bwd",
              "moe_unpermute_combine", "moe_workspace_size", "moe_get_device_error"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in declared_functions():
        assert hasattr(lib, n), n
    assert set(B.EXPORTS) == set(declared_functions())


def test_capacity_and_workspace_sizes(lib):
    d = B.dims(16384, 4096, 14336, 8, 2)
    cap = B.moe_rows_capacity(d)
    assert cap == 32768 + 128 * 8
    fwd = B.moe_workspace_size(d, False)
    bwd = B.moe_workspace_size(d, True)
    assert fwd >= cap * 14336 * (1 + 1 / 32)
    assert bwd > fwd + 2 * cap * 2 * 14336
    assert B.moe_rows_capacity(B.dims(10, 100, 128, 4, 2)) == 0       # H not a multiple of 128
    assert B.moe_rows_capacity(B.dims(10, 128, 128, 4, 9)) == 0       # k > 8


def test_host_checks_fail_before_launch(lib):
    s = lib.mxfp8_quantize(None, 1, 128, 128, 0, None, None, None)
    assert s == 1
    assert b"NULL" in lib.moe_last_error_message()
    s = lib.mxfp8_quantize(ctypes.c_void_p(16), 1, 100, 128, 0, ctypes.c_void_p(16), ctypes.c_void_p(16), None)
    assert s == 2
    s = lib.mxfp8_quantize(ctypes.c_void_p(8), 1, 128, 128, 0, ctypes.c_void_p(16), ctypes.c_void_p(16), None)
    assert s == 3
    d = B.dims(64, 128, 128, 4, 2)
    s = lib.grouped_mlp_fwd(ctypes.byref(d), *([ctypes.c_void_p(256)] * 9), None, None, None,
                            ctypes.c_void_p(256), 16, None)
    assert s == 4                                                     # workspace too small
    assert lib.moe_status_string(6) == b"MOE_ERR_DEVICE_TIMEOUT"


def header_param_counts():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    out = {}
    for m in re.finditer(r"\b(\w+)\s*\(([^;{]*?)\)\s*;", text, flags=re.S):
        params = m.group(2).strip()
        out[m.group(1)] = 0 if params in ("", "void") else params.count(",") + 1
    return out


def test_binding_signatures_match_header(lib):
    counts = header_param_counts()
    for name in B.EXPORTS:
        assert len(getattr(lib, name).argtypes) == counts[name], name


def test_selftest_checks_arguments_before_launch(lib):
    code, site = ctypes.c_int32(0), ctypes.c_int32(0)
    s = lib.moe_selftest_wait_timeout(ctypes.c_void_p(256), 1024, 20_000_000, ctypes.byref(code),
                                      ctypes.byref(site), None)
    assert s == 4                                                     # scratch too small
    s = lib.moe_selftest_wait_timeout(ctypes.c_void_p(256), 1 << 20, 10, ctypes.byref(code),
                                      ctypes.byref(site), None)
    assert s == 1                                                     # limit out of range


def test_expert_pointer_arrays_checked_on_the_host(lib):
    P = ctypes.c_void_p
    good = (P * 2)(256, 512)
    s = lib.mxfp8_quantize_experts(None, 2, 128, 128, P(256), P(256), None, None, None)
    assert s == 1                                                     # no pointer array
    s = lib.mxfp8_quantize_experts(good, 0, 128, 128, P(256), P(256), None, None, None)
    assert s == 2                                                     # E out of range
    s = lib.mxfp8_quantize_experts((P * 2)(256, 520), 2, 128, 128, P(256), P(256), None, None, None)
    assert s == 3 and b"expert 1" in lib.moe_last_error_message()   # misaligned expert weight
    s = lib.mxfp8_quantize_experts((P * 2)(256, None), 2, 128, 128, P(256), P(256), None, None, None)
    assert s == 1 and b"expert 1" in lib.moe_last_error_message()
    s = lib.mxfp8_quantize_experts(good, 2, 128, 128, P(256), P(256), P(256), None, None)
    assert s == 1                                                     # codes_t without scales_t
    s = lib.fp8_tensor_quantize_experts(good, 300, 128, 128, P(256), P(256), None)
    assert s == 2
    s = lib.fp8_tensor_quantize_experts(good, 2, 128, 100, P(256), P(256), None)
    assert s == 2                                                     # cols not a multiple of 8


def test_training_path_entry_points_check_arguments_on_the_host(lib):
    P = ctypes.c_void_p
    d = B.dims(64, 128, 128, 4, 2)
    # workspace smaller than the mode each backward needs
    for name, n_ptr in (("grouped_mlp_bwd_bf16", 15), ("grouped_mlp_bwd_fp8_tensor", 19)):   # pointers incl. ws
        s = getattr(lib, name)(ctypes.byref(d), *([P(256)] * n_ptr), 16, None)
        assert s == 4, name
    assert lib.moe_workspace_size(ctypes.byref(d), 2) > lib.moe_workspace_size(ctypes.byref(d), 1)
    assert lib.moe_workspace_size(ctypes.byref(d), 3) > lib.moe_workspace_size(ctypes.byref(d), 1)
    assert lib.moe_workspace_size(ctypes.byref(d), 4) == 0
    # a NULL amax array
    args = [P(256)] * 19
    args[7] = None                                                    # amax_x
    s = lib.grouped_mlp_bwd_fp8_tensor(ctypes.byref(d), *args, 1 << 40, None)
    assert s == 1 and b"amax" in lib.moe_last_error_message()
    # transposes take multiples of 128
    assert lib.moe_transpose_bf16(P(256), 1, 128, 100, P(256), None) == 2
    assert lib.moe_transpose_bf16(None, 1, 128, 128, P(256), None) == 1
    # the bf16 forward checks the optional saved_gu's alignment
    s = lib.grouped_mlp_fwd_bf16(ctypes.byref(d), *([P(256)] * 7), P(8), P(256), 1 << 40, None)
    assert s == 3


def test_router_entry_points_check_arguments_on_the_host(lib):
    P = ctypes.c_void_p
    d = B.dims(64, 128, 128, 4, 2)
    need = lib.moe_workspace_size(ctypes.byref(d), 0)
    s = lib.moe_router_fwd(ctypes.byref(d), P(256), P(256), P(256), None, need, None)
    assert s == 4                                                     # no workspace
    s = lib.moe_router_fwd(ctypes.byref(d), P(256), P(256), P(256), P(256), need - 1, None)
    assert s == 4                                                     # workspace too small
    s = lib.moe_router_fwd(ctypes.byref(d), P(264), P(256), P(256), P(256), need, None)
    assert s == 3 and b"x" in lib.moe_last_error_message()           # x not 16-byte aligned
    s = lib.moe_router_fwd(ctypes.byref(d), None, P(256), P(256), P(256), need, None)
    assert s == 1
    s = lib.moe_router_bwd(ctypes.byref(d), *([P(256)] * 10), 16, None)
    assert s == 4                                                     # workspace too small


def test_workspace_tensor_offsets(lib):
    """Named workspace tensors: sizes follow their documented shapes, they are 256-byte
    aligned, disjoint and inside moe_workspace_size; backward tensors need a training
    workspace."""
    d = B.dims(300, 256, 384, 6, 2)
    cap = B.moe_rows_capacity(d)
    H, I = 256, 384
    want = {"a_codes": cap * I, "a_scales": cap * I // 32, "dy_codes": cap * H, "dy_scales": cap * H // 32,
            "dy_col_codes": H * cap, "dy_col_scales": H * cap // 32, "dh_codes": cap * 2 * I,
            "dh_scales": cap * 2 * I // 32, "dh_col_codes": 2 * I * cap, "dh_col_scales": 2 * I * cap // 32}
    for training in (1, 2, 3):
        total = B.moe_workspace_size(d, training)
        spans = []
        for name, n in want.items():
            off, got = B.moe_workspace_tensor(d, training, name)
            assert got == n, name
            assert off % 256 == 0 and off + n <= total, name
            spans.append((off, off + n))
        spans.sort()
        assert all(a[1] <= b[0] for a, b in zip(spans, spans[1:]))
        assert spans[0][0] >= 256                       # the device error word comes first
    off, n = B.moe_workspace_tensor(d, 0, "a_codes")
    assert n == cap * I and off + n <= B.moe_workspace_size(d, 0)
    with pytest.raises(B.MoeError):
        B.moe_workspace_tensor(d, 0, "dy_codes")
    off_c, size = ctypes.c_size_t(0), ctypes.c_size_t(0)
    assert lib.moe_workspace_tensor(ctypes.byref(d), 1, 99, ctypes.byref(off_c), ctypes.byref(size)) == 1


def test_selftest_entry_points_check_their_arguments(lib):
    p = ctypes.c_void_p(256)
    pairs = ctypes.c_int32(0)
    assert lib.moe_selftest_mma_issue(0, p, 256, ctypes.byref(pairs), None) == 1          # k_steps < 1
    assert lib.moe_selftest_mma_issue(10, ctypes.c_void_p(16), 256, ctypes.byref(pairs), None) == 3
    assert lib.moe_selftest_mma_issue(10, p, 64, ctypes.byref(pairs), None) == 4          # scratch too small
    assert lib.moe_selftest_epilogue_quant(p, 128, 100, p, p, p, p, None) == 2           # cols % 128
    assert lib.moe_selftest_epilogue_quant(None, 128, 128, p, p, p, p, None) == 1


def test_noalloc_names_the_bad_field(lib):
    """The workspace-free routing call applies moe_route_permute's own size checks."""
    p = ctypes.c_void_p(256)
    d = B.dims(64, 128, 128, 4, 5)                   # k > E
    assert lib.moe_route_permute_noalloc(ctypes.byref(d), *([p] * 12), None) == 2
    assert b"k=5" in lib.moe_last_error_message()
    d = B.dims(64, 100, 128, 4, 2)                   # H not a multiple of 128
    assert lib.moe_route_permute_noalloc(ctypes.byref(d), *([p] * 12), None) == 2
    assert b"H=100" in lib.moe_last_error_message()
