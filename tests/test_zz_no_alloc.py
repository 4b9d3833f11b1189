"""moe_route_permute_noalloc: the routing/permutation entry point for callers
that cannot allocate device memory (no workspace argument; its permutation
tables live in a fixed array inside the library).  Its results must equal those
of moe_route_permute on the same inputs, on consecutive calls sharing that
array.  This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

from moe_expert_ffn_03_gb300 import binding as B
from moe_expert_ffn_03_gb300 import build, configs, synth
from oracle import mxfp8 as mx
from oracle import routing as rt

pytestmark = pytest.mark.gpu

OUTS = ("idx", "prob", "split_sizes", "row_of", "src_of", "prob_perm", "xq", "xq_s", "xq_col", "xq_col_s")


def buffers(wl, d):
    cap = B.moe_rows_capacity(d)
    dev = "cuda"
    e = lambda *s, dt: torch.full(s, 0x5A if dt == torch.uint8 else 7, dtype=dt, device=dev)  # noqa: E731
    return {"idx": e(wl.T, wl.k, dt=torch.int32), "prob": e(wl.T, wl.k, dt=torch.float32),
            "split_sizes": e(wl.E, dt=torch.int32), "row_of": e(wl.T, wl.k, dt=torch.int32),
            "src_of": e(cap, dt=torch.int32), "prob_perm": e(cap, dt=torch.float32),
            "xq": e(cap, wl.H, dt=torch.uint8), "xq_s": e(cap * wl.H // 32, dt=torch.uint8),
            "xq_col": e(wl.H, cap, dt=torch.uint8), "xq_col_s": e(wl.H * cap // 32, dt=torch.uint8)}


def run_both(wl, seed):
    d = B.dims(wl.T, wl.H, wl.I, wl.E, wl.k)
    inp = synth.make_inputs(wl, seed, device="cuda")
    ref, got = buffers(wl, d), buffers(wl, d)
    ws = torch.zeros(B.moe_workspace_size(d, True), dtype=torch.uint8, device="cuda")
    B.moe_route_permute(d, inp["logits"], inp["x"], ref["idx"], ref["prob"], ref["split_sizes"], ref["row_of"],
                        ref["src_of"], ref["prob_perm"], ref["xq"], ref["xq_s"], ref["xq_col"], ref["xq_col_s"], ws)
    B.moe_route_permute_noalloc(d, inp["logits"], inp["x"], got["idx"], got["prob"], got["split_sizes"],
                                got["row_of"], got["src_of"], got["prob_perm"], got["xq"], got["xq_s"],
                                got["xq_col"], got["xq_col_s"])
    torch.cuda.synchronize()
    rows = int(((ref["split_sizes"].long() + 127) // 128 * 128).sum())
    for k in OUTS:
        a, b = ref[k], got[k]
        if k in ("src_of", "prob_perm", "xq"):
            a, b = a[:rows], b[:rows]
        elif k == "xq_col":
            a, b = a[:, :rows], b[:, :rows]
        if a.dtype.is_floating_point:
            # same kernels on the same inputs: identical values (tolerance of the parity tests, here exact)
            assert torch.allclose(a, b, rtol=0, atol=0), k
        else:
            assert torch.equal(a, b), k
    # and directly against the oracle: routing, permutation and x codes bit-exact
    idx, prob = rt.route_topk(inp["logits"].cpu().numpy(), wl.k)
    perm = rt.permute(idx, wl.E)
    assert np.array_equal(got["idx"].cpu().numpy(), idx)
    assert np.allclose(got["prob"].cpu().numpy(), prob, rtol=2e-6, atol=1e-7)
    assert np.array_equal(got["split_sizes"].cpu().numpy(), perm["split_sizes"])
    assert np.array_equal(got["row_of"].cpu().numpy(), perm["row_of"])
    assert np.array_equal(got["src_of"][:rows].cpu().numpy(), perm["src_of"])
    x = inp["x"].float().cpu().numpy().astype(np.float64)
    x_perm = np.zeros((rows, wl.H))
    valid = perm["src_of"] >= 0
    x_perm[valid] = x[perm["src_of"][valid]]
    ref_c, _ = mx.quantize_blocks(x_perm, axis=1)
    assert np.array_equal(got["xq"][:rows].cpu().numpy(), ref_c)
    ref_c, _ = mx.quantize_blocks(x_perm, axis=0)
    assert np.array_equal(got["xq_col"][:, :rows].cpu().numpy(), ref_c.T)
    return ref


def test_noalloc_matches_workspace_entry_point_on_consecutive_calls():
    build.build()
    first = configs.small(1000, 256, 256, 16, 4, routing="biased", backward=True)
    second = configs.small(333, 384, 128, 6, 2, routing="normal", backward=True)
    r1 = run_both(first, seed=3)
    r2 = run_both(second, seed=4)
    assert int(r1["split_sizes"].sum()) == 1000 * 4 and int(r2["split_sizes"].sum()) == 333 * 2


def test_noalloc_rejects_sizes_beyond_its_scratch():
    build.build()
    d = B.dims(32768 * 16, 128, 128, 64, 2)      # E*ceil(T/32) = 1,048,576 > 262,144
    p = ctypes.c_void_p(256)
    s = B.lib().moe_route_permute_noalloc(ctypes.byref(d), *([p] * 12), None)
    assert s == 2
    assert b"scratch limit" in B.lib().moe_last_error_message()
