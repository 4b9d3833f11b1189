"""GPU router (forward logits, backward through the top-k softmax) vs the oracle.

The oracle computes its own logits (float64 sums rounded to float32) and routes
on them; the device routes on its float32 sums.  The inputs are checked, on the
oracle side, to keep every token's k-th and (k+1)-th logits further apart than
the two sides' sums can differ, so both take the same top-k decisions; the
device's choice must then equal the oracle's exactly.
"""
import numpy as np
import pytest
import torch

from helpers import assert_close, rel_frob
from moe_expert_ffn_03_gb300 import binding as B, build, configs, synth
from moe_expert_ffn_03_gb300.layer import ExpertFFN
from oracle import expert_ffn as ef
from oracle import router as ro
from oracle import routing as rt

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()


def f64(t):
    return t.float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("T,H,E", [(300, 256, 8), (70, 128, 64), (1000, 384, 256), (16384, 4096, 8),
                                   (257, 128, 5), (130, 640, 100), (40000, 256, 64)])
def test_router_logits(T, H, E):
    """Cases with E not a multiple of 16 (the staged W_r tile has stale rows past E, which must
    not reach a written column), T not a multiple of 128, and more CTAs than SMs."""
    wl = configs.small(T, H, 128, E, 2, backward=False)
    x = synth.make_inputs(wl, 0, device="cuda")["x"]
    w_r = synth.make_router_weight(wl, 0, device="cuda")
    L = ExpertFFN(T, H, 128, E, 2, training=False)
    logits = L.router_forward(x, w_r)
    torch.cuda.synchronize()
    assert_close(logits.cpu().numpy(), ro.router_logits(f64(x), f64(w_r)), "logits")


@pytest.mark.parametrize("renorm", [1, 0])
@pytest.mark.parametrize("T,H,I,E,k", [(256, 128, 256, 4, 2), (600, 256, 384, 16, 4)])
def test_trainable_layer_with_router(T, H, I, E, k, renorm):
    wl = configs.small(T, H, I, E, k, routing="normal", backward=True)
    inp = {kk: v.cuda() for kk, v in synth.make_inputs(wl, 0).items()}
    w_r = synth.make_router_weight(wl, 0, device="cuda")
    L = ExpertFFN(T, H, I, E, k, training=True, renormalize=bool(renorm))
    L.quantize_weights(inp["w_gu"], inp["w_d"])
    logits = L.router_forward(inp["x"], w_r)
    L.forward(logits, inp["x"])
    L.backward(inp["dout"])
    L.router_backward(inp["x"], w_r)
    torch.cuda.synchronize()
    assert L.device_error() == (0, 0)

    x, w_gu, w_d, dout = f64(inp["x"]), f64(inp["w_gu"]), f64(inp["w_d"]), f64(inp["dout"])
    lg = ro.router_logits(x, f64(w_r))
    # float32 sums over H <= 256 products of magnitude <= 0.1 differ from the rounded
    # float64 sums by far less than 5e-6: no top-k decision of these inputs is that close
    s = np.sort(lg, axis=1)[:, ::-1]
    assert (s[:, k - 1] - s[:, k]).min() > 5e-6
    assert_close(logits.cpu().numpy(), lg, "logits")
    idx, prob = rt.route_topk(lg.astype(np.float32), k, renormalize=bool(renorm))
    assert np.array_equal(L.idx.cpu().numpy(), idx)
    fwd = ef.forward(x, idx, prob.astype(np.float64), w_gu, w_d)
    bwd = ef.backward(fwd, dout)
    dl = ro.router_backward(lg, idx, prob, bwd["dprob"], bool(renorm))
    dx_r, dw_r = ro.router_input_grads(dl, x, f64(w_r))
    assert_close(L.dlogits.cpu().numpy(), dl, "dlogits")
    assert_close(L.dw_r.cpu().numpy(), dw_r, "dW_r")
    assert_close(f64(L.dx), ro.add_to_bf16(bwd["dx"], dx_r), "dx (experts + router)")


@pytest.mark.parametrize("renorm", [1, 0])
@pytest.mark.parametrize("T,H,E,k", [(8192, 2048, 64, 6), (4096, 4096, 8, 2), (1000, 384, 256, 8), (70, 128, 4, 2),
                                     (3000, 1280, 100, 4)])
def test_router_backward_direct(T, H, E, k, renorm):
    """moe_router_bwd alone at the fine-grained and Mixtral hidden sizes (and ragged ones):
    logits, routing and dprob are made on the host (seeded), so dlogits, the router's
    dx term and dW_r are compared with the oracle on exactly the device's inputs."""
    wl = configs.small(T, H, 128, E, k, backward=False)
    inp = synth.make_inputs(wl, 0)
    x, logits = inp["x"], inp["logits"]
    w_r = synth.make_router_weight(wl, 0)
    idx, prob = rt.route_topk(logits.numpy(), k, renormalize=bool(renorm))
    dprob = np.random.default_rng(7).normal(0.0, 1e-2, size=(T, k)).astype(np.float32)
    L = ExpertFFN(T, H, 128, E, k, training=True, renormalize=bool(renorm))
    dev = lambda a, dt: torch.as_tensor(np.ascontiguousarray(a)).to(device="cuda", dtype=dt)
    dlogits = torch.empty(T, E, dtype=torch.float32, device="cuda")
    dx = torch.zeros(T, H, dtype=torch.bfloat16, device="cuda")
    dw_r = torch.empty(E, H, dtype=torch.float32, device="cuda")
    B.moe_router_bwd(L.d, x.cuda(), w_r.cuda(), logits.cuda(), dev(idx, torch.int32), dev(prob, torch.float32),
                     dev(dprob, torch.float32), dlogits, dx, dw_r, L.ws)
    torch.cuda.synchronize()
    assert L.device_error() == (0, 0)
    dl = ro.router_backward(logits.numpy(), idx, prob, dprob, bool(renorm))
    dx_r, dw_ref = ro.router_input_grads(dl, f64(x), f64(w_r))
    assert_close(dlogits.cpu().numpy(), dl, "dlogits")
    assert_close(dw_r.cpu().numpy(), dw_ref, "dW_r")
    # dW_r runs on the tensor cores with dl as two bf16 terms (hi + lo, dl to about
    # 2^-17 relative) and f32 accumulation: float32-level accuracy, far inside the bf16
    # level (about 1e-3) that dl rounded once to bf16 would reach
    assert rel_frob(dw_r.cpu().numpy(), dw_ref) < 1e-4
    assert_close(f64(dx), ro.add_to_bf16(np.zeros((T, H)), dx_r), "router dx")
