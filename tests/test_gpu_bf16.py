"""BF16 grouped forward (no quantization) vs the oracle with the bf16-activation numerics."""
import numpy as np
import pytest
import torch

from helpers import assert_close
from moe_expert_ffn_03_gb300 import build, configs, synth
from moe_expert_ffn_03_gb300.layer import ExpertFFN
from oracle import expert_ffn as ef
from oracle import routing as rt

pytestmark = [pytest.mark.gpu, pytest.mark.filterwarnings("error::RuntimeWarning")]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()


def f64(t):
    return t.float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("name_or_dims", [
    configs.TINY,
    (300, 256, 384, 6, 2, "biased"),
    (513, 384, 640, 5, 3, "normal"),
    configs.UNEVEN,
])
def test_bf16_forward_matches_oracle(name_or_dims):
    wl = configs.get(name_or_dims) if isinstance(name_or_dims, str) else configs.small(*name_or_dims[:5],
                                                                                         routing=name_or_dims[5])
    inp = {k: v.cuda() for k, v in synth.make_inputs(wl, 0, with_grad=False).items()}
    L = ExpertFFN(wl.T, wl.H, wl.I, wl.E, wl.k, training=False)
    L.route(inp["logits"], inp["x"])
    out = L.forward_bf16(inp["x"], inp["w_gu"], inp["w_d"])
    torch.cuda.synchronize()
    assert L.device_error() == (0, 0)
    idx, prob = rt.route_topk(inp["logits"].cpu().numpy(), wl.k)
    fwd = ef.forward(f64(inp["x"]), idx, prob.astype(np.float64), f64(inp["w_gu"]), f64(inp["w_d"]), ef.BF16_PATH)
    rows = fwd["perm"]["rows"]
    assert np.array_equal(f64(L.x_perm[:rows]), fwd["x_perm"])
    assert_close(f64(L.a_perm[:rows]), ef.q_rowwise(fwd["a"], ef.BF16_PATH), "a (bf16)")
    assert_close(f64(L.y_b16[:rows]), fwd["y"], "y")
    assert_close(f64(out), fwd["out"], "out")


@pytest.mark.parametrize("name_or_dims", [
    configs.TINY,
    (300, 256, 384, 6, 2, "biased"),
    (513, 384, 640, 5, 3, "normal"),
    (600, 128, 128, 256, 8, "biased"),
])
def test_bf16_training_step_matches_oracle(name_or_dims):
    """bf16 forward (saving g, u) + bf16 backward vs the oracle's BF16-path backward."""
    wl = configs.get(name_or_dims) if isinstance(name_or_dims, str) else configs.small(*name_or_dims[:5],
                                                                                         routing=name_or_dims[5])
    inp = {k: v.cuda() for k, v in synth.make_inputs(wl, 0, with_grad=True).items()}
    L = ExpertFFN(wl.T, wl.H, wl.I, wl.E, wl.k, training=True, bf16_training=True)
    L.route(inp["logits"], inp["x"])
    L.forward_bf16(inp["x"], inp["w_gu"], inp["w_d"])
    L.transpose_weights_bf16(inp["w_gu"], inp["w_d"])
    dx = L.backward_bf16(inp["dout"])
    torch.cuda.synchronize()
    assert L.device_error() == (0, 0)
    idx, prob = rt.route_topk(inp["logits"].cpu().numpy(), wl.k)
    fwd = ef.forward(f64(inp["x"]), idx, prob.astype(np.float64), f64(inp["w_gu"]), f64(inp["w_d"]), ef.BF16_PATH)
    bwd = ef.backward(fwd, f64(inp["dout"]), ef.BF16_PATH)
    rows = fwd["perm"]["rows"]
    I = wl.I
    assert_close(f64(L.saved_gu[:rows, :I]), fwd["g"], "g")
    assert_close(f64(L.saved_gu[:rows, I:]), fwd["u"], "u")
    assert_close(f64(dx), bwd["dx"], "dx")
    assert_close(f64(L.dwgu16), bwd["dw_gu"], "dW_gu")
    assert_close(f64(L.dwd16), bwd["dw_d"], "dW_d")
    assert_close(L.dprob16.cpu().numpy().astype(np.float64), bwd["dprob"], "dprob")


def test_transpose_bf16_is_exact():
    g = torch.Generator().manual_seed(5)
    w = torch.randn(3, 256, 384, generator=g).to(torch.bfloat16).cuda()
    out = torch.empty(3, 384, 256, dtype=torch.bfloat16, device="cuda")
    from moe_expert_ffn_03_gb300 import binding as B
    B.moe_transpose_bf16(w, 3, 256, 384, out)
    torch.cuda.synchronize()
    assert torch.equal(out, w.transpose(1, 2))


@pytest.mark.parametrize("dims", [(500, 256, 384, 6, 2, "biased"), (300, 128, 256, 64, 6, "biased"),
                                  (200, 384, 128, 3, 2, "normal")])
def test_bf16_per_expert_weight_tensors_equal_stacked(dims):
    """One weight tensor per expert (the pages' weight0, weight1, ...): the forward reads each
    expert's own tensor through its own TMA descriptor, the transposes read one pointer per
    expert; the training step is bit-identical to the stacked weights'."""
    wl = configs.small(*dims[:5], routing=dims[5])
    inp = {k: v.cuda() for k, v in synth.make_inputs(wl, 0, with_grad=True).items()}
    res = []
    for as_list in (False, True):
        L = ExpertFFN(wl.T, wl.H, wl.I, wl.E, wl.k, training=True, bf16_training=True)
        w_gu = [w.clone() for w in inp["w_gu"]] if as_list else inp["w_gu"]
        w_d = [w.clone() for w in inp["w_d"]] if as_list else inp["w_d"]
        L.route(inp["logits"], inp["x"])
        L.forward_bf16(inp["x"], w_gu, w_d)
        L.transpose_weights_bf16(w_gu, w_d)
        L.backward_bf16(inp["dout"])
        torch.cuda.synchronize()
        assert L.device_error() == (0, 0)
        rows = L.padded_rows()                                    # a_perm rows past the segments are unwritten
        res.append([t.clone() for t in (L.out_b16, L.a_perm[:rows], L.dx16, L.dwgu16, L.dwd16, L.dprob16, L.wguT16,
                                        L.wdT16)])
    for a, b in zip(*res):
        assert torch.equal(a, b)


def test_bf16_per_expert_host_checks():
    from moe_expert_ffn_03_gb300 import binding as B
    wl = configs.small(64, 128, 128, 129, 2)                       # E above the per-expert map limit
    L = ExpertFFN(wl.T, wl.H, wl.I, wl.E, wl.k, training=False)
    w = [torch.zeros(256, 128, dtype=torch.bfloat16, device="cuda")] * wl.E
    with pytest.raises(B.MoeError):
        B.grouped_mlp_fwd_bf16_experts(L.d, L.xq, L.split_sizes, L.prob_perm, w, w, L.y, L.y, L.ws)
