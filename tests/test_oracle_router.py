"""Pins of the oracle's router: brute-force loops, finite differences, library softmax Jacobian."""
import numpy as np
import pytest
import torch

from oracle import router as ro
from oracle import routing as rt


def test_logits_equal_brute_force_loops():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((5, 7))
    w = rng.standard_normal((3, 7))
    got = ro.router_logits(x, w, rounded=False)
    for t in range(5):
        for e in range(3):
            assert abs(got[t, e] - sum(x[t, h] * w[e, h] for h in range(7))) < 1e-12


def _fd_dlogits(logits, idx, dprob, renormalize, h=1e-6):
    num = np.zeros_like(logits)
    for t in range(logits.shape[0]):
        for e in range(logits.shape[1]):
            lp, lm = logits.copy(), logits.copy()
            lp[t, e] += h
            lm[t, e] -= h
            fp = np.sum(dprob * ro.probs_from_logits(lp, idx, renormalize))
            fm = np.sum(dprob * ro.probs_from_logits(lm, idx, renormalize))
            num[t, e] = (fp - fm) / (2 * h)
    return num


@pytest.mark.parametrize("renormalize", [True, False])
def test_dlogits_match_finite_differences(renormalize):
    rng = np.random.default_rng(1)
    T, E, k = 6, 8, 3
    logits = rng.standard_normal((T, E))
    idx, _ = rt.route_topk(logits.astype(np.float32), k)
    p = ro.probs_from_logits(logits, idx, renormalize)
    dprob = rng.standard_normal((T, k))
    got = ro.router_backward(logits, idx, p, dprob, renormalize)
    assert np.allclose(got, _fd_dlogits(logits, idx, dprob, renormalize), atol=1e-7)


def test_k_equals_E_is_the_softmax_jacobian_of_torch():
    rng = np.random.default_rng(2)
    T, E = 4, 5
    logits = rng.standard_normal((T, E))
    idx, _ = rt.route_topk(logits.astype(np.float32), E)
    p = ro.probs_from_logits(logits, idx, True)
    dprob = rng.standard_normal((T, E))
    got = ro.router_backward(logits, idx, p, dprob, True)
    L = torch.tensor(logits, requires_grad=True)
    s = torch.softmax(L, dim=1)
    g = torch.zeros(T, E, dtype=torch.float64)
    g.scatter_(1, torch.tensor(idx, dtype=torch.int64), torch.tensor(dprob))
    (s * g).sum().backward()
    assert np.allclose(got, L.grad.numpy(), atol=1e-12)


def test_input_gradients_match_finite_differences():
    rng = np.random.default_rng(3)
    T, H, E, k = 4, 6, 5, 2
    x = rng.standard_normal((T, H))
    w = rng.standard_normal((E, H))
    dprob = rng.standard_normal((T, k))
    idx, _ = rt.route_topk(ro.router_logits(x, w).astype(np.float32), k)

    def loss(xx, ww):
        return np.sum(dprob * ro.probs_from_logits(ro.router_logits(xx, ww, rounded=False), idx, True))

    logits = ro.router_logits(x, w, rounded=False)
    dl = ro.router_backward(logits, idx, ro.probs_from_logits(logits, idx, True), dprob, True)
    dx, dw = ro.router_input_grads(dl, x, w)
    h = 1e-6
    for arr, grad in ((x, dx), (w, dw)):
        for i in np.ndindex(arr.shape):
            ap, am = arr.copy(), arr.copy()
            ap[i] += h
            am[i] -= h
            args_p = (ap, w) if arr is x else (x, ap)
            args_m = (am, w) if arr is x else (x, am)
            num = (loss(*args_p) - loss(*args_m)) / (2 * h)
            assert abs(num - grad[i]) < 1e-7


def test_planted_sign_error_in_dlogits_is_caught():
    rng = np.random.default_rng(4)
    logits = rng.standard_normal((4, 6))
    idx, _ = rt.route_topk(logits.astype(np.float32), 2)
    p = ro.probs_from_logits(logits, idx, True)
    dprob = rng.standard_normal((4, 2))
    wrong = np.zeros_like(logits)
    np.put_along_axis(wrong, idx, p * (dprob + np.sum(p * dprob, axis=1, keepdims=True)), axis=1)
    assert not np.allclose(wrong, _fd_dlogits(logits, idx, dprob, True), atol=1e-5)
