"""Pins of the oracle's routing and permutation: brute force, closed forms, invariants."""
import numpy as np
import pytest
import scipy.special

from oracle import routing as rt


def brute_topk(logits, k):
    out = []
    for row in logits:
        order = sorted(range(len(row)), key=lambda e: (-float(row[e]), e))
        out.append(order[:k])
    return np.array(out)


@pytest.mark.parametrize("T,E,k", [(37, 8, 2), (50, 64, 6), (9, 5, 5), (16, 256, 8)])
def test_topk_matches_brute_force_sort(T, E, k):
    rng = np.random.default_rng(T * E + k)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    # plant exact ties
    logits[0, 3] = logits[0, 1]
    logits[1, :] = 0.5
    idx, prob = rt.route_topk(logits, k)
    assert np.array_equal(idx, brute_topk(logits, k))
    assert np.allclose(prob.sum(axis=1), 1.0, atol=1e-6)
    assert np.all(np.diff(prob, axis=1) <= 0)               # slots in descending order
    assert list(idx[1]) == list(range(k))                    # all tied -> lowest indices


def brute_topk_total_order(row, k):
    """Pairwise comparison sort written out: a beats b when b is NaN and a is not, or
    both are numbers and a > b, or they tie (both NaN, or equal numbers) and a has the
    lower index."""
    E = len(row)

    def beats(a, b):
        na, nb = np.isnan(row[a]), np.isnan(row[b])
        if na != nb:
            return nb
        if not na and row[a] != row[b]:
            return row[a] > row[b]
        return a < b

    chosen = []
    rest = list(range(E))
    for _ in range(k):
        best = rest[0]
        for c in rest[1:]:
            if beats(c, best):
                best = c
        chosen.append(best)
        rest.remove(best)
    return chosen


@pytest.mark.filterwarnings("ignore:invalid value encountered")
def test_nan_logits_rank_last_and_the_row_still_fills():
    nan, inf = np.float32(np.nan), np.float32(np.inf)
    logits = np.array([
        [nan, 1.0, nan, -2.0, 0.5, nan],          # fewer numbers (3) than k (4): one NaN expert joins
        [nan, nan, nan, nan, nan, nan],           # all NaN: the lowest ids
        [-inf, nan, -inf, 3.0, nan, -1.0],        # -inf still beats NaN
        [0.0, -0.0, 0.0, -0.0, -1.0, nan],        # signed zeros tie: index order
        [inf, 1.0, inf, nan, -inf, 2.0],
    ], dtype=np.float32)
    k = 4
    idx, prob = rt.route_topk(logits, k)
    for t in range(len(logits)):
        assert list(idx[t]) == brute_topk_total_order(logits[t], k), t
        assert len(set(idx[t])) == k
    assert list(idx[0]) == [1, 4, 3, 0] and np.all(np.isnan(prob[0]))
    assert list(idx[1]) == [0, 1, 2, 3]
    assert list(idx[2]) == [3, 5, 0, 2]                      # -inf beats NaN; exp(-inf - 3) = 0
    assert np.allclose(prob[2], [1 / (1 + np.exp(-4.0)), 1 - 1 / (1 + np.exp(-4.0)), 0, 0], rtol=1e-6)
    assert list(idx[3]) == [0, 1, 2, 3]
    assert np.allclose(prob[3], 0.25)


def test_k_equals_E_is_plain_softmax():
    rng = np.random.default_rng(7)
    logits = rng.standard_normal((20, 6)).astype(np.float32)
    idx, prob = rt.route_topk(logits, 6)
    ref = scipy.special.softmax(logits.astype(np.float64), axis=1)
    got = np.zeros_like(ref)
    np.put_along_axis(got, idx.astype(np.int64), prob.astype(np.float64), axis=1)
    assert np.allclose(got, ref, rtol=1e-6, atol=1e-7)


def test_unrenormalized_probs_are_softmax_entries():
    rng = np.random.default_rng(8)
    logits = rng.standard_normal((30, 16)).astype(np.float32)
    idx, prob = rt.route_topk(logits, 4, renormalize=False)
    ref = scipy.special.softmax(logits.astype(np.float64), axis=1)
    assert np.allclose(prob, np.take_along_axis(ref, idx.astype(np.int64), axis=1), rtol=1e-6)
    # renormalising them gives the default probabilities
    idx2, prob2 = rt.route_topk(logits, 4)
    assert np.allclose(prob2, prob / prob.sum(axis=1, keepdims=True), rtol=1e-6)


def brute_permutation(idx, E):
    """Direct counting: walk experts, then tokens in order."""
    T, k = idx.shape
    split = [0] * E
    for t in range(T):
        for j in range(k):
            split[idx[t, j]] += 1
    offs = [0]
    for e in range(E):
        offs.append(offs[-1] + (split[e] + 127) // 128 * 128)
    row_of = np.full((T, k), -1)
    for e in range(E):
        r = offs[e]
        for t in range(T):
            for j in range(k):
                if idx[t, j] == e:
                    row_of[t, j] = r
                    r += 1
    return np.array(split), np.array(offs), row_of


@pytest.mark.parametrize("T,E,k,routing", [(300, 8, 2, "normal"), (200, 16, 4, "skew"), (64, 4, 1, "normal")])
def test_permutation_invariants(T, E, k, routing):
    rng = np.random.default_rng(T + E)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    if routing == "skew":
        logits[:, 0] += 3.0
        logits[:, 5] -= 100.0          # expert 5 empty
    idx, _ = rt.route_topk(logits, k)
    p = rt.permute(idx, E)
    split, offs, row_of = brute_permutation(idx, E)
    assert np.array_equal(p["split_sizes"], split)
    assert p["split_sizes"].sum() == T * k
    assert np.array_equal(p["offsets_pad"], offs)
    assert np.array_equal(p["row_of"], row_of)
    assert np.all(p["offsets_pad"] % 128 == 0)
    # bijection between (t, j) pairs and non-padding rows
    flat = p["row_of"].ravel()
    assert len(np.unique(flat)) == T * k
    src = p["src_of"]
    assert np.array_equal(src[flat], np.repeat(np.arange(T), k))
    assert np.count_nonzero(src < 0) == p["rows"] - T * k
    # expert-major, ascending token inside each segment
    for e in range(E):
        seg = src[offs[e]:offs[e] + split[e]]
        assert np.all(np.diff(seg) > 0)
        assert np.all(src[offs[e] + split[e]:offs[e + 1]] == -1)
    if routing == "skew":
        assert p["split_sizes"][5] == 0
