"""Pins of the oracle's top-k routing against brute force and closed forms."""
import math

import numpy as np
import pytest

from oracle import moe_ref as ref


def brute_topk(logits, k):
    """Pure-Python top-k: sort expert ids by (-logit, id); gates by math.exp."""
    T, E = len(logits), len(logits[0])
    idx, w = [], []
    for t in range(T):
        row = [float(v) for v in logits[t]]
        chosen = sorted(range(E), key=lambda e: (-row[e], e))[:k]
        m = max(row[e] for e in chosen)
        z = [math.exp(row[e] - m) for e in chosen]
        s = sum(z)
        idx.append(chosen)
        w.append([v / s for v in z])
    return np.array(idx), np.array(w)


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("E,k", [(1, 1), (4, 2), (8, 2), (5, 5), (16, 3), (64, 6)])
def test_topk_matches_bruteforce_with_ties(seed, E, k):
    rng = np.random.default_rng(seed)
    T = 37
    # integer-valued logits force many exact ties
    logits = rng.integers(-2, 3, size=(T, E)).astype(np.float32)
    if seed % 2:
        logits = logits + rng.standard_normal((T, E)).astype(np.float32) * np.float32(seed > 2)
    idx, w = ref.route_topk(logits, k)
    bidx, bw = brute_topk(logits.tolist(), k)
    assert idx.dtype == np.int32
    np.testing.assert_array_equal(idx, bidx)
    np.testing.assert_allclose(w, bw, rtol=0, atol=1e-15)


def test_all_equal_logits_pick_lowest_ids():
    logits = np.zeros((5, 8), np.float32)
    idx, w = ref.route_topk(logits, 3)
    np.testing.assert_array_equal(idx, np.tile([0, 1, 2], (5, 1)))
    np.testing.assert_allclose(w, 1 / 3, atol=1e-15)


def test_negative_zero_ties_positive_zero():
    logits = np.array([[-0.0, 0.0, -1.0]], np.float32)
    idx, _ = ref.route_topk(logits, 2)
    np.testing.assert_array_equal(idx, [[0, 1]])


def test_gates_sum_to_one_and_descend():
    rng = np.random.default_rng(3)
    logits = rng.standard_normal((200, 16)).astype(np.float32) * 4
    idx, w = ref.route_topk(logits, 5)
    np.testing.assert_allclose(w.sum(1), 1.0, atol=1e-12)
    chosen = np.take_along_axis(logits, idx.astype(np.int64), 1)
    assert np.all(np.diff(chosen, axis=1) <= 0)
    assert np.all(np.diff(w, axis=1) <= 0)
    for t in range(200):
        assert len(set(idx[t].tolist())) == 5


def test_k1_gate_is_one():
    rng = np.random.default_rng(4)
    logits = rng.standard_normal((50, 7)).astype(np.float32)
    idx, w = ref.route_topk(logits, 1)
    assert np.all(w == 1.0)
    np.testing.assert_array_equal(idx[:, 0], np.argmax(logits, 1))


def test_two_gate_closed_form():
    # k = 2: w0 = 1 / (1 + exp(l1 - l0)), the logistic of the logit gap
    rng = np.random.default_rng(5)
    logits = rng.standard_normal((100, 6)).astype(np.float32) * 3
    idx, w = ref.route_topk(logits, 2)
    l = logits.astype(np.float64)
    for t in range(100):
        a, b = l[t, idx[t, 0]], l[t, idx[t, 1]]
        assert abs(w[t, 0] - 1.0 / (1.0 + math.exp(b - a))) < 1e-15


def test_k_equals_E_is_full_softmax():
    rng = np.random.default_rng(6)
    logits = rng.standard_normal((20, 6)).astype(np.float32)
    idx, w = ref.route_topk(logits, 6)
    full = np.exp(logits.astype(np.float64))
    full /= full.sum(1, keepdims=True)
    np.testing.assert_allclose(w, np.take_along_axis(full, idx.astype(np.int64), 1), rtol=1e-13)


def test_logits_are_compared_as_float32():
    # two float64 values that collapse to the same float32 must tie
    a = np.float64(1.0) + 2.0 ** -30
    logits = np.array([[1.0, a]], dtype=np.float64)
    idx, _ = ref.route_topk(logits, 1)
    assert idx[0, 0] == 0
