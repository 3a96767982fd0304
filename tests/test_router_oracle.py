"""Pins of the router oracle (the routing step in front of the decode layer:
softmax top-k renormalised, and sigmoid top-k normalised times a scale),
against closed forms, ties, invariances and a brute-force full sort."""
import math

import numpy as np
import pytest

import oracle
from mixture_experts_decode_gb300 import inputs


def test_hand_example_softmax():
    # p proportional to (1, 2, 3, 1): the top two are experts 2 and 1, renormalised 3/5 and 2/5
    ids, w = oracle.router_topk(np.array([[0.0, math.log(2), math.log(3), 0.0]], np.float32), 2)
    assert ids.tolist() == [[2, 1]]
    np.testing.assert_allclose(w, [[0.6, 0.4]], rtol=1e-6)


def test_hand_example_sigmoid():
    # sigmoid(0) = 1/2, sigmoid(ln 3) = 3/4: top two 3/4 and 1/2 -> 2.5 * (3/5, 2/5)
    ids, w = oracle.router_topk(np.array([[0.0, -5.0, math.log(3), -1.0]], np.float32), 2, "sigmoid", 2.5)
    assert ids.tolist() == [[2, 0]]
    np.testing.assert_allclose(w, [[1.5, 1.0]], rtol=1e-6)


@pytest.mark.parametrize("score,scale", [("softmax", 1.0), ("sigmoid", 2.5)])
def test_ties_take_lower_expert_first(score, scale):
    E, k = 16, 5
    lg = np.full((3, E), 0.25, np.float32)
    lg[1, 7] = 1.0  # one clear winner, then the tie
    ids, w = oracle.router_topk(lg, k, score, scale)
    assert ids[0].tolist() == [0, 1, 2, 3, 4]
    np.testing.assert_allclose(w[0], scale / k, rtol=1e-12)
    assert ids[1].tolist() == [7, 0, 1, 2, 3]


def _brute(lg, k, score, scale):
    lg = lg.astype(np.float64)
    if score == "softmax":
        e = np.exp(lg - lg.max(axis=1, keepdims=True))
        sc = e / e.sum(axis=1, keepdims=True)
    else:
        sc = 1.0 / (1.0 + np.exp(-lg))
    ids = np.empty((lg.shape[0], k), np.int32)
    w = np.empty((lg.shape[0], k))
    for b in range(lg.shape[0]):
        order = sorted(range(lg.shape[1]), key=lambda e_: (-sc[b, e_], e_))[:k]
        ids[b] = order
        w[b] = scale * sc[b, order] / sc[b, order].sum()
    return ids, w


@pytest.mark.parametrize("kind,E,k,score,scale", [("softmax_uniform", 128, 8, "softmax", 1.0),
                                                  ("sigmoid_scaled", 256, 8, "sigmoid", 2.5),
                                                  ("softmax_normal", 64, 32, "softmax", 1.0)])
def test_matches_full_sort(kind, E, k, score, scale):
    lg = inputs.router_logits(kind, 16, E, "router-pin", E).numpy()
    ids, w = oracle.router_topk(lg, k, score, scale)
    ids2, w2 = _brute(lg, k, score, scale)
    assert np.array_equal(ids, ids2)
    np.testing.assert_allclose(w, w2, rtol=1e-12)
    np.testing.assert_allclose(w.sum(axis=1), scale, rtol=1e-12)
    assert (np.diff(w, axis=1) <= 0).all()  # descending


def test_all_experts_is_the_full_softmax():
    lg = inputs.router_logits("softmax_normal", 4, 12, "router-pin-all").numpy()
    ids, w = oracle.router_topk(lg, 12)
    full = np.exp(lg.astype(np.float64))
    full /= full.sum(axis=1, keepdims=True)
    for b in range(4):
        np.testing.assert_allclose(w[b], full[b, ids[b]], rtol=1e-12)
        assert sorted(ids[b].tolist()) == list(range(12))


def test_softmax_shift_invariance_sigmoid_not():
    lg = inputs.router_logits("softmax_normal", 8, 32, "router-pin-shift").numpy()
    a_ids, a_w = oracle.router_topk(lg, 4)
    b_ids, b_w = oracle.router_topk(lg + np.float32(3.0), 4)
    assert np.array_equal(a_ids, b_ids)
    np.testing.assert_allclose(a_w, b_w, rtol=1e-6)
    c_ids, c_w = oracle.router_topk(lg, 4, "sigmoid", 1.0)
    d_ids, d_w = oracle.router_topk(lg + np.float32(3.0), 4, "sigmoid", 1.0)
    assert np.array_equal(c_ids, d_ids)             # monotone: same choice
    assert np.abs(c_w - d_w).max() > 1e-3           # but not the same weights


def test_rejects_bad_arguments():
    with pytest.raises(ValueError):
        oracle.router_topk(np.zeros((2, 4), np.float32), 5)


def test_selection_follows_the_logits_where_fp64_scores_saturate():
    # sigmoid(40) and sigmoid(41) are both 1.0 in FP64; the exact order (41 first) is kept
    lg = np.array([[40.0, 41.0, -3.0, 0.0]], np.float32)
    ids, w = oracle.router_topk(lg, 2, "sigmoid", 2.5)
    assert ids.tolist() == [[1, 0]]
    np.testing.assert_allclose(w, [[1.25, 1.25]], rtol=1e-12)
