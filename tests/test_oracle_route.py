"""Pins of the oracle's router (softmax -> top-k -> renormalised weights).

Each test checks the oracle against something other than itself: closed forms,
special cases that reduce to a library routine (numpy's stable sort, scipy's
softmax), and invariants of the definition.
"""
import math

import numpy as np
import pytest
from scipy.special import softmax

import oracle
from activation_paging_gb300 import inputs


def test_closed_form_two_of_four():
    # logits ln(1..4): top-2 are experts 3 and 2 with weights 4/7 and 3/7
    l = np.log(np.array([[1.0, 2.0, 3.0, 4.0]])).astype(np.float32)
    idx, w = oracle.route_topk(l, 2)
    assert idx.tolist() == [[3, 2]]
    # exact weights of the rounded logits
    e3, e2 = math.exp(float(l[0, 3])), math.exp(float(l[0, 2]))
    assert abs(w[0, 0] - e3 / (e3 + e2)) <= 2 ** -24
    assert abs(w[0, 1] - e2 / (e3 + e2)) <= 2 ** -24
    assert abs(w[0, 0] - 4 / 7) < 1e-6 and abs(w[0, 1] - 3 / 7) < 1e-6


def test_k_equals_E_is_softmax_and_sort():
    l = inputs.router_logits(3, 64, 16)
    idx, w = oracle.route_topk(l, 16)
    order = np.argsort(-l, axis=1, kind="stable")  # ties keep the lower id
    assert np.array_equal(idx, order)
    p = softmax(l.astype(np.float64), axis=1)
    np.testing.assert_allclose(w, np.take_along_axis(p, order, 1), rtol=2 ** -22, atol=0)


def test_single_expert():
    l = np.array([[0.3], [-7.0]], np.float32)
    idx, w = oracle.route_topk(l, 1)
    assert idx.tolist() == [[0], [0]]
    assert w.tolist() == [[1.0], [1.0]]


def test_ties_go_to_lower_expert():
    l = np.zeros((3, 6), np.float32)
    l[1, 4] = 1.0  # one clear winner, rest tied
    l[2, :] = [0.5, 2.0, 0.5, 2.0, 0.5, 0.5]
    idx, w = oracle.route_topk(l, 3)
    assert idx[0].tolist() == [0, 1, 2]
    assert idx[1].tolist() == [4, 0, 1]
    assert idx[2].tolist() == [1, 3, 0]
    assert np.all(w[0] == np.float32(1 / 3))
    assert w[2, 0] == w[2, 1]


def test_random_against_library_sort():
    for (T, E, k) in [(300, 128, 8), (200, 64, 6), (100, 256, 8), (256, 8, 2)]:
        l = inputs.router_logits(11, T, E)
        idx, w = oracle.route_topk(l, k)
        order = np.argsort(-l, axis=1, kind="stable")[:, :k]
        assert np.array_equal(idx, order)
        # distinct experts per token
        assert all(len(set(r)) == k for r in idx.tolist())
        # weights sum to one and descend with the logits
        assert np.all(np.abs(w.astype(np.float64).sum(1) - 1.0) <= k * 2 ** -23)
        assert np.all(np.diff(w, axis=1) <= 0)
        # ratio of two weights is exp of the logit difference
        li = np.take_along_axis(l, idx, 1).astype(np.float64)
        ratio = w[:, 1].astype(np.float64) / w[:, 0]
        np.testing.assert_allclose(ratio, np.exp(li[:, 1] - li[:, 0]), rtol=2 ** -21)


def test_shift_invariance():
    l = inputs.router_logits(5, 128, 32)
    i1, w1 = oracle.route_topk(l, 4)
    i2, w2 = oracle.route_topk(l + np.float32(16.0), 4)
    # adding 16 (a power of two) keeps the ordering of the rounded logits
    assert np.array_equal(i1, i2)
    np.testing.assert_allclose(w1, w2, rtol=2 ** -16)


def test_zipf_bias_skews_load():
    wl = inputs.WORKLOADS["skewed"]
    from oracle.calibrate_zipf import load_ratio
    r = load_ratio(wl.zipf_beta, wl)
    assert 7.5 <= r <= 8.5
