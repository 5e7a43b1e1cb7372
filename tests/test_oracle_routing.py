"""Pins of the oracle's routing step (top-k of router logits, softmax weights).

The golden reference MoE of TensorRT-LLM PR #17865 starts from router logits
(`routing_method.apply(router_logits)`); the pages name no routing method,
and the reading taken is the one the workloads' routing weights follow: the
K largest logits (descending, ties to the lower expert ID) with a softmax
over them, or, without renormalisation, their probabilities under a softmax
over all experts.  Pinned here against numpy's stable argsort, scipy's
softmax, closed forms and invariants.
"""
import numpy as np
import pytest
from scipy.special import softmax

import oracle


def _rng(seed):
    return np.random.default_rng(seed)


@pytest.mark.parametrize("T,E,K", [(1, 1, 1), (7, 8, 8), (33, 896, 16), (5, 100, 7), (64, 37, 16)])
def test_ids_are_the_stable_descending_order(T, E, K):
    # integer-valued logits from a small set: many ties, broken by the lower ID
    l = _rng(T * E + K).integers(-3, 4, (T, E)).astype(np.float32)
    ids, _ = oracle.route_topk(l, K)
    ref = np.argsort(-l, axis=1, kind="stable")[:, :K]
    assert np.array_equal(ids, ref)


def test_signed_zero_ties_and_large_logits():
    l = np.array([[0.0, -0.0, 0.0, -1.0], [1e30, -1e30, 1e30, 3e38]], np.float32)
    ids, w = oracle.route_topk(l, 3)
    assert ids[0].tolist() == [0, 1, 2]          # +0 and -0 are equal: lower IDs first
    assert ids[1].tolist() == [3, 0, 2]
    # the max is subtracted first: no overflow at 3e38
    assert np.all(np.isfinite(w))
    assert w[1, 0] == 1.0 and w[1, 1] == 0.0 and w[1, 2] == 0.0
    np.testing.assert_array_equal(w[0], np.float32(1.0 / 3.0))


@pytest.mark.parametrize("renormalize", [True, False])
def test_weights_match_scipy_softmax(renormalize):
    rng = _rng(3)
    T, E, K = 50, 896, 16
    l = (rng.standard_normal((T, E)) * 2.0).astype(np.float32)
    ids, w = oracle.route_topk(l, K, renormalize=renormalize)
    sel = np.take_along_axis(l.astype(np.float64), ids, axis=1)
    if renormalize:
        ref = softmax(sel, axis=1)
    else:
        ref = np.take_along_axis(softmax(l.astype(np.float64), axis=1), ids, axis=1)
    # one rounding to fp32 of (nearly) the same fp64 value
    np.testing.assert_allclose(w, ref, rtol=2.0 ** -23, atol=0)
    if renormalize:
        assert np.all(np.abs(w.astype(np.float64).sum(1) - 1.0) < K * 2.0 ** -24)
    else:
        assert np.all(w.astype(np.float64).sum(1) < 1.0 + K * 2.0 ** -24)
    # descending logits give non-increasing weights
    assert np.all(np.diff(w, axis=1) <= 0)


def test_two_experts_closed_form():
    # K = 2: the weights are sigmoid(+-d), d the logit gap
    d = np.linspace(-20, 20, 41, dtype=np.float32)
    l = np.stack([d, np.zeros_like(d)], axis=1)
    ids, w = oracle.route_topk(l, 2)
    hi = np.maximum(d, 0).astype(np.float64)
    gap = np.abs(d).astype(np.float64)
    np.testing.assert_allclose(w[:, 0], 1.0 / (1.0 + np.exp(-gap)), rtol=2.0 ** -23)
    np.testing.assert_allclose(w[:, 1], 1.0 / (1.0 + np.exp(gap)), rtol=2.0 ** -23)
    assert np.all(np.take_along_axis(l, ids, 1)[:, 0] == hi.astype(np.float32))


def test_single_expert_and_all_selected():
    l = _rng(5).standard_normal((9, 12)).astype(np.float32)
    ids, w = oracle.route_topk(l, 1)
    assert np.array_equal(ids[:, 0], np.argmax(l, axis=1))
    assert np.all(w == 1.0)
    ids, w = oracle.route_topk(l, 12)
    # every expert selected: renormalised weights are the full softmax
    np.testing.assert_allclose(w, np.take_along_axis(softmax(l.astype(np.float64), axis=1), ids, 1),
                               rtol=2.0 ** -23)
    _, w0 = oracle.route_topk(l, 12, renormalize=False)
    np.testing.assert_array_equal(w, w0)


def test_bad_sizes():
    with pytest.raises(ValueError):
        oracle.route_topk(np.zeros((2, 4), np.float32), 5)
    with pytest.raises(ValueError):
        oracle.route_topk(np.zeros((2, 4), np.float32), 0)
