"""Pins for the routing oracle (softmax -> top-k), CPU only.

Ties ``oracle.routing`` to torch's float64 softmax and topk (library
routines), to k = E (the full sorted softmax, weights summing to one), to
constructed ties (lower expert index first), to E = 2, k = 1 (argmax), and to
brute force over every subset on tiny rows.
"""

import itertools
import math

import numpy as np
import pytest
import torch

from oracle import routing as Rt


def test_softmax_matches_torch():
    rng = np.random.default_rng(0)
    x = (rng.standard_normal((64, 256)) * 2).astype(np.float32)
    p = Rt.softmax(x)
    ref = torch.softmax(torch.from_numpy(x).double(), dim=1).numpy()
    np.testing.assert_allclose(p, ref, rtol=1e-13, atol=1e-300)


@pytest.mark.parametrize("E,k", [(256, 8), (64, 2), (33, 5), (8, 8)])
def test_topk_matches_torch_on_distinct_logits(E, k):
    rng = np.random.default_rng(E + k)
    x = (rng.standard_normal((200, E)) * 2).astype(np.float32)
    idx, w = Rt.softmax_topk(x, k, renormalize=False)
    p = torch.softmax(torch.from_numpy(x).double(), dim=1)
    tv, ti = torch.topk(p, k, dim=1, largest=True, sorted=True)
    np.testing.assert_array_equal(idx, ti.numpy())
    np.testing.assert_allclose(w, tv.numpy(), rtol=1e-14)
    idx2, w2 = Rt.softmax_topk(x, k, renormalize=True)
    np.testing.assert_array_equal(idx2, idx)
    np.testing.assert_allclose(w2, tv.numpy() / tv.numpy().sum(1, keepdims=True), rtol=1e-13)


def test_k_equals_e_is_full_sorted_softmax():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((10, 16)).astype(np.float32)
    idx, w = Rt.softmax_topk(x, 16, renormalize=True)
    np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=1e-14)
    for t in range(10):
        assert sorted(idx[t].tolist()) == list(range(16))
        assert np.all(np.diff(x[t, idx[t]]) <= 0)


def test_ties_go_to_lower_index():
    x = np.array([[1.0, 3.0, 3.0, 0.5, 3.0, -1.0],
                  [0.0, 0.0, 0.0, 0.0, 0.0, 0.0],
                  [2.0, -5.0, 2.0, 2.0, 7.0, 7.0]], dtype=np.float32)
    idx, w = Rt.softmax_topk(x, 4, renormalize=True)
    assert idx[0].tolist() == [1, 2, 4, 0]
    assert idx[1].tolist() == [0, 1, 2, 3]
    assert idx[2].tolist() == [4, 5, 0, 2]
    np.testing.assert_allclose(w[1], 0.25, rtol=1e-15)


def test_two_experts_top1_is_argmax():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((500, 2)).astype(np.float32)
    idx, w = Rt.softmax_topk(x, 1, renormalize=False)
    np.testing.assert_array_equal(idx[:, 0], np.argmax(x, axis=1))
    # the weight of the winner of two is the logistic of the logit gap
    gap = np.abs(x[:, 0].astype(np.float64) - x[:, 1])
    np.testing.assert_allclose(w[:, 0], 1.0 / (1.0 + np.exp(-gap)), rtol=1e-14)
    _, wr = Rt.softmax_topk(x, 1, renormalize=True)
    assert np.all(wr == 1.0)


@pytest.mark.parametrize("E", [2, 3, 5, 8])
def test_brute_force_subsets(E):
    rng = np.random.default_rng(20 + E)
    x = rng.standard_normal((12, E)).astype(np.float32)
    for k in range(1, E + 1):
        idx, w = Rt.softmax_topk(x, k, renormalize=True)
        for t in range(x.shape[0]):
            row = [float(v) for v in x[t]]
            # the best subset of size k maximises the summed logits (all
            # logits are distinct here), then sort it by (-logit, index)
            best = max(itertools.combinations(range(E), k), key=lambda c: sum(row[i] for i in c))
            best = sorted(best, key=lambda i: (-row[i], i))
            assert idx[t].tolist() == best
            z = sum(math.exp(row[i]) for i in best)
            np.testing.assert_allclose(w[t], [math.exp(row[i]) / z for i in best], rtol=1e-13)


def test_order_beyond_exp_underflow():
    # exp(x - m) is 0 in float64 for all three losers; they must still be
    # listed by logit, not by expert index
    x = np.array([[10.0, -900.0, -800.0, -1000.0]], dtype=np.float32)
    idx, w = Rt.softmax_topk(x, 3, renormalize=True)
    assert idx[0].tolist() == [0, 2, 1]
    assert w[0].tolist() == [1.0, 0.0, 0.0]
    idx, _ = Rt.softmax_topk(x, 4, renormalize=False)
    assert idx[0].tolist() == [0, 2, 1, 3]


def test_order_where_probabilities_are_equal_subnormals():
    # gaps near 744: exp rounds the two probabilities to the same subnormal
    # double, yet the logits differ
    x = np.array([[0.0, -744.25, -744.0, 5.0]], dtype=np.float32)
    m = 5.0
    assert np.exp(np.float64(x[0, 1]) - m) == np.exp(np.float64(x[0, 2]) - m)
    idx, _ = Rt.softmax_topk(x, 4, renormalize=False)
    assert idx[0].tolist() == [3, 0, 2, 1]


def test_masked_experts_with_ties():
    # masked experts at large finite negatives, mixed with exact ties
    x = np.array([[-1e4, 3.0, -1e4, 3.0, -3e38, -1e4, 2.0, -3e38]], dtype=np.float32)
    idx, w = Rt.softmax_topk(x, 7, renormalize=True)
    assert idx[0].tolist() == [1, 3, 6, 0, 2, 5, 4]
    z = 2 * math.exp(0.0) + math.exp(-1.0)
    np.testing.assert_allclose(w[0, :3], [1 / z, 1 / z, math.exp(-1.0) / z], rtol=1e-15)
    assert np.all(w[0, 3:] == 0.0)


@pytest.mark.parametrize("E", [3, 5, 8])
def test_brute_force_subsets_with_wide_gaps(E):
    # logits spread over +-2e4, far beyond exp's range: the best subset of
    # size k maximises the summed logits whatever the probabilities underflow to
    rng = np.random.default_rng(40 + E)
    x = (rng.standard_normal((12, E)) * 1e4).astype(np.float32)
    for k in range(1, E + 1):
        idx, _ = Rt.softmax_topk(x, k, renormalize=False)
        for t in range(x.shape[0]):
            row = [float(v) for v in x[t]]
            best = max(itertools.combinations(range(E), k), key=lambda c: sum(row[i] for i in c))
            assert idx[t].tolist() == sorted(best, key=lambda i: (-row[i], i))
