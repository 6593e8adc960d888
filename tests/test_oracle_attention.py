"""Pins for the attention oracle (CPU only).

Each test ties ``oracle.attention`` to something other than itself: the
worked example spoken in the RedFuser episode transcript (cue 15), closed
forms, the merge invariant and identity element (transcript cues 21, 27, 29,
39), brute force on tiny inputs, and torch's float64
scaled-dot-product attention (a library routine).
"""

import math
import os

import numpy as np
import pytest
import torch

from oracle import attention as A

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_example.txt")


def _golden():
    vals = {}
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *rest = line.split()
            vals[key] = [float(r) for r in rest]
    return vals


def _worked_example_inputs(D=64):
    g = _golden()
    scores = g["scores_tile_a"] + g["scores_tile_b"]
    L = len(scores)
    q = np.zeros(D)
    q[0] = 1.0
    K = np.zeros((L, D))
    K[:, 0] = scores
    V = np.zeros((L, D))
    V[:, 0] = g["v"]
    return q, K, V, g


def test_worked_example_printed_values():
    q, K, V, g = _worked_example_inputs()
    m, l, acc = A.segment_states(q[None], K[None], V[None], 1.0, 2)
    # tile A = keys {0, 1} (scores 1, 3), tile B = key {2} (score 5)
    assert m[0, 0] == 3.0 and m[0, 1] == 5.0
    corr = math.exp(m[0, 0] - m[0, 1])
    assert round(corr, 2) == g["printed_correction"][0]
    assert round(l[0, 0], 2) == g["printed_l_tile_a"][0]
    _, lse = A.merge_states(m, l, acc)
    l_total = math.exp(lse[0] - 5.0)
    assert round(l_total, 2) == g["printed_l_total"][0]


def test_worked_example_closed_forms():
    q, K, V, _ = _worked_example_inputs()
    m, l, acc = A.segment_states(q[None], K[None], V[None], 1.0, 2)
    e2, e4 = math.exp(-2.0), math.exp(-4.0)
    # tile A relative to its own max 3: l = e^-2 + 1, acc = 2 e^-2 - 1
    assert l[0, 0] == pytest.approx(e2 + 1.0, rel=1e-15)
    assert acc[0, 0, 0] == pytest.approx(2 * e2 - 1.0, rel=1e-14)
    # tile B relative to 5: l = 1, acc = 4
    assert l[0, 1] == 1.0 and acc[0, 1, 0] == 4.0
    # the incremental denominator equals the from-scratch one
    assert l[0, 0] * e2 + 1.0 == pytest.approx(e4 + e2 + 1.0, rel=1e-15)
    out, mm, ll = A.softmax_v(q, K, V, 1.0)
    assert mm == 5.0
    assert ll == pytest.approx(e4 + e2 + 1.0, rel=1e-15)
    expect = (2 * e4 - e2 + 4.0) / (e4 + e2 + 1.0)
    assert out[0] == pytest.approx(expect, rel=1e-15)
    assert np.all(out[1:] == 0.0)
    mo, lse = A.merge_states(m, l, acc)
    assert mo[0, 0] == pytest.approx(expect, rel=1e-15)
    assert lse[0] == pytest.approx(5.0 + math.log(e4 + e2 + 1.0), rel=1e-15)


def test_closed_form_constant_values():
    rng = np.random.default_rng(0)
    L, D = 37, 16
    q = rng.standard_normal(D)
    K = rng.standard_normal((L, D))
    row = rng.standard_normal(D)
    V = np.tile(row, (L, 1))
    out, _, _ = A.softmax_v(q, K, V, 0.3)
    np.testing.assert_allclose(out, row, rtol=1e-13, atol=1e-14)


def test_closed_form_equal_scores_give_mean():
    rng = np.random.default_rng(1)
    L, D = 29, 8
    K = rng.standard_normal((L, D))
    V = rng.standard_normal((L, D))
    out, m, l = A.softmax_v(np.zeros(D), K, V, 1.0)
    assert m == 0.0 and l == L
    np.testing.assert_allclose(out, V.mean(axis=0), rtol=1e-13, atol=1e-15)


def test_closed_form_dominant_key():
    rng = np.random.default_rng(2)
    L, D = 20, 8
    K = rng.standard_normal((L, D)) * 0.01
    q = np.zeros(D)
    q[3] = 1.0
    K[7, 3] = 1000.0
    V = rng.standard_normal((L, D))
    out, _, _ = A.softmax_v(q, K, V, 1.0)
    np.testing.assert_allclose(out, V[7], rtol=0, atol=1e-12)


def _brute(q, K, V, scale):
    L, D = len(K), len(q)
    s = [scale * sum(q[d] * K[j][d] for d in range(D)) for j in range(L)]
    mx = max(s)
    w = [math.exp(x - mx) for x in s]
    tot = sum(w)
    return [sum(w[j] * V[j][d] for j in range(L)) / tot for d in range(len(V[0]))]


@pytest.mark.parametrize("L", [1, 2, 3, 5, 8])
def test_brute_force_tiny(L):
    rng = np.random.default_rng(10 + L)
    D = 4
    q = rng.standard_normal(D)
    K = rng.standard_normal((L, D))
    V = rng.standard_normal((L, D))
    out, _, _ = A.softmax_v(q, K, V, 0.7)
    np.testing.assert_allclose(out, _brute(q.tolist(), K.tolist(), V.tolist(), 0.7), rtol=1e-13)


@pytest.mark.parametrize("S", [1, 2, 3, 4, 7, 16, 40, 64])
def test_merge_of_any_split_equals_single_pass(S):
    rng = np.random.default_rng(100 + S)
    R, L, D = 3, 40, 8
    q = rng.standard_normal((R, D))
    K = rng.standard_normal((R, L, D)) * 2
    V = rng.standard_normal((R, L, D))
    m, l, acc = A.segment_states(q, K, V, 0.5, S)
    out, lse = A.merge_states(m, l, acc)
    ref, mref, lref = A.softmax_v_rows(q, K, V, 0.5)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(lse, mref + np.log(lref), rtol=1e-13)
    if S > L:
        # segments past the end carry the identity state
        assert np.all(np.isneginf(m[:, L:])) and np.all(l[:, L:] == 0) and np.all(acc[:, L:] == 0)


def test_identity_state_is_neutral_and_merge_order_free():
    rng = np.random.default_rng(7)
    R, S, D = 4, 5, 6
    m = rng.standard_normal((R, S)) * 3
    l = rng.uniform(0.5, 3.0, (R, S))
    acc = rng.standard_normal((R, S, D))
    out, lse = A.merge_states(m, l, acc)
    # add identity states anywhere
    m2 = np.concatenate([np.full((R, 2), -np.inf), m, np.full((R, 1), -np.inf)], axis=1)
    l2 = np.concatenate([np.zeros((R, 2)), l, np.zeros((R, 1))], axis=1)
    acc2 = np.concatenate([np.zeros((R, 2, D)), acc, np.zeros((R, 1, D))], axis=1)
    out2, lse2 = A.merge_states(m2, l2, acc2)
    np.testing.assert_allclose(out2, out, rtol=1e-14)
    np.testing.assert_allclose(lse2, lse, rtol=1e-14)
    perm = rng.permutation(S)
    out3, lse3 = A.merge_states(m[:, perm], l[:, perm], acc[:, perm])
    np.testing.assert_allclose(out3, out, rtol=1e-13)
    # grouping: merge two halves first, then merge the two results
    a_out, a_lse = A.merge_states(m[:, :2], l[:, :2], acc[:, :2])
    b_out, b_lse = A.merge_states(m[:, 2:], l[:, 2:], acc[:, 2:])
    # a merged state (out, lse) is the state (m=lse, l=1, acc=out)
    mm = np.stack([a_lse, b_lse], axis=1)
    ll = np.ones_like(mm)
    aa = np.stack([a_out, b_out], axis=1)
    out4, lse4 = A.merge_states(mm, ll, aa)
    np.testing.assert_allclose(out4, out, rtol=1e-13)
    np.testing.assert_allclose(lse4, lse, rtol=1e-13)


@pytest.mark.parametrize("causal", [True, False])
def test_prefill_against_torch_sdpa(causal):
    rng = np.random.default_rng(11)
    N, D = 50, 16
    Q = rng.standard_normal((N, D))
    K = rng.standard_normal((N, D))
    V = rng.standard_normal((N, D))
    out, lse = A.causal_attention(Q, K, V, 0.25, causal=causal)
    t = lambda a: torch.from_numpy(a)[None, None]
    ref = torch.nn.functional.scaled_dot_product_attention(
        t(Q), t(K), t(V), is_causal=causal, scale=0.25)[0, 0].numpy()
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-14)
    # row-wise path agrees with the batched one
    for i in (0, 1, N // 2, N - 1):
        o_i, lse_i = A.causal_attention_row(Q[i], K, V, 0.25, i, causal=causal)
        np.testing.assert_allclose(o_i, out[i], rtol=1e-12, atol=1e-14)
        assert lse_i == pytest.approx(lse[i], rel=1e-13)


def test_prefill_causal_row0_is_v0_and_lse_by_logsumexp():
    rng = np.random.default_rng(12)
    N, D = 9, 4
    Q, K, V = (rng.standard_normal((N, D)) for _ in range(3))
    out, lse = A.causal_attention(Q, K, V, 1.0)
    np.testing.assert_array_equal(out[0], V[0])
    s = Q @ K.T
    for i in range(N):
        assert lse[i] == pytest.approx(float(torch.logsumexp(torch.from_numpy(s[i, :i + 1]), 0)),
                                       rel=1e-14)


def test_softmax_v_against_torch_softmax():
    rng = np.random.default_rng(13)
    R, L, D = 5, 33, 8
    q = rng.standard_normal((R, D))
    K = rng.standard_normal((R, L, D))
    V = rng.standard_normal((R, L, D))
    out, _, _ = A.softmax_v_rows(q, K, V, 0.125)
    s = torch.einsum("rld,rd->rl", torch.from_numpy(K), torch.from_numpy(q)) * 0.125
    ref = torch.einsum("rl,rld->rd", torch.softmax(s, dim=1), torch.from_numpy(V)).numpy()
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-15)


def test_segment_bounds():
    assert A.segment_bounds(10, 3) == [(0, 4), (4, 8), (8, 10)]
    assert A.segment_bounds(3, 5) == [(0, 1), (1, 2), (2, 3), (3, 3), (3, 3)]
    assert A.segment_bounds(32768, 16)[-1] == (30720, 32768)
