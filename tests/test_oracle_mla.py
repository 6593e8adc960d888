"""Pins for the MLA decode oracle (CPU only): torch's float64 scaled-dot-product
attention with the latent rows as every head's keys, closed forms (zero query,
identical latent rows), the rotary-dims invariance that fixes which latent
dims are the value, the segment-merge invariant with empty segments, and brute
force on a tiny case."""

import math

import numpy as np
import pytest
import torch

from oracle import attention as att
from oracle import mla


def _case(B, H, L, Dk, seed):
    rng = np.random.default_rng(seed)
    return rng.standard_normal((B, H, Dk)), rng.standard_normal((B, L, Dk))


def test_matches_torch_sdpa_with_shared_latent_keys():
    B, H, L, Dk, dv = 2, 4, 37, 24, 16
    q, C = _case(B, H, L, Dk, 0)
    scale = 1 / math.sqrt(12)
    out, m, l = mla.mla_decode(q, C, dv, scale)
    Q = torch.from_numpy(q)[:, :, None, :]                          # [B, H, 1, Dk]
    K = torch.from_numpy(C)[:, None, :, :].expand(B, H, L, Dk)      # every head reads C
    V = torch.from_numpy(C[:, :, :dv])[:, None, :, :].expand(B, H, L, dv)
    ref = torch.nn.functional.scaled_dot_product_attention(Q, K, V, scale=scale)[:, :, 0, :]
    np.testing.assert_allclose(out, ref.numpy(), rtol=1e-12, atol=1e-13)
    lse_ref = torch.logsumexp(scale * torch.einsum("bhd,bld->bhl", torch.from_numpy(q),
                                                   torch.from_numpy(C)), dim=2)
    np.testing.assert_allclose(m + np.log(l), lse_ref.numpy(), rtol=1e-13)


def test_value_is_the_leading_latent_dims():
    # with the query's rotary dims zero, the rotary dims of the cache affect nothing
    B, H, L, Dk, dv = 1, 3, 20, 12, 8
    q, C = _case(B, H, L, Dk, 1)
    q[:, :, dv:] = 0
    C2 = C.copy()
    C2[:, :, dv:] = np.random.default_rng(9).standard_normal((B, L, Dk - dv)) * 5
    a, _, _ = mla.mla_decode(q, C, dv, 0.3)
    b, _, _ = mla.mla_decode(q, C2, dv, 0.3)
    np.testing.assert_allclose(a, b, rtol=1e-14)
    # ... while with uniform weights (scale 0) output dim 0 is the mean of latent dim 0
    c, _, _ = mla.mla_decode(q, C2, dv, 0.0)
    np.testing.assert_allclose(c[0, :, 0], C2[0, :, 0].mean(), rtol=1e-13)


def test_closed_forms():
    B, H, L, Dk, dv = 2, 2, 50, 10, 6
    q, C = _case(B, H, L, Dk, 2)
    # zero query: uniform weights, the output is the mean value row
    out, m, l = mla.mla_decode(np.zeros_like(q), C, dv, 0.5)
    np.testing.assert_allclose(out, np.broadcast_to(C[:, None, :, :dv].mean(axis=2), out.shape),
                               rtol=1e-13)
    np.testing.assert_allclose(l, L)
    assert np.all(m == 0)
    # identical latent rows: the output is that row, whatever the query
    Cs = np.broadcast_to(C[:, :1, :], C.shape).copy()
    out, _, l = mla.mla_decode(q, Cs, dv, 0.5)
    np.testing.assert_allclose(out, np.broadcast_to(Cs[:, None, 0, :dv], out.shape), rtol=1e-13)
    np.testing.assert_allclose(l, L, rtol=1e-13)


@pytest.mark.parametrize("S", [1, 3, 7, 64])
def test_segment_merge_equals_single_pass(S):
    B, H, L, Dk, dv = 2, 3, 45, 16, 8        # S = 64 > L leaves segments empty
    q, C = _case(B, H, L, Dk, 3)
    out, m, l = mla.mla_decode(q, C, dv, 0.25)
    sm, sl, sacc = mla.mla_segment_states(q, C, dv, 0.25, S)
    if S > L:
        assert np.isneginf(sm[..., -1]).all() and (sl[..., -1] == 0).all()
    mo, lse = att.merge_states(sm.reshape(B * H, S), sl.reshape(B * H, S),
                               sacc.reshape(B * H, S, dv))
    np.testing.assert_allclose(mo.reshape(B, H, dv), out, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(lse.reshape(B, H), m + np.log(l), rtol=1e-13)


def test_brute_force_tiny():
    B, H, L, Dk, dv = 1, 2, 3, 5, 3
    q, C = _case(B, H, L, Dk, 4)
    scale = 0.7
    out, m, l = mla.mla_decode(q, C, dv, scale)
    for h in range(H):
        s = [scale * sum(q[0][h][d] * C[0][j][d] for d in range(Dk)) for j in range(L)]
        mx = max(s)
        w = [math.exp(x - mx) for x in s]
        den = sum(w)
        for v in range(dv):
            assert out[0, h, v] == pytest.approx(sum(w[j] * C[0][j][v] for j in range(L)) / den,
                                                 rel=1e-13)
        assert m[0, h] == pytest.approx(mx) and l[0, h] == pytest.approx(den)
