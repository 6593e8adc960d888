"""Pins for the single-row cascade oracles (CPU only): library routines
(torch float64 softmax, numpy var), closed forms (uniform rows, arithmetic
sequences, two masses, rings), invariants (shift invariance, the parallel-
axis theorem) and brute force on tiny inputs."""

import math

import numpy as np
import pytest
import torch

from oracle import rowcascades as rc


def test_softmax_matches_torch_and_invariants():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((7, 1000)) * 3
    y = rc.row_softmax(x)
    np.testing.assert_allclose(y, torch.softmax(torch.from_numpy(x), dim=1).numpy(), rtol=1e-13)
    np.testing.assert_allclose(y.sum(axis=1), 1.0, rtol=1e-14)
    np.testing.assert_allclose(rc.row_softmax(x + 123.0), y, rtol=1e-12)   # shift invariance
    u = rc.row_softmax(np.full((2, 64), -4.0))
    np.testing.assert_allclose(u, 1 / 64, rtol=1e-15)


def test_variance_closed_forms_and_numpy():
    n = 4097
    x = np.arange(n, dtype=np.float64)[None, :]
    mean, var = rc.row_variance(x)
    assert mean[0] == (n - 1) / 2
    assert var[0] == pytest.approx((n * n - 1) / 12, rel=1e-14)
    rng = np.random.default_rng(1)
    y = rng.standard_normal((5, 333)) * 7 + 2
    mean, var = rc.row_variance(y)
    np.testing.assert_allclose(mean, y.mean(axis=1), rtol=1e-13)
    np.testing.assert_allclose(var, y.var(axis=1), rtol=1e-12)
    _, v0 = rc.row_variance(np.full((1, 50), 3.25))
    assert v0[0] == 0.0
    _, vs = rc.row_variance(y + 1e3)
    np.testing.assert_allclose(vs, var, rtol=1e-9)


def test_moment_of_inertia_closed_forms():
    # two unit masses a distance d apart: each sits d/2 from the centre
    d = 3.0
    mass = np.array([[1.0, 1.0]])
    pos = np.zeros((1, 3, 2))
    pos[0, 0] = [0.0, d]
    c, inertia = rc.moment_of_inertia(mass, pos)
    np.testing.assert_allclose(c[0], [d / 2, 0, 0])
    assert inertia[0] == pytest.approx(d * d / 2)
    # ring of equal masses of radius rho around (1, 2, 3): I = M rho^2
    k, rho = 360, 2.5
    t = np.arange(k) * 2 * math.pi / k
    pos = np.stack([1 + rho * np.cos(t), 2 + rho * np.sin(t), np.full(k, 3.0)])[None]
    mass = np.full((1, k), 0.5)
    c, inertia = rc.moment_of_inertia(mass, pos)
    np.testing.assert_allclose(c[0], [1, 2, 3], atol=1e-12)
    assert inertia[0] == pytest.approx(0.5 * k * rho * rho, rel=1e-12)


def test_moment_of_inertia_parallel_axis_and_brute_force():
    rng = np.random.default_rng(2)
    R, n = 4, 9
    mass = rng.uniform(0.1, 2.0, (R, n))
    pos = rng.standard_normal((R, 3, n))
    c, inertia = rc.moment_of_inertia(mass, pos)
    for r in range(R):
        M = sum(mass[r])
        cx = [sum(mass[r][i] * pos[r][a][i] for i in range(n)) / M for a in range(3)]
        ii = sum(mass[r][i] * sum((pos[r][a][i] - cx[a]) ** 2 for a in range(3)) for i in range(n))
        np.testing.assert_allclose(c[r], cx, rtol=1e-12)
        assert inertia[r] == pytest.approx(ii, rel=1e-12)
        # parallel-axis theorem: about the origin = about the centre + M |c|^2
        about_origin = sum(mass[r][i] * sum(pos[r][a][i] ** 2 for a in range(3)) for i in range(n))
        assert about_origin == pytest.approx(inertia[r] + M * sum(v * v for v in cx), rel=1e-12)


def test_layer_norm_matches_torch_and_closed_form():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((6, 777)) * 3 + 1
    g = rng.standard_normal(777)
    b = rng.standard_normal(777)
    y = rc.layer_norm(x, g, b, 1e-5)
    ref = torch.nn.functional.layer_norm(torch.from_numpy(x), (777,), torch.from_numpy(g),
                                         torch.from_numpy(b), 1e-5).numpy()
    np.testing.assert_allclose(y, ref, rtol=1e-11, atol=1e-12)
    # with unit gain and zero bias every row has mean 0 and variance var/(var+eps)
    z = rc.layer_norm(x, np.ones(777), np.zeros(777), 0.0)
    np.testing.assert_allclose(z.mean(axis=1), 0.0, atol=1e-12)
    np.testing.assert_allclose(z.var(axis=1), 1.0, rtol=1e-12)


def test_rms_norm_matches_torch_closed_forms_and_brute_force():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((5, 333)) * 2 - 0.5
    g = rng.standard_normal(333)
    y = rc.rms_norm(x, g, 1e-6)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(x), (333,), torch.from_numpy(g), 1e-6)
    np.testing.assert_allclose(y, ref.numpy(), rtol=1e-11, atol=1e-12)
    # a constant row c normalises to sign(c) when eps = 0; scale invariance
    c = rc.rms_norm(np.full((2, 64), -3.5), np.ones(64), 0.0)
    np.testing.assert_allclose(c, -1.0, rtol=1e-15)
    np.testing.assert_allclose(rc.rms_norm(x * 7.25, g, 0.0), rc.rms_norm(x, g, 0.0), rtol=1e-12)
    # unit gain: every row has mean square ms/(ms + eps), 1 for eps = 0
    z = rc.rms_norm(x, np.ones(333), 0.0)
    np.testing.assert_allclose((z * z).mean(axis=1), 1.0, rtol=1e-12)
    # brute force on a tiny row
    row, gam, eps = [1.0, -2.0, 0.5], [2.0, 1.0, -1.0], 0.25
    ms = sum(v * v for v in row) / 3
    want = [row[i] / math.sqrt(ms + eps) * gam[i] for i in range(3)]
    np.testing.assert_allclose(rc.rms_norm(np.array([row]), np.array(gam), eps)[0], want, rtol=1e-14)
