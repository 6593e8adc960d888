"""Parity of the single-row cascades (rf_row_softmax, rf_row_variance,
rf_moment_of_inertia) with the oracle through the C ABI, at every fusion
level (unfused, thread, warp, block).  fp32 outputs: |g - r| <= 2e-3 |r| +
1e-6 (variance and inertia scale the absolute term by the row's size).

Cases: rows of 4 to 8192 elements (ragged against the 128- and 1024-element
tiles), the benchmark's sizes on sampled rows, a constant row (variance 0),
shifted data, two point masses (I = d^2/2) and uneven masses."""

import numpy as np
import pytest
import torch

from helpers import assert_close_f32, f64
from oracle import rowcascades as rc

pytestmark = pytest.mark.gpu

LEVELS = [0, 1, 2, 3]


@pytest.fixture(scope="module")
def rf():
    import cascaded_reductions_gb300 as m
    return m


def softmax(rf, x, level):
    R, n = x.shape
    xd = x.cuda()
    y = torch.empty_like(xd)
    work = torch.empty(2 * R, device="cuda") if level == 0 else None
    rf.rf_row_softmax(xd, y, level, work)
    torch.cuda.synchronize()
    return f64(y)


@pytest.mark.parametrize("level", LEVELS)
@pytest.mark.parametrize("n", [4, 1000, 1024, 1028, 2052, 4096, 8192])
def test_softmax(rf, level, n):
    g = torch.Generator().manual_seed(n + level)
    x = torch.randn(17, n, generator=g) * 3
    assert_close_f32(softmax(rf, x, level), rc.row_softmax(x.numpy()), f"n={n} level={level}")


@pytest.mark.parametrize("level", LEVELS)
def test_softmax_unfused_long_rows(rf, level):
    if level != 0:
        pytest.skip("fused levels hold rows of at most 8192 in registers")
    x = torch.randn(3, 20000, generator=torch.Generator().manual_seed(5))
    assert_close_f32(softmax(rf, x, 0), rc.row_softmax(x.numpy()), "n=20000")


def variance(rf, x, level):
    R = x.shape[0]
    mean = torch.empty(R, device="cuda")
    var = torch.empty(R, device="cuda")
    rf.rf_row_variance(x.cuda(), mean, var, level)
    torch.cuda.synchronize()
    return f64(mean), f64(var)


@pytest.mark.parametrize("level", LEVELS)
@pytest.mark.parametrize("n", [4, 1000, 4096, 10004])
def test_variance(rf, level, n):
    g = torch.Generator().manual_seed(100 + n + level)
    x = torch.randn(9, n, generator=g) * torch.rand(9, 1, generator=g) * 4 + torch.randn(9, 1, generator=g)
    x[0] = 2.5                                       # constant row: variance 0
    gm, gv = variance(rf, x, level)
    rm, rv = rc.row_variance(x.numpy())
    assert_close_f32(gm, rm, f"mean n={n} level={level}")
    # fp32 accumulation over n values: absolute slack scales with the row's second moment
    scale = (x.double() ** 2).mean(dim=1).numpy()
    assert np.all(np.abs(gv - rv) <= 2e-3 * np.abs(rv) + 1e-6 * scale + 1e-7), (gv, rv)
    assert abs(gv[0]) <= 1e-6


def inertia(rf, mass, pos, level):
    R = mass.shape[0]
    c = torch.empty(R, 3, device="cuda")
    i = torch.empty(R, device="cuda")
    rf.rf_moment_of_inertia(mass.cuda(), pos.cuda(), c, i, level)
    torch.cuda.synchronize()
    return f64(c), f64(i)


@pytest.mark.parametrize("level", LEVELS)
@pytest.mark.parametrize("n", [4, 1000, 4096])
def test_moment_of_inertia(rf, level, n):
    g = torch.Generator().manual_seed(200 + n + level)
    mass = torch.rand(7, n, generator=g) + 0.05
    pos = torch.randn(7, 3, n, generator=g) * 2 + 1
    gc, gi = inertia(rf, mass, pos, level)
    rcen, ri = rc.moment_of_inertia(mass.numpy(), pos.numpy())
    assert np.all(np.abs(gc - rcen) <= 2e-3 * np.abs(rcen) + 1e-4), (gc, rcen)
    assert_close_f32(gi, ri, f"inertia n={n} level={level}")


@pytest.mark.parametrize("level", LEVELS)
def test_two_masses(rf, level):
    n, d = 8, 3.0
    mass = torch.zeros(1, n)
    mass[0, :2] = 1.0
    mass[0, 2:] = 1e-30                              # tiny but positive
    pos = torch.zeros(1, 3, n)
    pos[0, 0, 1] = d
    gc, gi = inertia(rf, mass, pos, level)
    assert gi[0] == pytest.approx(d * d / 2, rel=1e-5)
    assert gc[0, 0] == pytest.approx(d / 2, rel=1e-6)


@pytest.mark.parametrize("level", LEVELS)
def test_benchmark_sizes_sampled(rf, level):
    """The sizes the benchmark times: softmax rows of 8192 (8192 rows), variance
    and inertia rows of 4096 (16384 and 4096 rows); 16 sampled rows each."""
    g = torch.Generator(device="cuda").manual_seed(7)
    rows = np.random.default_rng(level).choice(8192, 16, replace=False)
    x = torch.randn(8192, 8192, device="cuda", generator=g) * 2
    y = torch.empty_like(x)
    work = torch.empty(2 * 8192, device="cuda") if level == 0 else None
    rf.rf_row_softmax(x, y, level, work)
    torch.cuda.synchronize()
    assert_close_f32(f64(y[rows]), rc.row_softmax(f64(x[rows])), "softmax 8192x8192")
    xv = torch.randn(16384, 4096, device="cuda", generator=g)
    mean = torch.empty(16384, device="cuda")
    var = torch.empty(16384, device="cuda")
    rf.rf_row_variance(xv, mean, var, level)
    torch.cuda.synchronize()
    rm, rv = rc.row_variance(f64(xv[rows]))
    assert_close_f32(f64(mean[rows]), rm, "mean")
    assert np.all(np.abs(f64(var[rows]) - rv) <= 2e-3 * rv + 1e-6)
    del x, y, xv
    torch.cuda.empty_cache()


@pytest.mark.parametrize("level", LEVELS)
@pytest.mark.parametrize("n", [4, 1000, 4096, 8192])
def test_layer_norm(rf, level, n):
    g = torch.Generator().manual_seed(300 + n + level)
    x = torch.randn(11, n, generator=g) * 3 + 2
    gamma = torch.randn(n, generator=g)
    beta = torch.randn(n, generator=g)
    y = torch.empty(11, n, device="cuda")
    work = torch.empty(22, device="cuda") if level == 0 else None
    rf.rf_layer_norm(x.cuda(), gamma.cuda(), beta.cuda(), 1e-5, y, level, work)
    torch.cuda.synchronize()
    ref = rc.layer_norm(x.numpy(), gamma.numpy(), beta.numpy(), 1e-5)
    # normalised values are O(1): relative bound plus a small absolute term
    assert np.all(np.abs(f64(y) - ref) <= 2e-3 * np.abs(ref) + 1e-4), np.abs(f64(y) - ref).max()


@pytest.mark.parametrize("level", LEVELS)
@pytest.mark.parametrize("n", [4, 1000, 4096, 8192])
def test_rms_norm(rf, level, n):
    g = torch.Generator().manual_seed(400 + n + level)
    x = torch.randn(13, n, generator=g) * 3 - 1
    x[5] = 0.0                                  # all-zero row: y = 0 (eps > 0)
    gamma = torch.randn(n, generator=g)
    y = torch.empty(13, n, device="cuda")
    work = torch.empty(13, device="cuda") if level == 0 else None
    rf.rf_rms_norm(x.cuda(), gamma.cuda(), 1e-6, y, level, work)
    torch.cuda.synchronize()
    ref = rc.rms_norm(x.numpy(), gamma.numpy(), 1e-6)
    assert_close_f32(f64(y), ref, f"rms norm n={n} level={level}")
