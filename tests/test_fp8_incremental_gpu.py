"""Parity of the incremental FP8 quantise-in-GEMM (rf_incremental_quant_fp8_gemm)
with the oracle's incremental form, through the C ABI: Y within the bf16
tolerance, the final per-row scales bit-exact.

Cases: one K-tile; several tiles where the abs-max grows (outliers placed
late, so the accumulator is rescaled); rows whose abs-max comes first (then
the result equals the two-phase cascade's); zero rows and a zero prefix;
scales below 2^-90 and growth from 1e-30 to O(1) (the division paths); and
the full workload [4096 x 7168] x [4096 x 7168] on sampled rows.  N = 512 and
1024 run the one-CTA kernel; N = 2048 runs clusters of 4 CTAs and N = 4096
with few rows clusters of 8 (the full workload takes clusters of 4, which
need fewer waves), each CTA quantising one row band for the cluster, so
those shapes repeat the rescale and zero cases."""

import numpy as np
import pytest
import torch

from helpers import assert_close_bf16, f64
from oracle import bf16 as obf16
from oracle import fp8 as ofp8
import synthetic_inputs as si

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rf():
    import cascaded_reductions_gb300 as m
    return m


def run(rf, x, wq, sw):
    M, K = x.shape
    N = wq.shape[0]
    y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    sx = torch.empty(M, device="cuda")
    rf.rf_incremental_quant_fp8_gemm(x.cuda(), wq.cuda(), sw.cuda(), y, sx)
    torch.cuda.synchronize()
    assert rf.rf_device_error() == 0
    return f64(y), sx.cpu().numpy()


def check(rf, x, wq, sw, what, rows=None):
    gy, gs = run(rf, x, wq, sw)
    xs = x if rows is None else x[rows]
    ry, rs = ofp8.incremental_quant_gemm(obf16.decode(xs.view(torch.int16).numpy()), wq.numpy(),
                                         sw.numpy())
    if rows is not None:
        gy, gs = gy[rows], gs[rows]
    assert np.array_equal(gs, rs), f"{what}: final scales differ"
    assert_close_bf16(gy, ry, what)


@pytest.mark.parametrize("M,K,N", [(128, 128, 512), (256, 1024, 512), (128, 2048, 1024),
                                   (128, 128, 2048), (256, 896, 2048), (128, 128, 4096),
                                   (256, 1280, 4096)])
def test_shapes(rf, M, K, N):
    x, wq, sw = si.quant_gemm_inputs(M, K, N, seed=M + K + N)
    check(rf, x, wq, sw, f"M={M} K={K} N={N}")


@pytest.mark.parametrize("N", [512, 2048, 4096])
def test_growing_abs_max_rescales(rf, N):
    M, K = 128, 1024
    x, wq, sw = si.quant_gemm_inputs(M, K, N, seed=21)
    xf = x.float()
    # the row maximum grows tile after tile: each later tile gets a larger outlier
    for t in range(K // 128):
        xf[:, t * 128 + 5] = 2.0 * (t + 1) * torch.sign(xf[:, t * 128 + 5] + 0.5)
    check(rf, xf.to(torch.bfloat16), wq, sw, f"growing N={N}")


@pytest.mark.parametrize("N", [2048, 4096])
def test_growth_in_some_rows_only(rf, N):
    # only a few rows grow, in different row bands and tiles: warps whose
    # 32 rows did not grow leave their accumulator rows alone
    M, K = 128, 1536
    x, wq, sw = si.quant_gemm_inputs(M, K, N, seed=24)
    xf = x.float()
    for i, r in enumerate([3, 40, 77, 127]):
        t = 2 + 3 * i
        xf[r, t * 128 + 9] = 25.0 * (i + 1)
    check(rf, xf.to(torch.bfloat16), wq, sw, f"some rows N={N}")


@pytest.mark.parametrize("N", [512, 4096])
def test_max_first_equals_two_phase(rf, N):
    M, K = 128, 1024
    x, wq, sw = si.quant_gemm_inputs(M, K, N, seed=22)
    xf = x.float()
    xf[:, 0] = 60.0
    x = xf.to(torch.bfloat16)
    gy, gs = run(rf, x, wq, sw)
    xq, sx, y2 = rf.absmax_quant_fp8_gemm(x.cuda(), wq.cuda(), sw.cuda())
    torch.cuda.synchronize()
    assert np.array_equal(gs, sx.cpu().numpy())
    assert_close_bf16(gy, f64(y2), "vs two-phase")


@pytest.mark.parametrize("N", [512, 4096])
def test_zero_rows_and_zero_prefix(rf, N):
    M, K = 128, 768
    x, wq, sw = si.quant_gemm_inputs(M, K, N, seed=23)
    xf = x.float()
    xf[0] = 0.0
    xf[1, :300] = 0.0
    check(rf, xf.to(torch.bfloat16), wq, sw, f"zeros N={N}")
    gy, gs = run(rf, xf.to(torch.bfloat16), wq, sw)
    assert gs[0] == 0 and np.all(gy[0] == 0)


@pytest.mark.parametrize("N", [512, 2048])
def test_tiny_scales(rf, N):
    # row 0 stays near 1e-30 (scale below 2^-90: the division-per-element
    # encoder); row 1 starts near 1e-30 and jumps to O(1) (rescale factor by
    # the division fallback); row 2 starts at O(1e-20) and grows slowly
    M, K = 128, 768
    x, wq, sw = si.quant_gemm_inputs(M, K, N, seed=25)
    xf = x.float()
    xf[0] *= 1e-30
    xf[1, :384] *= 1e-30
    xf[2] *= 1e-20
    xf[2, 700] = 3e-20
    xb = xf.to(torch.bfloat16)
    check(rf, xb, wq, sw, f"tiny scales N={N}")
    # the absolute part of the bf16 tolerance says nothing about rows this
    # small: compare them again brought up to O(1)
    gy, gs = run(rf, xb, wq, sw)
    ry, rs = ofp8.incremental_quant_gemm(obf16.decode(xb.view(torch.int16).numpy()), wq.numpy(),
                                         sw.numpy())
    for r, f in ((0, 1e30), (2, 1e20)):
        assert_close_bf16(gy[r] * f, ry[r] * f, f"row {r} scaled by {f:g}, N={N}")


def test_full_size_sampled_rows(rf):
    # 256 rows of the full workload: two whole 128-row blocks (the first and
    # the last; every row of a block is quantised by the cluster that shares
    # it) and 64 rows drawn across the rest
    cfg = si.FULL["quant_gemm"]
    M = cfg["M"]
    x, wq, sw = si.quant_gemm_inputs(M, cfg["K"], cfg["N"], seed=si.SEEDS["quant_gemm"])
    rows = set(range(0, 128)) | set(range(M - 128, M))
    rows |= set(np.random.default_rng(0).choice(np.arange(128, M - 128), 64, replace=False).tolist())
    rows = sorted(rows)
    assert len(rows) >= 256
    check(rf, x, wq, sw, "4096x7168x4096", rows=rows)
