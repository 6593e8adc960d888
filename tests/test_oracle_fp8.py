"""Pins for the FP8 quant -> GEMM oracle and the oracle's codecs (CPU only).

* e4m3 decode of all 256 codes against torch's float8_e4m3fn (library);
* encode: every finite code round-trips; every midpoint between neighbours
  rounds to the even mantissa; values above 448 saturate; agreement with
  torch's float8 cast on random values within range (torch rounds to nearest
  even but does not saturate beyond 464, so the comparison stays below it);
* quantisation: rows already on the e4m3 grid with amax = 448 give identity
  codes and scale 1; the zero row; dequantised values within half a step of
  the input (the rounding bound);
* GEMM: identity weight codes reduce Y to dequantised X; brute force on
  tiny shapes;
* bf16 codec against torch's bfloat16 view and cast.
"""

import numpy as np
import pytest
import torch

from oracle import bf16, fp8


ALL = np.arange(256, dtype=np.uint8)


def _torch_decode(codes):
    return torch.from_numpy(np.asarray(codes, np.uint8)).view(torch.float8_e4m3fn).double().numpy()


def test_decode_all_codes_matches_torch():
    mine = fp8.e4m3_decode(ALL)
    ref = _torch_decode(ALL)
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(mine[ok], ref[ok])
    assert np.isnan(mine[0x7F]) and np.isnan(mine[0xFF])
    assert mine[0x7E] == 448.0 and mine[0x01] == 2.0 ** -9 and mine[0x38] == 1.0
    assert mine[0x08] == 2.0 ** -6 and mine[0x07] == 7 * 2.0 ** -9


def test_encode_roundtrip_all_finite_codes():
    finite = np.array([c for c in ALL if (c & 0x7F) != 0x7F], dtype=np.uint8)
    vals = fp8.e4m3_decode(finite).astype(np.float32)
    codes = fp8.e4m3_encode(vals)
    np.testing.assert_array_equal(codes, finite)


def test_encode_midpoints_round_to_even():
    pos = np.arange(0, 0x7E, dtype=np.uint8)          # 0 .. 0x7D, next code exists
    lo = fp8.e4m3_decode(pos)
    hi = fp8.e4m3_decode(pos + 1)
    mid = ((lo + hi) / 2).astype(np.float32)
    assert np.all(mid.astype(np.float64) == (lo + hi) / 2)   # midpoints are exact in fp32
    codes = fp8.e4m3_encode(mid)
    expect = np.where(pos % 2 == 0, pos, pos + 1).astype(np.uint8)
    np.testing.assert_array_equal(codes, expect)
    np.testing.assert_array_equal(fp8.e4m3_encode(-mid), expect | 0x80)
    # a hair either side of the midpoint goes to the nearer neighbour
    above = np.nextafter(mid, np.float32(np.inf))
    below = np.nextafter(mid, np.float32(0))
    np.testing.assert_array_equal(fp8.e4m3_encode(above), pos + 1)
    np.testing.assert_array_equal(fp8.e4m3_encode(below), pos)


def test_encode_saturates_and_keeps_sign_and_nan():
    big = np.array([448.0, 448.5, 463.9, 464.0, 470.0, 479.0, 480.0, 1e6, 3.0e38], np.float32)
    np.testing.assert_array_equal(fp8.e4m3_encode(big), 0x7E)
    np.testing.assert_array_equal(fp8.e4m3_encode(-big), 0xFE)
    tiny = np.array([0.0, 1e-30, 2.0 ** -10], np.float32)
    np.testing.assert_array_equal(fp8.e4m3_encode(tiny), 0x00)
    np.testing.assert_array_equal(fp8.e4m3_encode(-tiny), 0x80)
    assert fp8.e4m3_encode(np.array([np.nan], np.float32))[0] == 0x7F


def test_encode_matches_torch_cast_in_range():
    rng = np.random.default_rng(0)
    v = np.concatenate([
        rng.uniform(-463.0, 463.0, 200000),
        rng.standard_normal(200000) * 0.01,
        rng.standard_normal(200000) * 2.0 ** -8,
        rng.standard_normal(200000) * 30,
    ]).astype(np.float32)
    mine = fp8.e4m3_encode(v)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(mine, ref)


def test_quant_on_grid_row_is_identity():
    rng = np.random.default_rng(1)
    finite = np.array([c for c in ALL if (c & 0x7F) not in (0x7F,)], dtype=np.uint8)
    codes = rng.choice(finite, size=(3, 256))
    codes[:, 5] = 0x7E          # amax exactly 448
    x = fp8.e4m3_decode(codes)
    xq, sx = fp8.absmax_quant(x)
    np.testing.assert_array_equal(sx, np.float32(1.0))
    # -0 codes and +0 codes both decode to 0; compare values, then signs of non-zeros
    np.testing.assert_array_equal(fp8.e4m3_decode(xq), x)
    nz = x != 0
    np.testing.assert_array_equal(xq[nz], codes[nz])


def test_quant_zero_row_and_error_bound():
    rng = np.random.default_rng(2)
    x = bf16.decode(bf16.encode_from_f32(rng.standard_normal((8, 512)).astype(np.float32)))
    x[3] = 0.0
    x[5, 17] = 20.0 * x[5].max()     # outlier
    xq, sx = fp8.absmax_quant(x)
    assert sx[3] == 0.0 and np.all(xq[3] == 0)
    for r in range(8):
        if r == 3:
            continue
        amax = np.abs(x[r]).max()
        assert sx[r] == np.float32(amax / 448.0)
        # the largest magnitude maps to 448 (up to the fp32 scale rounding)
        assert fp8.e4m3_decode(xq[r][np.argmax(np.abs(x[r]))]) == pytest.approx(
            np.sign(x[r][np.argmax(np.abs(x[r]))]) * 448.0, rel=2 ** -3)
        v = x[r] / float(sx[r])
        dq = fp8.e4m3_decode(xq[r])
        # RNE bound: half a step; the step is 2**(e-3) in the binade of |v|,
        # 2**-9 below 2**-6
        e = np.floor(np.log2(np.maximum(np.abs(v), 2.0 ** -6)))
        half_step = 2.0 ** (e - 4)
        assert np.all(np.abs(dq - v) <= half_step * (1 + 1e-6))


def test_gemm_identity_weights_reduce_to_dequantised_x():
    rng = np.random.default_rng(3)
    M, K = 6, 32
    x = rng.standard_normal((M, K))
    xq, sx = fp8.absmax_quant(x)
    wq = np.zeros((K, K), np.uint8)
    np.fill_diagonal(wq, 0x38)                # code of 1.0
    sw = np.full(K, 1.0, np.float32)
    y = fp8.scaled_gemm(xq, sx, wq, sw)
    np.testing.assert_array_equal(y, fp8.e4m3_decode(xq) * sx.astype(np.float64)[:, None])


def test_gemm_brute_force_tiny():
    rng = np.random.default_rng(4)
    M, N, K = 5, 7, 16
    xq = rng.integers(0, 256, (M, K)).astype(np.uint8)
    wq = rng.integers(0, 256, (N, K)).astype(np.uint8)
    xq[(xq & 0x7F) == 0x7F] = 0x11
    wq[(wq & 0x7F) == 0x7F] = 0x22
    sx = rng.uniform(0.1, 2, M).astype(np.float32)
    sw = rng.uniform(0.1, 2, N).astype(np.float32)
    y = fp8.scaled_gemm(xq, sx, wq, sw)
    a = _torch_decode(xq)
    b = _torch_decode(wq)
    for m in range(M):
        for n in range(N):
            acc = sum(float(a[m, k]) * float(b[n, k]) for k in range(K))
            assert y[m, n] == pytest.approx(acc * float(sx[m]) * float(sw[n]), rel=1e-13, abs=1e-13)


def test_bf16_codec_matches_torch():
    rng = np.random.default_rng(5)
    f = np.concatenate([rng.standard_normal(100000).astype(np.float32) * s for s in (1e-3, 1, 1e3)])
    mine = bf16.encode_from_f32(f)
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(mine, ref)
    bits = np.arange(0, 65536, dtype=np.uint32).astype(np.uint16)
    dec = bf16.decode(bits)
    refd = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    ok = ~np.isnan(refd)
    np.testing.assert_array_equal(dec[ok], refd[ok])
    assert np.array_equal(np.isnan(dec), np.isnan(refd))


def _nearest_f32(fr):
    """Correctly rounded float32 of a positive Fraction (ties to even), by search."""
    from fractions import Fraction
    f = np.float32(float(fr))             # within an ulp or so
    cands = [np.nextafter(f, np.float32(0)), f, np.nextafter(f, np.float32(np.inf))]
    best = min(cands, key=lambda c: (abs(Fraction(float(c)) - fr),
                                     int(np.array(c, np.float32).view(np.uint32)) & 1))
    return best


def _nearest_code_brute(v):
    """Nearest finite e4m3 code to float value v by exhaustive search; ties to even mantissa;
    above 448 clamps to 448."""
    finite = [c for c in range(128) if c != 0x7F]
    vals = fp8.e4m3_decode(np.array(finite, np.uint8))
    a = min(abs(float(v)), 448.0)
    d = np.abs(vals - a)
    best = d.min()
    ties = [c for c, dd in zip(finite, d) if dd == best]
    c = [t for t in ties if t % 2 == 0][0] if len(ties) > 1 else ties[0]
    return c | (0x80 if np.signbit(v) else 0)


def test_quant_scale_and_quotient_are_correctly_rounded_fp32():
    """sx = fp32(amax/448) and each v = fp32(x/sx) must be the correctly rounded
    float32 quotients (checked with exact rationals), and each code the nearest
    e4m3 value (checked by exhaustive search)."""
    from fractions import Fraction
    rng = np.random.default_rng(6)
    x = bf16.decode(bf16.encode_from_f32((rng.standard_normal((64, 96)) *
                                          rng.uniform(0.01, 50, (64, 1))).astype(np.float32)))
    xq, sx = fp8.absmax_quant(x)
    for r in range(64):
        amax = Fraction(float(np.abs(x[r]).max()))
        assert sx[r] == _nearest_f32(amax / 448)
        s = Fraction(float(sx[r]))
        for kk in range(0, 96, 7):
            xv = Fraction(float(x[r, kk]))
            v = _nearest_f32(abs(xv) / s)
            v = np.float32(-v) if xv < 0 else np.float32(v)
            assert xq[r, kk] == _nearest_code_brute(v)


def test_incremental_equals_two_phase_when_the_max_comes_first():
    """If every row's abs-max sits in the first K-tile the running scale never
    changes: the incremental form uses the final scale throughout and must give
    the two-phase result."""
    rng = np.random.default_rng(7)
    M, K, N = 6, 512, 40
    x = bf16.decode(bf16.encode_from_f32(rng.standard_normal((M, K)).astype(np.float32)))
    x[:, 3] = 50.0 * np.sign(rng.standard_normal(M))
    wq = rng.integers(0, 0x7E, (N, K)).astype(np.uint8)
    sw = rng.uniform(0.5, 2, N).astype(np.float32)
    y_inc, s_inc = fp8.incremental_quant_gemm(x, wq, sw)
    xq, sx = fp8.absmax_quant(x)
    np.testing.assert_array_equal(s_inc, sx)
    np.testing.assert_allclose(y_inc, fp8.scaled_gemm(xq, sx, wq, sw), rtol=1e-12, atol=1e-12)


def test_incremental_rescale_closed_form():
    """Row [112, 896] in two tiles of one column: tile 0 has scale 112/448 = 1/4
    and code 448; tile 1 raises the scale to 2 (code 448) and rescales the
    accumulator by (1/4)/2.  Every scale is a power of two and every value lies
    on the e4m3 grid, so with w = [1, 0.5]: Y = 112 * 1 + 896 * 0.5 exactly."""
    x = np.array([[112.0, 896.0]])
    wq = np.array([[0x38, 0x30]], dtype=np.uint8)     # 1.0 and 0.5
    y, s = fp8.incremental_quant_gemm(x, wq, np.ones(1, np.float32), tile_k=1)
    assert s[0] == np.float32(2.0)
    assert y[0, 0] == 112.0 * 1.0 + 896.0 * 0.5


def test_incremental_differs_from_two_phase():
    """Row [1.09375, 896] in two tiles of one column, weights [1, 0]: the
    incremental form quantises 1.09375 with its own scale s0 = fp32(1.09375 /
    448) (code 448), so Y = 448 s0, within fp32 rounding of 1.09375; with the
    final scale 2 throughout (the two-phase cascade) it would be coded as
    0.546875 -> 0.5625 (the nearer e4m3 value) and Y = 1.125.  Catches an
    incremental form that uses the final scale for every tile."""
    x = np.array([[1.09375, 896.0]])
    wq = np.array([[0x38, 0x00]], dtype=np.uint8)     # 1.0 and 0
    y, s = fp8.incremental_quant_gemm(x, wq, np.ones(1, np.float32), tile_k=1)
    assert s[0] == np.float32(2.0)
    assert abs(y[0, 0] - 1.09375) <= 1.09375 * 2.0 ** -22
    xq, sx = fp8.absmax_quant(x)
    y2 = fp8.scaled_gemm(xq, sx, wq, np.ones(1, np.float32))
    assert y2[0, 0] == 1.125


def test_incremental_zero_prefix_and_error_bound():
    rng = np.random.default_rng(8)
    M, K, N = 4, 384, 16
    x = bf16.decode(bf16.encode_from_f32(rng.standard_normal((M, K)).astype(np.float32)))
    x[0, :200] = 0.0                                  # scale 0 for the first tile, then grows
    x[1] = 0.0                                        # all-zero row
    wq = rng.integers(0, 0x7E, (N, K)).astype(np.uint8)
    sw = np.ones(N, np.float32)
    y, s = fp8.incremental_quant_gemm(x, wq, sw)
    assert s[1] == 0 and np.all(y[1] == 0)
    # each tile is quantised at most as coarsely as with the final scale, so the
    # result stays within the e4m3 rounding bound of the exact product
    exact = x @ fp8.e4m3_decode(wq).T
    bound = (np.abs(x) * 2.0 ** -4).sum(axis=1)[:, None] * np.abs(fp8.e4m3_decode(wq)).max()
    assert np.all(np.abs(y - exact) <= bound + 1e-9)
