"""Parity of the FP8 GEMM (rf_fp8_gemm_scaled) and of the whole quant -> GEMM
cascade (rf_absmax_quant_fp8_gemm) with the oracle, through the C ABI.

The GEMM consumes the e4m3 codes; the oracle recomputes Y in float64 from
the same codes (which are first checked bit-exact against the oracle's own
quantisation).  Y is bf16: |g - r| <= 2e-2 + 1e-2 |r|.

Cases: one tile with one K block; several tiles and K blocks (the shared
memory ring wraps); ragged M, N and K on every edge; more tiles than SMs (persistent loop, both TMEM
accumulators reused); identity weights (Y = dequantised X * sw); the full
workload X [4096 x 7168] with Wq [4096 x 7168], compared in full.
"""

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


def run_cascade(rf, x, wq, sw):
    xq, sx, y = rf.absmax_quant_fp8_gemm(x.cuda(), wq.cuda(), sw.cuda())
    torch.cuda.synchronize()
    assert rf.rf_device_error() == 0
    return xq.cpu().numpy(), sx.cpu().numpy(), f64(y)


def check(rf, M, K, N, seed, what):
    x, wq, sw = si.quant_gemm_inputs(M, K, N, seed=seed)
    gq, gs, gy = run_cascade(rf, x, wq, sw)
    rq, rs = ofp8.absmax_quant(obf16.decode(x.view(torch.int16).numpy()))
    assert np.array_equal(gq, rq), f"{what}: codes differ"
    assert np.array_equal(gs, rs), f"{what}: scales differ"
    ry = ofp8.scaled_gemm(rq, rs, wq.numpy(), sw.numpy())
    assert_close_bf16(gy, ry, what)


@pytest.mark.parametrize("M,K,N", [(128, 128, 256), (128, 512, 256), (256, 1024, 512),
                                   (384, 640, 768)])
def test_small(rf, M, K, N):
    check(rf, M, K, N, seed=M + K + N, what=f"M={M} K={K} N={N}")


@pytest.mark.parametrize("M,K,N", [(1, 16, 1), (1, 16, 8), (3, 48, 5), (130, 144, 300),
                                   (77, 7184, 5), (200, 16, 264), (513, 1040, 1000), (129, 2064, 257)])
def test_ragged(rf, M, K, N):
    # partial tiles on every edge: rows past M, columns past N, a last K block
    # shorter than 128 bytes; N not a multiple of 8 takes the element-wise stores
    check(rf, M, K, N, seed=M * 7 + K + N, what=f"ragged M={M} K={K} N={N}")


@pytest.mark.parametrize("M,K,N", [(2560, 272, 2048), (2500, 272, 2000)])
def test_half_tile_last_wave(rf, M, K, N):
    # 160 output tiles on 152 SMs: one whole wave, then the 8 tiles left run
    # as 16 half tiles (128 x 128); the second shape also has ragged edges
    check(rf, M, K, N, seed=M + N, what=f"half-tile wave M={M} K={K} N={N}")


def test_more_tiles_than_sms(rf):
    # 32 x 12 = 384 output tiles: every CTA runs several tiles
    check(rf, 4096, 256, 3072, seed=11, what="persistent")


def test_identity_weights(rf):
    M, K = 256, 512
    N = 512
    x, _, _ = si.quant_gemm_inputs(M, K, N, seed=5)
    wq = torch.zeros(N, K, dtype=torch.uint8)
    wq[torch.arange(K), torch.arange(K)] = 0x38          # e4m3 code of 1.0
    sw = torch.linspace(0.5, 2.0, N, dtype=torch.float32)
    gq, gs, gy = run_cascade(rf, x, wq, sw)
    expect = ofp8.e4m3_decode(gq) * gs.astype(np.float64)[:, None] * sw.numpy().astype(np.float64)[None, :K]
    assert_close_bf16(gy[:, :K], expect, "identity")
    assert np.all(gy[:, K:] == 0)


def test_gemm_alone_matches_oracle(rf):
    M, K, N = 256, 384, 256
    g = torch.Generator().manual_seed(3)
    finite = torch.tensor([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=torch.uint8)
    xq = finite[torch.randint(0, len(finite), (M, K), generator=g)]
    wq = finite[torch.randint(0, len(finite), (N, K), generator=g)]
    sx = torch.rand(M, generator=g) + 0.01
    sw = torch.rand(N, generator=g) + 0.01
    y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    rf.rf_fp8_gemm_scaled(xq.cuda(), sx.cuda(), wq.cuda(), sw.cuda(), y)
    torch.cuda.synchronize()
    ry = ofp8.scaled_gemm(xq.numpy(), sx.numpy(), wq.numpy(), sw.numpy())
    assert_close_bf16(f64(y), ry, "gemm alone")


def test_full_size(rf):
    cfg = si.FULL["quant_gemm"]
    check(rf, cfg["M"], cfg["K"], cfg["N"], seed=si.SEEDS["quant_gemm"], what="4096x7168x4096")
