"""Parity of causal prefill attention (rf_attn_prefill) with the oracle
through the C ABI.  out is bf16 (|g - r| <= 2e-2 + 1e-2 |r|); lse is fp32
(|g - r| <= 2e-3 |r| + 1e-6).

Cases: one tile (N = 128) causal and not; several key tiles so the K/V ring
and the two S buffers wrap; ragged lengths (N = 1 … 1000, not multiples of
128) causal and not; several batches and heads; peaked scores (large
scale) that move the running max often; enough heads that every
persistent cluster takes several work items; the full workload B=4, H=32,
N=8192 with sampled rows compared one by one, and its closed form (causal
row 0 equals V row 0 exactly).
"""

import numpy as np
import pytest
import torch

from helpers import assert_close_bf16, assert_close_f32, f64
from oracle import attention as A
import synthetic_inputs as si

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rf():
    import cascaded_reductions_gb300 as m
    return m


def run(rf, q, k, v, causal, scale):
    out, lse = rf.attn_prefill(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert rf.rf_device_error() == 0
    return f64(out), f64(lse)


def check_all(rf, B, H, N, causal, seed, scale=None):
    q, k, v = si.prefill_inputs(B, H, N, 128, seed=seed)
    scale = scale if scale is not None else 128 ** -0.5
    out, lse = run(rf, q, k, v, causal, scale)
    for b in range(B):
        for h in range(H):
            ro, rl = A.causal_attention(f64(q[b, h]), f64(k[b, h]), f64(v[b, h]), scale, causal)
            assert_close_bf16(out[b, h], ro, f"out b={b} h={h}")
            assert_close_f32(lse[b, h], rl, f"lse b={b} h={h}")


@pytest.mark.parametrize("causal", [True, False])
def test_single_tile(rf, causal):
    check_all(rf, 1, 1, 128, causal, seed=1)


@pytest.mark.parametrize("N", [256, 384, 1024])
@pytest.mark.parametrize("causal", [True, False])
def test_several_key_tiles(rf, N, causal):
    check_all(rf, 1, 2, N, causal, seed=N)


@pytest.mark.parametrize("N", [1, 77, 129, 200, 333, 1000])
@pytest.mark.parametrize("causal", [True, False])
def test_ragged_lengths(rf, N, causal):
    # a partial last tile: its keys past N are the next head's rows (or the
    # zero fill past the tensor) and must be left out; rows past N not stored
    check_all(rf, 2, 2, N, causal, seed=N + 3)


def test_batches_and_heads(rf):
    check_all(rf, 2, 3, 512, True, seed=7)


@pytest.mark.parametrize("causal", [True, False])
def test_several_items_per_cluster(rf, causal):
    # 2 x 64 heads of 5 tiles (3 pairs, the last one half past N): 384 work
    # items, several per persistent cluster, so Q buffers alternate, the
    # epilogue of one item runs inside the next item's first block, and the
    # items of a cluster differ in key-block count (causal)
    check_all(rf, 2, 64, 600, causal, seed=11)


def test_peaked_scores(rf):
    check_all(rf, 1, 2, 768, True, seed=8, scale=1.0)


def test_full_size_sampled_rows(rf):
    cfg = si.FULL["prefill"]
    B, H, N, D = cfg["B"], cfg["H"], cfg["N"], cfg["D"]
    q, k, v = si.prefill_inputs(B, H, N, D, seed=si.SEEDS["prefill"], device="cuda")
    scale = D ** -0.5
    out, lse = rf.attn_prefill(q, k, v, causal=True, scale=scale)
    torch.cuda.synchronize()
    assert rf.rf_device_error() == 0
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
    # closed form: query 0 sees only key 0
    assert torch.equal(out[:, :, 0, :], v[:, :, 0, :])
    rng = np.random.default_rng(0)
    picks = [(0, 0, 1), (3, 31, N - 1), (1, 7, 127), (2, 12, 128), (0, 5, 4095)]
    picks += [(int(rng.integers(B)), int(rng.integers(H)), int(rng.integers(N))) for _ in range(40)]
    for b, h, i in picks:
        ro, rl = A.causal_attention_row(f64(q[b, h, i]), f64(k[b, h, :i + 1]), f64(v[b, h, :i + 1]),
                                        scale, i)
        assert_close_bf16(f64(out[b, h, i]), ro, f"out ({b},{h},{i})")
        assert_close_f32(np.array([f64(lse[b, h, i])]), np.array([rl]), f"lse ({b},{h},{i})")
    # two whole heads, every one of their 8192 rows element by element: the
    # first head (computed first in the launch's heavy-first pair order) and
    # the last
    for b, h in ((0, 0), (B - 1, H - 1)):
        ro, rl = A.causal_attention(f64(q[b, h]), f64(k[b, h]), f64(v[b, h]), scale, causal=True)
        assert_close_bf16(f64(out[b, h]), ro, f"out head ({b},{h})")
        assert_close_f32(f64(lse[b, h]), rl, f"lse head ({b},{h})")
