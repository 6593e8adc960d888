"""Parity of split-KV decode (rf_attn_decode_split + rf_state_merge) with the
oracle, through the C ABI.

* the worked example of the RedFuser episode (scores 1, 3 | 5): the segment
  states must be the ones the transcript spells out (cue 15);
* single-row fp32 D=64 at its full size (L=4096) for every S;
* bf16 D=128 rows with ragged key counts, every S from 1 to past L;
* edge cases: L=1, S > L (identity states), S=1024;
* the full-size bf16 workload (B=32, H=32, L=32768, S=16, 16 GiB) on
  sampled rows, in the launch configuration the benchmark times.
"""

import math

import numpy as np
import pytest
import torch

from helpers import assert_close_bf16, assert_close_f32, assert_states_close, f64
from oracle import attention as A
import synthetic_inputs as si

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rf():
    import cascaded_reductions_gb300 as m
    return m


def run(rf, q, K, V, S, scale, out_dtype=None):
    out, lse, (sm, sl, sa) = rf.attn_decode(q.cuda(), K.cuda(), V.cuda(), S, scale,
                                            out_dtype=out_dtype, return_states=True)
    torch.cuda.synchronize()
    return out, lse, sm, sl, sa


def test_worked_example(rf):
    D, L = 64, 3
    q = torch.zeros(1, D)
    q[0, 0] = 1.0
    K = torch.zeros(1, L, D)
    K[0, :, 0] = torch.tensor([1.0, 3.0, 5.0])
    V = torch.zeros(1, L, D)
    V[0, :, 0] = torch.tensor([2.0, -1.0, 4.0])
    out, lse, sm, sl, sa = run(rf, q, K, V, 2, 1.0)
    e2, e4 = math.exp(-2), math.exp(-4)
    assert sm[0, 0].item() == pytest.approx(3.0, abs=1e-6)
    assert sm[0, 1].item() == pytest.approx(5.0, abs=1e-6)
    assert sl[0, 0].item() == pytest.approx(1 + e2, rel=1e-6)
    assert sa[0, 0, 0].item() == pytest.approx(2 * e2 - 1, rel=1e-5)
    assert sl[0, 1].item() == pytest.approx(1.0, rel=1e-6)
    assert sa[0, 1, 0].item() == pytest.approx(4.0, rel=1e-6)
    assert out[0, 0].item() == pytest.approx((2 * e4 - e2 + 4) / (e4 + e2 + 1), rel=1e-6)
    assert lse[0].item() == pytest.approx(5 + math.log(e4 + e2 + 1), rel=1e-6)
    assert torch.all(out[0, 1:] == 0)


@pytest.mark.parametrize("S", [1, 2, 4, 8, 16, 32, 64, 4096])
def test_single_row_fp32_full_size(rf, S):
    cfg = si.FULL["decode_f32"]
    q, K, V = si.decode_inputs(cfg["R"], cfg["L"], cfg["D"], torch.float32, seed=si.SEEDS["decode_f32"])
    scale = si.decode_scale(cfg["D"])
    out, lse, sm, sl, sa = run(rf, q, K, V, S, scale)
    ref, m, l = A.softmax_v_rows(f64(q), f64(K), f64(V), scale)
    assert_close_f32(f64(out), ref, f"out S={S}")
    assert_close_f32(f64(lse), m + np.log(l), f"lse S={S}")
    rm, rl, racc = A.segment_states(f64(q), f64(K), f64(V), scale, S)
    assert_states_close(f64(sm), f64(sl), f64(sa), rm, rl, racc, f"states S={S}")


@pytest.mark.parametrize("L,S", [(1, 1), (1, 7), (3, 2), (17, 5), (255, 16), (1000, 3), (1001, 64),
                                 (4099, 8), (40, 1024), (2048, 16)])
def test_bf16_ragged(rf, L, S):
    R, D = 6, 128
    q, K, V = si.decode_inputs(R, L, D, torch.bfloat16, seed=100 + L)
    scale = si.decode_scale(D)
    out, lse, sm, sl, sa = run(rf, q, K, V, S, scale)
    ref, m, l = A.softmax_v_rows(f64(q), f64(K), f64(V), scale)
    assert_close_bf16(f64(out), ref, f"out L={L} S={S}")
    assert_close_f32(f64(lse), m + np.log(l), f"lse L={L} S={S}")
    rm, rl, racc = A.segment_states(f64(q), f64(K), f64(V), scale, S)
    assert_states_close(f64(sm), f64(sl), f64(sa), rm, rl, racc, f"states L={L} S={S}")


def test_fp32_output_of_bf16_inputs_and_large_scores(rf):
    """Peaked softmax (large scale): the running max changes often and the
    rescale factors span many orders of magnitude."""
    R, L, D = 4, 777, 128
    q, K, V = si.decode_inputs(R, L, D, torch.bfloat16, seed=7)
    scale = 1.5
    out, lse, sm, sl, sa = run(rf, q, K, V, 9, scale, out_dtype=torch.float32)
    ref, m, l = A.softmax_v_rows(f64(q), f64(K), f64(V), scale)
    # fp32 out of an fp32-accumulated path whose scores carry fp32 rounding
    # amplified by the large scale: compare with the bf16 bound
    assert_close_bf16(f64(out), ref, "out")
    rm, rl, racc = A.segment_states(f64(q), f64(K), f64(V), scale, 9)
    assert np.allclose(f64(sm), rm, rtol=1e-5, atol=1e-4)


def test_full_size_bf16_sampled_rows(rf):
    """B=32, H=32, L=32768, D=128 bf16 (16 GiB of K and V) with S=16, the
    benchmark's launch configuration: every row is checked for finite output;
    64 rows spread over every batch and head (the first and last row, one
    row of every 16, and 6 more drawn at random) are compared element by
    element with the oracle, segment states included."""
    cfg = si.FULL["decode_bf16"]
    B, H, L, D = cfg["B"], cfg["H"], cfg["L"], cfg["D"]
    R, S = B * H, 16
    q, K, V = si.decode_inputs(R, L, D, torch.bfloat16, seed=si.SEEDS["decode_bf16"], device="cuda")
    scale = si.decode_scale(D)
    out, lse, (sm, sl, sa) = rf.attn_decode(q, K, V, S, scale, return_states=True)
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
    rows = set(range(0, R, 16)) | {0, R - 1}
    rows |= set(np.random.default_rng(0).choice(R, 6, replace=False).tolist())
    rows = sorted(rows)
    assert len(rows) >= 64
    for r in rows:
        qr, Kr, Vr = f64(q[r:r + 1]), f64(K[r:r + 1]), f64(V[r:r + 1])
        ref, m, l = A.softmax_v_rows(qr, Kr, Vr, scale)
        assert_close_bf16(f64(out[r:r + 1]), ref, f"out row {r}")
        assert_close_f32(f64(lse[r:r + 1]), m + np.log(l), f"lse row {r}")
        rm, rl, racc = A.segment_states(qr, Kr, Vr, scale, S)
        assert_states_close(f64(sm[r:r + 1]), f64(sl[r:r + 1]), f64(sa[r:r + 1]), rm, rl, racc,
                            f"states row {r}")
    del q, K, V
    torch.cuda.empty_cache()
