"""Parity of the non-incremental split-KV decode (rf_attn_decode_split_twopass)
with the oracle's segment states and merged output, through the C ABI, and its
limit on segment length (transcript cue 45: the non-incremental form only fits
short per-block sequences)."""

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


def run(rf, q, K, V, S, scale):
    R, L, D = K.shape
    q, K, V = q.cuda(), K.cuda(), V.cuda()
    sm = torch.empty(R, S, device="cuda")
    sl = torch.empty(R, S, device="cuda")
    sa = torch.empty(R, S, D, device="cuda")
    rf.rf_attn_decode_split_twopass(q, K, V, S, scale, sm, sl, sa)
    out = torch.empty(R, D, dtype=K.dtype, device="cuda")
    lse = torch.empty(R, device="cuda")
    rf.rf_state_merge(sm, sl, sa, out, lse)
    torch.cuda.synchronize()
    return out, lse, sm, sl, sa


@pytest.mark.parametrize("L,S", [(1, 1), (3, 2), (17, 5), (1001, 64), (4099, 8), (40, 1024),
                                 (16384, 1), (32768, 2)])
def test_bf16(rf, L, S):
    R, D = 4, 128
    q, K, V = si.decode_inputs(R, L, D, torch.bfloat16, seed=500 + L)
    scale = si.decode_scale(D)
    out, lse, sm, sl, sa = run(rf, q, K, V, S, scale)
    ref, m, l = A.softmax_v_rows(f64(q), f64(K), f64(V), scale)
    assert_close_bf16(f64(out), ref, f"out L={L} S={S}")
    assert_close_f32(f64(lse), m + np.log(l), f"lse L={L} S={S}")
    rm, rl, racc = A.segment_states(f64(q), f64(K), f64(V), scale, S)
    assert_states_close(f64(sm), f64(sl), f64(sa), rm, rl, racc, f"states L={L} S={S}")


def test_fp32_single_row(rf):
    q, K, V = si.decode_inputs(1, 4096, 64, torch.float32, seed=1)
    scale = si.decode_scale(64)
    out, lse, *_ = run(rf, q, K, V, 8, scale)
    ref, m, l = A.softmax_v_rows(f64(q), f64(K), f64(V), scale)
    assert_close_f32(f64(out), ref, "fp32 out")


@pytest.mark.parametrize("S", [1, 2, 4, 8])
def test_fp32_short_rows_both_forms(rf, S):
    # the short-sequence ablation's shape (512 keys, D = 64 fp32) on 64 rows:
    # the incremental and non-incremental kernels both match the oracle
    q, K, V = si.decode_inputs(64, 512, 64, torch.float32, seed=7)
    scale = si.decode_scale(64)
    ref, m, l = A.softmax_v_rows(f64(q), f64(K), f64(V), scale)
    rm, rl, racc = A.segment_states(f64(q), f64(K), f64(V), scale, S)
    out, lse, sm, sl, sa = run(rf, q, K, V, S, scale)
    assert_close_f32(f64(out), ref, f"non-incremental out S={S}")
    assert_states_close(f64(sm), f64(sl), f64(sa), rm, rl, racc, f"non-incremental states S={S}")
    out2, lse2 = rf.attn_decode(q.cuda(), K.cuda(), V.cuda(), S, scale)
    torch.cuda.synchronize()
    assert_close_f32(f64(out2), ref, f"incremental out S={S}")
    assert_close_f32(f64(lse2), m + np.log(l), f"incremental lse S={S}")


def test_segments_longer_than_shared_memory_are_refused(rf):
    q, K, V = si.decode_inputs(1, 16385, 128, torch.bfloat16, seed=3)
    with pytest.raises(rf.RFError) as e:
        run(rf, q, K, V, 1, 0.1)
    assert e.value.status == rf.RF_ERR_UNSUPPORTED
