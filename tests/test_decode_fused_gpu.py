"""Parity of rf_attn_decode_fused (split-KV decode whose merge is done by each
row's last CTA, in one launch) with the oracle, and with the two-launch path
on the same inputs: the segment states it leaves are those of
rf_attn_decode_split, its output and lse those of rf_state_merge.  The
counters start at zero and every call leaves them at zero, so repeated calls
reuse them."""

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


def run(rf, q, K, V, S, scale, out_dtype, counters=None, calls=1):
    R, L, D = K.shape
    q, K, V = q.cuda(), K.cuda(), V.cuda()
    sm = torch.empty(R, S, device="cuda")
    sl = torch.empty(R, S, device="cuda")
    sa = torch.empty(R, S, D, device="cuda")
    out = torch.empty(R, D, device="cuda", dtype=out_dtype)
    lse = torch.empty(R, device="cuda")
    if counters is None:
        counters = torch.zeros(R, dtype=torch.int32, device="cuda")
    for _ in range(calls):
        rf.rf_attn_decode_fused(q, K, V, S, scale, sm, sl, sa, counters, out, lse)
    torch.cuda.synchronize()
    assert rf.rf_device_error() == 0
    assert int(counters.abs().sum()) == 0, "counters not back to zero"
    return out, lse, sm, sl, sa


@pytest.mark.parametrize("S", [1, 8, 32, 4096])
def test_single_row_fp32_full_size(rf, S):
    cfg = si.FULL["decode_f32"]
    q, K, V = si.decode_inputs(cfg["R"], cfg["L"], cfg["D"], torch.float32, seed=si.SEEDS["decode_f32"])
    scale = si.decode_scale(cfg["D"])
    out, lse, sm, sl, sa = run(rf, q, K, V, S, scale, torch.float32)
    ref, m, l = A.softmax_v_rows(f64(q), f64(K), f64(V), scale)
    assert_close_f32(f64(out), ref, f"out S={S}")
    assert_close_f32(f64(lse), m + np.log(l), f"lse S={S}")
    rm, rl, racc = A.segment_states(f64(q), f64(K), f64(V), scale, S)
    assert_states_close(f64(sm), f64(sl), f64(sa), rm, rl, racc, f"states S={S}")


@pytest.mark.parametrize("L,S", [(700, 1), (700, 5), (333, 16), (129, 1024)])
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_bf16_rows(rf, L, S, out_dtype):
    R, D = 6, 128
    q, K, V = si.decode_inputs(R, L, D, torch.bfloat16, seed=L + S)
    scale = si.decode_scale(D)
    out, lse, sm, sl, sa = run(rf, q, K, V, S, scale, out_dtype)
    ref, m, l = A.softmax_v_rows(f64(q), f64(K), f64(V), scale)
    if out_dtype == torch.float32:
        assert_close_f32(f64(out), ref, f"out L={L} S={S}")
    else:
        assert_close_bf16(f64(out), ref, f"out L={L} S={S}")
    assert_close_f32(f64(lse), m + np.log(l), f"lse L={L} S={S}")


def test_repeated_calls_reuse_counters_and_match_two_launches(rf):
    R, L, D, S = 12, 1000, 128, 7
    q, K, V = si.decode_inputs(R, L, D, torch.bfloat16, seed=77)
    scale = si.decode_scale(D)
    counters = torch.zeros(R, dtype=torch.int32, device="cuda")
    out, lse, sm, sl, sa = run(rf, q, K, V, S, scale, torch.bfloat16, counters=counters, calls=4)
    o2, l2, (m2, s2, a2) = rf.attn_decode(q.cuda(), K.cuda(), V.cuda(), S, scale, return_states=True)
    torch.cuda.synchronize()
    assert torch.equal(sm, m2) and torch.equal(sl, s2) and torch.equal(sa, a2), "states differ"
    assert torch.equal(out, o2), "output differs from rf_state_merge's"
    assert torch.allclose(lse, l2, rtol=1e-6, atol=1e-6), "lse differs from rf_state_merge's"
