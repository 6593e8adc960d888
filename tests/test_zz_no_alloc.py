"""rf_attn_decode_noalloc, the decode entry point for callers that cannot
allocate device memory (an engine plugin without an allocator, a serving loop
that cannot afford cudaMalloc's device-wide synchronisation, a fixed memory
budget).  It keeps the segment states in the library's own fixed 16 MiB device
array instead of caller buffers.

Through the C ABI, its output must agree with the oracle's softmax(q K^T
scale) V and log-sum-exp, and with the regular path (rf_attn_decode_split
into caller buffers, then rf_state_merge), within the tolerances the other
tests use, on two calls in a row: the second call is smaller than the first,
so part of the shared array still holds the first call's states and must not
leak into the result.  A request whose states do
not fit in the array is refused before anything is launched.

This file is named to be collected last, so a run that stops at the first
failure has run every other test before it.
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


def regular(rf, q, K, V, S, scale, out_dtype):
    return rf.attn_decode(q, K, V, S, scale, out_dtype=out_dtype)


def noalloc(rf, q, K, V, S, scale, out_dtype):
    R, L, D = K.shape
    out = torch.empty(R, D, dtype=out_dtype, device="cuda")
    lse = torch.empty(R, dtype=torch.float32, device="cuda")
    rf.rf_attn_decode_noalloc(q, K, V, S, scale, out, lse)
    return out, lse


def test_noalloc_matches_regular_path_twice(rf):
    # call 1: 64 rows x 16 segments of bf16 D=128 (about 0.5 MiB of states)
    q, K, V = (t.cuda() for t in si.decode_inputs(64, 3001, 128, torch.bfloat16, seed=41))
    scale = si.decode_scale(128)
    ref_out, ref_lse = regular(rf, q, K, V, 16, scale, torch.bfloat16)
    out, lse = noalloc(rf, q, K, V, 16, scale, torch.bfloat16)
    torch.cuda.synchronize()
    oracle_out, m, l = A.softmax_v_rows(f64(q), f64(K), f64(V), scale)
    assert_close_bf16(f64(out), oracle_out, "first call out vs oracle")
    assert_close_f32(f64(lse), m + np.log(l), "first call lse vs oracle")
    assert_close_bf16(f64(out), f64(ref_out), "first call out")
    assert_close_f32(f64(lse), f64(ref_lse), "first call lse")

    # call 2, right after: fewer rows, more segments than keys (identity
    # states), fp32 output; the array still holds call 1's states
    q2, K2, V2 = (t.cuda() for t in si.decode_inputs(8, 40, 128, torch.bfloat16, seed=42))
    ref_out2, ref_lse2 = regular(rf, q2, K2, V2, 64, scale, torch.float32)
    out2, lse2 = noalloc(rf, q2, K2, V2, 64, scale, torch.float32)
    torch.cuda.synchronize()
    oracle_out2, m2, l2 = A.softmax_v_rows(f64(q2), f64(K2), f64(V2), scale)
    assert_close_f32(f64(out2), oracle_out2, "second call out vs oracle")
    assert_close_f32(f64(lse2), m2 + np.log(l2), "second call lse vs oracle")
    assert_close_f32(f64(out2), f64(ref_out2), "second call out")
    assert_close_f32(f64(lse2), f64(ref_lse2), "second call lse")


def test_noalloc_fp32_single_row(rf):
    q, K, V = (t.cuda() for t in si.decode_inputs(1, 4096, 64, torch.float32, seed=1))
    scale = si.decode_scale(64)
    for _ in range(2):
        ref_out, ref_lse = regular(rf, q, K, V, 32, scale, torch.float32)
        out, lse = noalloc(rf, q, K, V, 32, scale, torch.float32)
        torch.cuda.synchronize()
        oracle_out, m, l = A.softmax_v_rows(f64(q), f64(K), f64(V), scale)
        assert_close_f32(f64(out), oracle_out, "fp32 out vs oracle")
        assert_close_f32(f64(lse), m + np.log(l), "fp32 lse vs oracle")
        assert_close_f32(f64(out), f64(ref_out), "fp32 out")
        assert_close_f32(f64(lse), f64(ref_lse), "fp32 lse")


def test_noalloc_refuses_states_larger_than_its_array(rf):
    # 1024 rows x 64 segments x (128 + 2) floats = 34 MB > 16 MiB
    q = torch.zeros(1024, 128, dtype=torch.bfloat16, device="cuda")
    K = torch.zeros(1024, 8, 128, dtype=torch.bfloat16, device="cuda")
    out = torch.empty(1024, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(rf.RFError) as e:
        rf.rf_attn_decode_noalloc(q, K, K, 64, 0.1, out)
    assert e.value.status == rf.RF_ERR_UNSUPPORTED
