"""Failure detection on the GPU without a fault: a bounded wait is made to run
out (a barrier that nothing arrives on) and the status comes back to the
host; the context stays usable for the next call."""

import numpy as np
import pytest
import torch

from helpers import assert_close_bf16, f64
from oracle import attention as A
import synthetic_inputs as si

pytestmark = pytest.mark.gpu

def test_bounded_wait_reports_timeout_and_context_survives():
    import cascaded_reductions_gb300 as rf
    assert rf.rf_device_error() == 0
    waited = torch.zeros(1, dtype=torch.int32, device="cuda")
    rf.rf_selftest_wait_timeout(waited)
    torch.cuda.synchronize()
    assert rf.rf_device_error() == rf.RF_ERR_TIMEOUT
    assert rf.rf_device_error() == 0                  # read and cleared
    ms = int(waited.item())
    assert 900 <= ms <= 10000, f"the wait lasted {ms} ms"
    # the next call on the same context still computes the right thing
    q, K, V = si.decode_inputs(4, 300, 128, torch.bfloat16, seed=12)
    out, lse = rf.attn_decode(q.cuda(), K.cuda(), V.cuda(), 3, si.decode_scale(128))
    torch.cuda.synchronize()
    ref, m, l = A.softmax_v_rows(f64(q), f64(K), f64(V), si.decode_scale(128))
    assert_close_bf16(f64(out), ref, "decode after a timeout")
    assert rf.rf_device_error() == 0
