"""Calls from several host threads on several CUDA streams at once.  The C
ABI promises thread-safe, stream-ordered calls with no per-call global
state: the one-time set-up (driver entry point, per-device shared-memory
opt-in) is guarded, and each call touches only its own buffers.  Here two
threads issue different cascades on their own streams, repeatedly and
interleaved (from a cold start of each kernel when this file runs alone),
and every result is checked against the oracle."""

import threading

import numpy as np
import pytest
import torch

from helpers import assert_close_bf16, assert_close_f32, f64
from oracle import attention as A
from oracle import routing as Rt
import synthetic_inputs as si

pytestmark = pytest.mark.gpu


def test_two_threads_two_streams():
    import cascaded_reductions_gb300 as rf
    B, H, N, D = 1, 2, 257, 128
    pq, pk, pv = si.prefill_inputs(B, H, N, D, seed=101)
    R, L, DD, S = 5, 900, 128, 4
    dq, dK, dV = si.decode_inputs(R, L, DD, torch.bfloat16, seed=102)
    x = si.routing_logits(200, 128, seed=103)
    results, errors = {}, []

    def prefill_worker():
        try:
            st = torch.cuda.Stream()
            with torch.cuda.stream(st):
                q, k, v = pq.cuda(), pk.cuda(), pv.cuda()
                outs = []
                for _ in range(4):
                    out = torch.empty_like(q)
                    lse = torch.empty(B, H, N, device="cuda")
                    rf.rf_attn_prefill(q, k, v, True, D ** -0.5, out, lse, stream=st)
                    outs.append((out, lse))
                st.synchronize()
                results["prefill"] = [(f64(o), f64(l)) for o, l in outs]
        except Exception as e:          # reported below, never hidden
            errors.append(e)

    def decode_routing_worker():
        try:
            st = torch.cuda.Stream()
            with torch.cuda.stream(st):
                q, K, V, xx = dq.cuda(), dK.cuda(), dV.cuda(), x.cuda()
                got = []
                for _ in range(4):
                    out, lse = rf.attn_decode(q, K, V, S, si.decode_scale(DD), stream=st)
                    idx, w = rf.softmax_topk(xx, 8, True, stream=st)
                    got.append((out, lse, idx, w))
                st.synchronize()
                results["decode"] = [(f64(o), f64(l), i.cpu().numpy(), w.cpu().numpy())
                                     for o, l, i, w in got]
        except Exception as e:
            errors.append(e)

    threads = [threading.Thread(target=prefill_worker), threading.Thread(target=decode_routing_worker)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=300)
    assert not any(t.is_alive() for t in threads), "a worker did not finish"
    assert not errors, errors
    assert rf.rf_device_error() == 0

    for out, lse in results["prefill"]:
        for h in range(H):
            ro, rl = A.causal_attention(f64(pq[0, h]), f64(pk[0, h]), f64(pv[0, h]), D ** -0.5, True)
            assert_close_bf16(out[0, h], ro, f"prefill h={h}")
            assert_close_f32(lse[0, h], rl, f"prefill lse h={h}")
    ref, m, l = A.softmax_v_rows(f64(dq), f64(dK), f64(dV), si.decode_scale(DD))
    ridx, rw = Rt.softmax_topk(x.numpy(), 8, True)
    for out, lse, idx, w in results["decode"]:
        assert_close_bf16(out, ref, "decode")
        assert_close_f32(lse, m + np.log(l), "decode lse")
        assert np.array_equal(idx, ridx), "routing indices"
        assert_close_f32(w, rw, "routing weights")
