"""Every cascade under CUDA-graph capture: the calls are captured once on
torch's capture stream, then the graph is replayed on new inputs written
into the same device buffers, and each replay is checked against the
oracle.  This is how a serving loop drives the library (fixed buffers, one
graph launch per step): it requires that no call synchronises, allocates or
reads the inputs on the host, and that nothing of a call depends on the
values it saw at capture time.  Each call is made once before capture (the
per-device setup of the tensor-core kernels, the shared-memory opt-in and
the driver entry point lookup, happens on a first call)."""

import numpy as np
import pytest
import torch

from helpers import assert_close_bf16, assert_close_f32, f64
from oracle import attention as A
from oracle import bf16 as obf16
from oracle import fp8 as ofp8
from oracle import mla as M
from oracle import routing as Rt
import synthetic_inputs as si

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rf():
    import cascaded_reductions_gb300 as m
    return m


def capture(fn):
    fn()                                   # first call outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def replay(rf, g):
    g.replay()
    torch.cuda.synchronize()
    assert rf.rf_device_error() == 0


def test_decode_split_and_merge(rf):
    R, L, D, S = 6, 700, 128, 5
    q = torch.empty(R, D, dtype=torch.bfloat16, device="cuda")
    K = torch.empty(R, L, D, dtype=torch.bfloat16, device="cuda")
    V = torch.empty_like(K)
    sm = torch.empty(R, S, device="cuda")
    sl = torch.empty(R, S, device="cuda")
    sa = torch.empty(R, S, D, device="cuda")
    out = torch.empty(R, D, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(R, device="cuda")
    scale = si.decode_scale(D)

    def step():
        rf.rf_attn_decode_split(q, K, V, S, scale, sm, sl, sa)
        rf.rf_state_merge(sm, sl, sa, out, lse)

    for i, seed in enumerate((41, 42, 43)):
        hq, hK, hV = si.decode_inputs(R, L, D, torch.bfloat16, seed=seed)
        q.copy_(hq)
        K.copy_(hK)
        V.copy_(hV)
        if i == 0:
            g = capture(step)
        replay(rf, g)
        ref, m, l = A.softmax_v_rows(f64(hq), f64(hK), f64(hV), scale)
        assert_close_bf16(f64(out), ref, f"decode replay {i}")
        assert_close_f32(f64(lse), m + np.log(l), f"decode lse replay {i}")


def test_decode_noalloc(rf):
    R, L, D, S = 4, 333, 64, 3
    q = torch.empty(R, D, device="cuda")
    K = torch.empty(R, L, D, device="cuda")
    V = torch.empty_like(K)
    out = torch.empty(R, D, device="cuda")
    scale = si.decode_scale(D)
    step = lambda: rf.rf_attn_decode_noalloc(q, K, V, S, scale, out)
    for i, seed in enumerate((51, 52)):
        hq, hK, hV = si.decode_inputs(R, L, D, torch.float32, seed=seed)
        q.copy_(hq)
        K.copy_(hK)
        V.copy_(hV)
        if i == 0:
            g = capture(step)
        replay(rf, g)
        ref, _, _ = A.softmax_v_rows(f64(hq), f64(hK), f64(hV), scale)
        assert_close_f32(f64(out), ref, f"no-alloc replay {i}")


def test_routing(rf):
    T, E, k = 300, 256, 8
    x = torch.empty(T, E, device="cuda")
    idx = torch.empty(T, k, dtype=torch.int32, device="cuda")
    w = torch.empty(T, k, device="cuda")
    step = lambda: rf.rf_softmax_topk(x, k, True, idx, w)
    for i, seed in enumerate((61, 62)):
        hx = si.routing_logits(T, E, seed=seed)
        x.copy_(hx)
        if i == 0:
            g = capture(step)
        replay(rf, g)
        ridx, rw = Rt.softmax_topk(hx.numpy(), k, True)
        assert np.array_equal(idx.cpu().numpy(), ridx), f"routing indices, replay {i}"
        assert_close_f32(w.cpu().numpy(), rw, f"routing weights, replay {i}")


def test_quant_gemm(rf):
    Mq, Kq, Nq = 256, 1024, 384
    x = torch.empty(Mq, Kq, dtype=torch.bfloat16, device="cuda")
    wq = torch.empty(Nq, Kq, dtype=torch.uint8, device="cuda")
    sw = torch.empty(Nq, device="cuda")
    xq = torch.empty(Mq, Kq, dtype=torch.uint8, device="cuda")
    sx = torch.empty(Mq, device="cuda")
    y = torch.empty(Mq, Nq, dtype=torch.bfloat16, device="cuda")
    step = lambda: rf.rf_absmax_quant_fp8_gemm(x, wq, sw, xq, sx, y)
    for i, seed in enumerate((71, 72)):
        hx, hwq, hsw = si.quant_gemm_inputs(Mq, Kq, Nq, seed=seed)
        x.copy_(hx)
        wq.copy_(hwq)
        sw.copy_(hsw)
        if i == 0:
            g = capture(step)
        replay(rf, g)
        rq, rs = ofp8.absmax_quant(obf16.decode(hx.view(torch.int16).numpy()))
        assert np.array_equal(xq.cpu().numpy(), rq), f"codes, replay {i}"
        assert np.array_equal(sx.cpu().numpy(), rs), f"scales, replay {i}"
        assert_close_bf16(f64(y), ofp8.scaled_gemm(rq, rs, hwq.numpy(), hsw.numpy()), f"Y, replay {i}")


@pytest.mark.parametrize("Nq", [512, 2048])
def test_incremental_quant_gemm(rf, Nq):
    # N = 2048 runs the cluster kernel (a cluster launch with distributed
    # shared memory inside the graph), N = 512 the one-CTA kernel
    Mq, Kq = 128, 768
    x = torch.empty(Mq, Kq, dtype=torch.bfloat16, device="cuda")
    wq = torch.empty(Nq, Kq, dtype=torch.uint8, device="cuda")
    sw = torch.empty(Nq, device="cuda")
    sx = torch.empty(Mq, device="cuda")
    y = torch.empty(Mq, Nq, dtype=torch.bfloat16, device="cuda")
    step = lambda: rf.rf_incremental_quant_fp8_gemm(x, wq, sw, y, sx)
    for i, seed in enumerate((73, 74)):
        hx, hwq, hsw = si.quant_gemm_inputs(Mq, Kq, Nq, seed=seed)
        x.copy_(hx)
        wq.copy_(hwq)
        sw.copy_(hsw)
        if i == 0:
            g = capture(step)
        replay(rf, g)
        ry, rs = ofp8.incremental_quant_gemm(obf16.decode(hx.view(torch.int16).numpy()),
                                             hwq.numpy(), hsw.numpy())
        assert np.array_equal(sx.cpu().numpy(), rs), f"final scales, replay {i}"
        assert_close_bf16(f64(y), ry, f"Y, replay {i}")


def test_prefill(rf):
    B, H, N, D = 1, 2, 300, 128
    q = torch.empty(B, H, N, D, dtype=torch.bfloat16, device="cuda")
    k = torch.empty_like(q)
    v = torch.empty_like(q)
    out = torch.empty_like(q)
    lse = torch.empty(B, H, N, device="cuda")
    scale = D ** -0.5
    step = lambda: rf.rf_attn_prefill(q, k, v, True, scale, out, lse)
    for i, seed in enumerate((81, 82)):
        hq, hk, hv = si.prefill_inputs(B, H, N, D, seed=seed)
        q.copy_(hq)
        k.copy_(hk)
        v.copy_(hv)
        if i == 0:
            g = capture(step)
        replay(rf, g)
        for h in range(H):
            ro, rl = A.causal_attention(f64(hq[0, h]), f64(hk[0, h]), f64(hv[0, h]), scale, True)
            assert_close_bf16(f64(out[0, h]), ro, f"prefill out h={h}, replay {i}")
            assert_close_f32(f64(lse[0, h]), rl, f"prefill lse h={h}, replay {i}")


def test_mla_split_and_merge(rf):
    B, H, L, S, DK, DV = 2, 16, 500, 3, 576, 512
    q = torch.empty(B, H, DK, dtype=torch.bfloat16, device="cuda")
    C = torch.empty(B, L, DK, dtype=torch.bfloat16, device="cuda")
    sm = torch.empty(B, H, S, device="cuda")
    sl = torch.empty(B, H, S, device="cuda")
    sa = torch.empty(B, H, S, DV, device="cuda")
    out = torch.empty(B * H, DV, dtype=torch.bfloat16, device="cuda")
    scale = si.mla_scale()

    def step():
        rf.rf_mla_decode_split(q, C, S, scale, sm, sl, sa)
        rf.rf_state_merge(sm.view(B * H, S), sl.view(B * H, S), sa.view(B * H, S, DV), out)

    for i, seed in enumerate((91, 92)):
        hq, hC = si.mla_inputs(B, H, L, DK, seed=seed)
        q.copy_(hq)
        C.copy_(hC)
        if i == 0:
            g = capture(step)
        replay(rf, g)
        ro, _, _ = M.mla_decode(f64(hq), f64(hC), DV, scale)
        assert_close_bf16(f64(out).reshape(ro.shape), ro, f"MLA replay {i}")
