"""Parity of multi-latent attention decode (rf_mla_decode_split +
rf_state_merge) with the oracle, through the C ABI.

Tolerances: the merged output is bf16 (2e-2 absolute + 1e-2 relative).  The
segment states are fp32 intermediates whose weights p pass through bf16 on
their way into the tensor-core product, and l sums those same rounded
weights, so they are held to: the segment max to fp32 rounding of the scores,
l to bf16's unit roundoff (each weight is within 2^-8 of its exact value, so
the sum is within 2^-8 relative), and each state's normalised partial output
acc / l to the bf16 output tolerance.

Cases: ragged key counts and tiles, every segment count from 1 to past L
(identity states), head counts 16 / 32 / 48 / 64 / 128 (one and several head
groups), several units per CTA crossing sequence boundaries, scores large
enough to move the running max many times, and the full-size workload
(B=64, H=16, L=32768, S=16, 2.4 GB of latent cache) on sampled sequences in
the launch configuration the benchmark times.
"""

import numpy as np
import pytest
import torch

from helpers import assert_close_bf16, assert_close_f32, f64
from oracle import attention as A
from oracle import mla as M
import synthetic_inputs as si

pytestmark = pytest.mark.gpu

DK, DV = 576, 512


@pytest.fixture(scope="module")
def rf():
    import cascaded_reductions_gb300 as m
    return m


def run(rf, q, C, S, scale):
    out, lse, (sm, sl, sa) = rf.mla_decode(q.cuda(), C.cuda(), S, scale, return_states=True)
    torch.cuda.synchronize()
    assert rf.rf_device_error() == 0
    return out, lse, sm, sl, sa


def check_states(gm, gl, ga, rm, rl, racc, what):
    gm, gl, ga = f64(gm), f64(gl), f64(ga)
    empty = np.isneginf(rm)
    assert np.array_equal(np.isneginf(gm), empty), f"{what}: identity states differ"
    assert np.all(gl[empty] == 0) and np.all(ga[empty] == 0), f"{what}: identity state not zero"
    live = ~empty
    assert np.all(np.abs(gm[live] - rm[live]) <= 1e-5 * (1 + np.abs(rm[live]))), f"{what}: max"
    err_l = np.abs(gl[live] - rl[live])
    assert np.all(err_l <= 2.0 ** -8 * rl[live] + 1e-6), f"{what} l: worst {(err_l / rl[live]).max()}"

    assert_close_bf16(ga[live] / gl[live][:, None], racc[live] / rl[live][:, None],
                      what + " acc/l")


def check(rf, B, H, L, S, scale, seed, C=None):
    q, C0 = si.mla_inputs(B, H, L, DK, seed=seed)
    C = C0 if C is None else C
    out, lse, sm, sl, sa = run(rf, q, C, S, scale)
    ro, rm, rl = M.mla_decode(f64(q), f64(C), DV, scale)
    assert_close_bf16(f64(out), ro, f"out B={B} H={H} L={L} S={S}")
    assert_close_f32(f64(lse), rm + np.log(rl), f"lse B={B} H={H} L={L} S={S}")
    em, el, ea = M.mla_segment_states(f64(q), f64(C), DV, scale, S)
    check_states(sm, sl, sa, em, el, ea, f"states B={B} H={H} L={L} S={S}")


@pytest.mark.parametrize("S", [1, 2, 3, 5, 8, 16])
def test_ragged_segments(rf, S):
    # L = 1000: 7 full tiles and a tail of 104 keys; segments cut tiles anywhere
    check(rf, 2, 16, 1000, S, si.mla_scale(), seed=60 + S)


@pytest.mark.parametrize("L", [1, 77, 128, 129, 255, 513])
def test_short_sequences(rf, L):
    check(rf, 3, 16, L, 2, si.mla_scale(), seed=70 + L)


def test_more_segments_than_keys(rf):
    # ceil(5 / 8) = 1 key per segment: segments 5..7 are empty (identity states)
    check(rf, 2, 16, 5, 8, si.mla_scale(), seed=80)


@pytest.mark.parametrize("H", [32, 48, 64, 128])
def test_head_groups(rf, H):
    check(rf, 2, H, 700, 3, si.mla_scale(), seed=90 + H)


def test_head_groups_with_empty_segments(rf):
    # several head groups (units dealt round-robin) and segments past the end
    check(rf, 3, 64, 5, 8, si.mla_scale(), seed=94)


def test_units_cross_sequences(rf):
    # 40 sequences x 8 segments = 320 units over the SMs: several units per
    # CTA, the query block reloaded where the sequence changes
    check(rf, 40, 16, 600, 8, si.mla_scale(), seed=95)


@pytest.mark.parametrize("scale", [0.5, 2.0])
def test_running_max_moves(rf, scale):
    # scores of tens of log2 units: the reference max moves tile after tile
    # and the accumulator columns are rescaled in tensor memory
    check(rf, 2, 16, 2048, 2, scale, seed=97)


def test_rising_scores(rf):
    # keys that grow along the sequence: every tile raises the max
    B, H, L = 1, 16, 3000
    q, C = si.mla_inputs(B, H, L, DK, seed=98)
    ramp = torch.linspace(0.2, 4.0, L)[None, :, None]
    C = (C.float() * ramp).to(torch.bfloat16)
    check(rf, B, H, L, 1, si.mla_scale(), seed=98, C=C)


def test_full_size_sampled():
    import cascaded_reductions_gb300 as rf
    cfg = si.FULL["mla"]
    B, H, L = cfg["B"], cfg["H"], cfg["L"]
    S = 16
    q, C = si.mla_inputs(B, H, L, DK, seed=si.SEEDS["mla"], device="cuda")
    out, lse = rf.mla_decode(q, C, S, si.mla_scale())
    torch.cuda.synchronize()
    assert rf.rf_device_error() == 0
    for b in (0, 17, B - 1):
        ro, rm, rl = M.mla_decode(f64(q[b:b + 1]), f64(C[b:b + 1]), DV, si.mla_scale())
        assert_close_bf16(f64(out[b:b + 1]), ro, f"full-size out b={b}")
        assert_close_f32(f64(lse[b:b + 1]), rm + np.log(rl), f"full-size lse b={b}")
    assert torch.isfinite(out.float()).all()
