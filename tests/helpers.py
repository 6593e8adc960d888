"""Shared test helpers: tolerances and tensor conversion.  No cascade arithmetic."""

import numpy as np
import torch

# fp32 outputs: |g - r| <= 2e-3 |r| + 1e-6 (the small absolute term covers
# outputs that happen to sit near zero)
F32_RTOL, F32_ATOL = 2e-3, 1e-6
# bf16 outputs: |g - r| <= 2e-2 + 1e-2 |r|
BF16_RTOL, BF16_ATOL = 1e-2, 2e-2


def f64(t):
    """torch tensor (any float dtype, any device) -> float64 numpy (exact widening)."""
    return t.detach().to("cpu").to(torch.float64).numpy()


def assert_close_f32(got, ref, what=""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.abs(got - ref)
    bound = F32_RTOL * np.abs(ref) + F32_ATOL
    bad = ~(err <= bound)
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside fp32 tolerance; "
                             f"first at {tuple(i)}: got {got[tuple(i)]!r} ref {ref[tuple(i)]!r}")


def assert_close_bf16(got, ref, what=""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.abs(got - ref)
    bound = BF16_ATOL + BF16_RTOL * np.abs(ref)
    bad = ~(err <= bound)
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside bf16 tolerance; "
                             f"first at {tuple(i)}: got {got[tuple(i)]!r} ref {ref[tuple(i)]!r}")


def assert_states_close(gm, gl, gacc, rm, rl, racc, what=""):
    """Segment states agree: same max (to fp32 rounding of the scores), and l,
    acc agree once both are expressed relative to the oracle's max."""
    gm, gl, gacc = (np.asarray(a, np.float64) for a in (gm, gl, gacc))
    empty = np.isneginf(rm)
    assert np.array_equal(np.isneginf(gm), empty), f"{what}: identity states differ"
    assert np.all(gl[empty] == 0) and np.all(gacc[empty] == 0), f"{what}: identity state not zero"
    live = ~empty
    dm = gm[live] - rm[live]
    assert np.all(np.abs(dm) <= 1e-5 * (1 + np.abs(rm[live]))), f"{what}: max differs, worst {np.abs(dm).max()}"
    f = np.exp(gm - np.where(live, rm, 0.0))
    f[empty] = 0
    assert_close_f32(gl[live] * f[live], rl[live], what + " l")
    scaled = gacc * f[..., None]
    err = np.abs(scaled - racc)
    bound = 2e-3 * np.abs(racc) + 1e-5 * rl[..., None]
    bad = ~(err <= bound)
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what} acc: {int(bad.sum())} outside tolerance; first at {tuple(i)}: "
                             f"got {scaled[tuple(i)]!r} ref {racc[tuple(i)]!r}")
