"""bfloat16 codec for the oracle (its own, written from the format definition).

bfloat16 is the upper half of an IEEE-754 binary32: 1 sign bit, 8 exponent
bits, 7 stored mantissa bits.  Widening to float32 appends 16 zero bits, so it
is exact.  Narrowing rounds to nearest, ties to even.

The pages fix no output precision; bf16 outputs follow the workload
descriptions (bf16 q/K/V and bf16 outputs for split-KV decode and prefill, bf16
Y for the FP8 GEMM).
"""

import numpy as np


def decode(bits):
    """uint16/int16 bit patterns -> float64 values (exact)."""
    b = np.asarray(bits).astype(np.uint16).astype(np.uint32) << np.uint32(16)
    with np.errstate(invalid="ignore"):     # NaN payloads widen to NaN
        return b.view(np.float32).astype(np.float64)


def encode_from_f32(x):
    """float32 values -> uint16 bfloat16 bit patterns, round-to-nearest-even.

    NaN maps to a quiet NaN (0x7FC0 with the input's sign).
    """
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    lower = u & np.uint64(0xFFFF)
    upper = u >> np.uint64(16)
    half = np.uint64(0x8000)
    # Round up when the dropped half is above one half, or exactly one half
    # and the kept part is odd.
    up = (lower > half) | ((lower == half) & ((upper & np.uint64(1)) == np.uint64(1)))
    out = (upper + up.astype(np.uint64)).astype(np.uint32)
    nan = np.isnan(f)
    out = np.where(nan, (upper & np.uint64(0x8000)).astype(np.uint32) | np.uint32(0x7FC0), out)
    return out.astype(np.uint16)
