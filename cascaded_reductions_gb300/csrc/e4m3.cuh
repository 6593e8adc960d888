// e4m3 encoding of x / s with the rounding the FP8 cascade fixes: the
// correctly rounded fp32 quotient, then round-to-nearest-even e4m3 with
// saturation at +-448.  The quotient comes from the correctly rounded
// reciprocal r = 1/s and two residual corrections q' = q + (x - q s) r, each
// residual exact in one fma; by Markstein's theorem (P. Markstein, IBM J. Res.
// Dev. 34(1), 1990: a faithful quotient corrected once with the correctly
// rounded reciprocal is the correctly rounded quotient) the result equals
// IEEE division.  Scales below 2^-90 take IEEE division per element so that
// no residual underflows where it matters.
#pragma once

#include <cuda_fp8.h>

#include "common.cuh"

namespace rf {

// two floats -> two e4m3 codes (x0 in the low byte), RNE, saturating
__device__ __forceinline__ uint32_t e4m3x2(float x0, float x1) {
  return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(x0, x1), __NV_SATFINITE, __NV_E4M3);
}

// correctly rounded x / s from r = RN(1/s) (see the file comment); the sign
// of a zero x is kept
__device__ __forceinline__ float quotient(float x, float s, float r) {
  float q = x * r;
  q = fmaf(fmaf(-q, s, x), r, q);
  q = fmaf(fmaf(-q, s, x), r, q);
  return copysignf(q, x);
}

__device__ __forceinline__ uint2 encode8(const uint4& u, float s, float r) {
  const uint32_t c0 = e4m3x2(quotient(bf16_lo(u.x), s, r), quotient(bf16_hi(u.x), s, r));
  const uint32_t c1 = e4m3x2(quotient(bf16_lo(u.y), s, r), quotient(bf16_hi(u.y), s, r));
  const uint32_t c2 = e4m3x2(quotient(bf16_lo(u.z), s, r), quotient(bf16_hi(u.z), s, r));
  const uint32_t c3 = e4m3x2(quotient(bf16_lo(u.w), s, r), quotient(bf16_hi(u.w), s, r));
  return make_uint2(c0 | (c1 << 16), c2 | (c3 << 16));
}

// The same quotients two at a time with the packed fp32x2 multiply and fma of
// sm_100+: each half of a packed operation is rounded exactly as the scalar
// one, so the codes are those of encode8, in half the instructions.
__device__ __forceinline__ uint64_t f32x2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ uint32_t e4m3x2_quotients(uint64_t x, uint64_t neg_s, uint64_t r) {
  uint64_t q, e;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(q) : "l"(x), "l"(r));
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(e) : "l"(q), "l"(neg_s), "l"(x));
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(q) : "l"(e), "l"(r), "l"(q));
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(e) : "l"(q), "l"(neg_s), "l"(x));
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(q) : "l"(e), "l"(r), "l"(q));
  q |= x & 0x8000000080000000ull;      // q has x's sign except when it is +0: copysign
  float q0, q1;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(q0), "=f"(q1) : "l"(q));
  return e4m3x2(q0, q1);
}

__device__ __forceinline__ uint2 encode8_x2(const uint4& u, float s, float r) {
  const uint64_t ns = f32x2_pack(-s, -s), rr = f32x2_pack(r, r);
  const uint32_t c0 = e4m3x2_quotients(f32x2_pack(bf16_lo(u.x), bf16_hi(u.x)), ns, rr);
  const uint32_t c1 = e4m3x2_quotients(f32x2_pack(bf16_lo(u.y), bf16_hi(u.y)), ns, rr);
  const uint32_t c2 = e4m3x2_quotients(f32x2_pack(bf16_lo(u.z), bf16_hi(u.z)), ns, rr);
  const uint32_t c3 = e4m3x2_quotients(f32x2_pack(bf16_lo(u.w), bf16_hi(u.w)), ns, rr);
  return make_uint2(c0 | (c1 << 16), c2 | (c3 << 16));
}

// rows with a tiny (or zero) scale: IEEE division per element, or zero codes
static __device__ __noinline__ uint2 encode8_exact(uint4 u, float s) {
  if (s == 0.f) return make_uint2(0u, 0u);
  const uint32_t c0 = e4m3x2(__fdiv_rn(bf16_lo(u.x), s), __fdiv_rn(bf16_hi(u.x), s));
  const uint32_t c1 = e4m3x2(__fdiv_rn(bf16_lo(u.y), s), __fdiv_rn(bf16_hi(u.y), s));
  const uint32_t c2 = e4m3x2(__fdiv_rn(bf16_lo(u.z), s), __fdiv_rn(bf16_hi(u.z), s));
  const uint32_t c3 = e4m3x2(__fdiv_rn(bf16_lo(u.w), s), __fdiv_rn(bf16_hi(u.w), s));
  return make_uint2(c0 | (c1 << 16), c2 | (c3 << 16));
}

// the reciprocal-and-correction path is valid for scales of 2^-90 and up
__device__ __forceinline__ bool fast_scale(float s) { return s >= 0x1p-90f; }

}  // namespace rf
