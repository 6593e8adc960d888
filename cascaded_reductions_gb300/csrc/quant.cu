// FP8 per-token quantisation, phase 1 of the abs-max -> quantise -> GEMM
// cascade (RedFuser episode transcript, cue 33).
//
// One CTA per row.  The row is read from HBM once into registers (each thread
// holds VPT 16-byte chunks = 8*VPT bf16 values), the abs-max is reduced across
// the CTA (warp shuffles, then one shared-memory step), and the same
// registers are encoded: sx = amax / 448 (IEEE fp32 division), code =
// e4m3(x / sx) with the hardware's round-to-nearest-even saturating convert.
// The element step is the correctly rounded fp32 quotient x / sx (not x times
// a rounded reciprocal, which can flip codes), so every code is the one the
// definition gives.  The quotient comes from the row's correctly rounded
// reciprocal r = 1/sx and two residual corrections q' = q + (x - q sx) r, each
// residual exact in one fma; by Markstein's theorem (P. Markstein, IBM J. Res.
// Dev. 34(1), 1990: a faithful quotient corrected once with the correctly
// rounded reciprocal is the correctly rounded quotient) the result equals
// IEEE division.  Rows whose scale is below 2^-90 use the library's IEEE
// division instead, so no residual can underflow where it matters (a quotient
// below 2^-10 encodes to zero whatever its last bits).  A row with amax = 0
// writes sx = 0 and zero codes.
// Rows longer than the register budget use a two-pass variant that reads
// the row a second time (from L2).

#include <cuda_fp8.h>
#include <math.h>

#include "common.cuh"

namespace rf {
namespace {

// running |x| maximum of 8 bf16 values, kept as a packed bf16x2 pair
// (the maximum of bf16 magnitudes is exact in bf16)
__device__ __forceinline__ uint32_t absmax8(const uint4& u, uint32_t a) {
  const uint32_t m = 0x7FFF7FFFu;
  uint32_t r;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(u.x & m), "r"(u.y & m));
  asm("max.bf16x2 %0, %0, %1;" : "+r"(r) : "r"(u.z & m));
  asm("max.bf16x2 %0, %0, %1;" : "+r"(r) : "r"(u.w & m));
  asm("max.bf16x2 %0, %0, %1;" : "+r"(r) : "r"(a));
  return r;
}

__device__ __forceinline__ float absmax_value(uint32_t pair) {
  return fmaxf(bf16_lo(pair), bf16_hi(pair));
}

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

// rows with a tiny (or zero) scale: IEEE division per element, or zero codes
__device__ __noinline__ uint2 encode8_exact(uint4 u, float s) {
  if (s == 0.f) return make_uint2(0u, 0u);
  const uint32_t c0 = e4m3x2(__fdiv_rn(bf16_lo(u.x), s), __fdiv_rn(bf16_hi(u.x), s));
  const uint32_t c1 = e4m3x2(__fdiv_rn(bf16_lo(u.y), s), __fdiv_rn(bf16_hi(u.y), s));
  const uint32_t c2 = e4m3x2(__fdiv_rn(bf16_lo(u.z), s), __fdiv_rn(bf16_hi(u.z), s));
  const uint32_t c3 = e4m3x2(__fdiv_rn(bf16_lo(u.w), s), __fdiv_rn(bf16_hi(u.w), s));
  return make_uint2(c0 | (c1 << 16), c2 | (c3 << 16));
}

// the reciprocal-and-correction path is valid for scales of 2^-90 and up
__device__ __forceinline__ bool fast_scale(float s) { return s >= 0x1p-90f; }

template <int THREADS>
__device__ __forceinline__ float block_max(float a, float* red) {
  a = group_max<32>(a);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) red[warp] = a;
  __syncthreads();
  float r = 0.f;
#pragma unroll
  for (int w = 0; w < THREADS / 32; ++w) r = fmaxf(r, red[w]);
  return r;
}

template <int THREADS, int VPT>
__global__ void __launch_bounds__(THREADS)
absmax_quant_kernel(const uint4* __restrict__ x, int K8, uint2* __restrict__ xq,
                    float* __restrict__ sx) {
  __shared__ float red[THREADS / 32];
  const size_t base = (size_t)blockIdx.x * K8;
  uint4 v[VPT];
  uint32_t a = 0u;
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int c = i * THREADS + threadIdx.x;
    if (c < K8) {
      v[i] = ld_stream_v4(x + base + c);
      a = absmax8(v[i], a);
    }
  }
  const float amax = block_max<THREADS>(absmax_value(a), red);
  const float s = __fdiv_rn(amax, 448.f);
  if (threadIdx.x == 0) sx[blockIdx.x] = s;
  if (fast_scale(s)) {
    const float r = __frcp_rn(s);
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int c = i * THREADS + threadIdx.x;
      if (c < K8) xq[base + c] = encode8(v[i], s, r);
    }
  } else {
#pragma unroll 1
    for (int i = 0; i < VPT; ++i) {
      const int c = i * THREADS + threadIdx.x;
      if (c < K8) xq[base + c] = encode8_exact(v[i], s);
    }
  }
}

// rows too long for the register-resident variant
template <int THREADS>
__global__ void __launch_bounds__(THREADS)
absmax_quant_long_kernel(const uint4* __restrict__ x, int K8, uint2* __restrict__ xq,
                         float* __restrict__ sx) {
  __shared__ float red[THREADS / 32];
  const size_t base = (size_t)blockIdx.x * K8;
  uint32_t a = 0u;
  for (int c = threadIdx.x; c < K8; c += THREADS) a = absmax8(x[base + c], a);
  const float amax = block_max<THREADS>(absmax_value(a), red);
  const float s = __fdiv_rn(amax, 448.f);
  if (threadIdx.x == 0) sx[blockIdx.x] = s;
  if (fast_scale(s)) {
    const float r = __frcp_rn(s);
    for (int c = threadIdx.x; c < K8; c += THREADS) xq[base + c] = encode8(x[base + c], s, r);
  } else {
    for (int c = threadIdx.x; c < K8; c += THREADS) xq[base + c] = encode8_exact(x[base + c], s);
  }
}

}  // namespace

rf_status launch_absmax_quant(const void* x, int M, int K, uint8_t* xq, float* sx,
                              cudaStream_t st) {
  const int K8 = K / 8;
  const auto* xv = static_cast<const uint4*>(x);
  auto* qv = reinterpret_cast<uint2*>(xq);
  constexpr int TH = 128;
  const int vpt = (K8 + TH - 1) / TH;
  const unsigned grid = (unsigned)M;
#define RF_QUANT_CASE(V) \
  case V: absmax_quant_kernel<TH, V><<<grid, TH, 0, st>>>(xv, K8, qv, sx); break;
  switch (vpt) {
    RF_QUANT_CASE(1) RF_QUANT_CASE(2) RF_QUANT_CASE(3) RF_QUANT_CASE(4)
    RF_QUANT_CASE(5) RF_QUANT_CASE(6) RF_QUANT_CASE(7) RF_QUANT_CASE(8)
    RF_QUANT_CASE(9) RF_QUANT_CASE(10) RF_QUANT_CASE(11) RF_QUANT_CASE(12)
    RF_QUANT_CASE(13) RF_QUANT_CASE(14) RF_QUANT_CASE(15) RF_QUANT_CASE(16)
    default:
      absmax_quant_long_kernel<256><<<grid, 256, 0, st>>>(xv, K8, qv, sx);
  }
#undef RF_QUANT_CASE
  return launch_status();
}

}  // namespace rf
