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

__device__ __forceinline__ float absmax8(const uint4& u, float a) {
  a = fmaxf(a, fabsf(bf16_lo(u.x))); a = fmaxf(a, fabsf(bf16_hi(u.x)));
  a = fmaxf(a, fabsf(bf16_lo(u.y))); a = fmaxf(a, fabsf(bf16_hi(u.y)));
  a = fmaxf(a, fabsf(bf16_lo(u.z))); a = fmaxf(a, fabsf(bf16_hi(u.z)));
  a = fmaxf(a, fabsf(bf16_lo(u.w))); a = fmaxf(a, fabsf(bf16_hi(u.w)));
  return a;
}

// two floats -> two e4m3 codes (x0 in the low byte), RNE, saturating
__device__ __forceinline__ uint32_t e4m3x2(float x0, float x1) {
  return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(x0, x1), __NV_SATFINITE, __NV_E4M3);
}

// Per-row divisor: s, its correctly rounded reciprocal, and which path to use.
struct Divisor {
  float s, r;
  bool exact_path;   // tiny scale: IEEE division for every element
  bool zero;         // amax == 0: all codes zero
};

__device__ __forceinline__ Divisor make_divisor(float s) {
  Divisor d;
  d.s = s;
  d.zero = s == 0.f;
  d.exact_path = s < 0x1p-90f;
  d.r = d.exact_path ? 0.f : __frcp_rn(s);
  return d;
}

// correctly rounded x / s (see the file comment); the sign of a zero x is kept
__device__ __forceinline__ float quotient(float x, const Divisor& d) {
  if (d.exact_path) return __fdiv_rn(x, d.s);
  float q = x * d.r;
  q = fmaf(fmaf(-q, d.s, x), d.r, q);
  q = fmaf(fmaf(-q, d.s, x), d.r, q);
  return copysignf(q, x);
}

__device__ __forceinline__ uint2 encode8(const uint4& u, const Divisor& d) {
  if (d.zero) return make_uint2(0u, 0u);
  const uint32_t c0 = e4m3x2(quotient(bf16_lo(u.x), d), quotient(bf16_hi(u.x), d));
  const uint32_t c1 = e4m3x2(quotient(bf16_lo(u.y), d), quotient(bf16_hi(u.y), d));
  const uint32_t c2 = e4m3x2(quotient(bf16_lo(u.z), d), quotient(bf16_hi(u.z), d));
  const uint32_t c3 = e4m3x2(quotient(bf16_lo(u.w), d), quotient(bf16_hi(u.w), d));
  return make_uint2(c0 | (c1 << 16), c2 | (c3 << 16));
}

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
  uint4 r[VPT];
  float a = 0.f;
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int c = i * THREADS + threadIdx.x;
    if (c < K8) {
      r[i] = ld_stream_v4(x + base + c);
      a = absmax8(r[i], a);
    }
  }
  const float amax = block_max<THREADS>(a, red);
  const float s = __fdiv_rn(amax, 448.f);
  const Divisor d = make_divisor(s);
  if (threadIdx.x == 0) sx[blockIdx.x] = s;
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int c = i * THREADS + threadIdx.x;
    if (c < K8) xq[base + c] = encode8(r[i], d);
  }
}

// rows too long for the register-resident variant
template <int THREADS>
__global__ void __launch_bounds__(THREADS)
absmax_quant_long_kernel(const uint4* __restrict__ x, int K8, uint2* __restrict__ xq,
                         float* __restrict__ sx) {
  __shared__ float red[THREADS / 32];
  const size_t base = (size_t)blockIdx.x * K8;
  float a = 0.f;
  for (int c = threadIdx.x; c < K8; c += THREADS) a = absmax8(x[base + c], a);
  const float amax = block_max<THREADS>(a, red);
  const float s = __fdiv_rn(amax, 448.f);
  const Divisor d = make_divisor(s);
  if (threadIdx.x == 0) sx[blockIdx.x] = s;
  for (int c = threadIdx.x; c < K8; c += THREADS) xq[base + c] = encode8(x[base + c], d);
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
