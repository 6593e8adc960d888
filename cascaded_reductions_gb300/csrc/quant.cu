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
#include "e4m3.cuh"

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
    if (c < K8 && RF_IDX_OK(base + c, (long long)gridDim.x * K8)) {   // M = gridDim.x rows of K8 chunks
      v[i] = ld_stream_v4(x + base + c);
      a = absmax8(v[i], a);
    }
  }
  const float amax = block_max<THREADS>(absmax_value(a), red);
  const float s = __fdiv_rn(amax, 448.f);
  if (threadIdx.x == 0 && RF_IDX_OK(blockIdx.x, gridDim.x)) sx[blockIdx.x] = s;
  if (fast_scale(s)) {
    const float r = __frcp_rn(s);
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int c = i * THREADS + threadIdx.x;
      if (c < K8 && RF_IDX_OK(base + c, (long long)gridDim.x * K8)) xq[base + c] = encode8_x2(v[i], s, r);
    }
  } else {
#pragma unroll 1
    for (int i = 0; i < VPT; ++i) {
      const int c = i * THREADS + threadIdx.x;
      if (c < K8 && RF_IDX_OK(base + c, (long long)gridDim.x * K8)) xq[base + c] = encode8_exact(v[i], s);
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
  for (int c = threadIdx.x; c < K8; c += THREADS)
    if (RF_IDX_OK(base + c, (long long)gridDim.x * K8)) a = absmax8(x[base + c], a);
  const float amax = block_max<THREADS>(absmax_value(a), red);
  const float s = __fdiv_rn(amax, 448.f);
  if (threadIdx.x == 0 && RF_IDX_OK(blockIdx.x, gridDim.x)) sx[blockIdx.x] = s;
  if (fast_scale(s)) {
    const float r = __frcp_rn(s);
    for (int c = threadIdx.x; c < K8; c += THREADS)
      if (RF_IDX_OK(base + c, (long long)gridDim.x * K8)) xq[base + c] = encode8_x2(x[base + c], s, r);
  } else {
    for (int c = threadIdx.x; c < K8; c += THREADS)
      if (RF_IDX_OK(base + c, (long long)gridDim.x * K8)) xq[base + c] = encode8_exact(x[base + c], s);
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

RF_BOUNDS_WORD_OF_THIS_FILE

}  // namespace rf
