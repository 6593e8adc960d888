// Incremental FP8 quantise-in-GEMM: the abs-max -> quantise -> GEMM cascade in
// one kernel, with the running abs-max rescaling the accumulator (RedFuser
// episode transcript, cue 33: the abs-max enters the GEMM as one
// multiplicative factor, so when the running abs-max grows the running
// accumulator is multiplied by the old abs-max over the new one).
//
// Per row and K-tile of 128 columns, in order:
//   a' = max(a, max |x| over the tile),  s' = fp32(a' / 448)
//   if a > 0 and a' > a:  acc *= s / s'            (TMEM rows, rescaled in place)
//   codes = e4m3(fp32(x / s'))                      (same rounding as the
//                                                    two-phase quantiser)
//   acc += codes . Wq_tile^T                        (tcgen05 kind::f8f6f4)
// and Y = bf16(acc * s_final * sw).  X is read as bf16 and never written out
// as codes; each CTA quantises its own rows (the quantisation work repeats
// once per 512-column block of Y).
//
// One CTA per 128 x 512 block of Y; 512 TMEM columns hold the fp32
// accumulator.
//   warp 0      TMA: bf16 X tiles (two 64-column boxes) and e4m3 Wq tiles
//               (two 256-row boxes), 128-byte swizzle, 2-stage rings;
//   warp 1      TMEM allocation and the MMAs (128x256x32, two per K-step);
//   warps 2-17  four threads per row (one per 32-column quarter of the
//               tile; sixteen warps give the latency-bound conversion enough
//               parallelism): partial abs-max, exchange with the other three
//               (bounded mbarrier per row quarter), running scale, quantise
//               into the swizzled A tile, rescale their quarter of the
//               accumulator row when the scale grew, and finally the epilogue.
// Every barrier wait is bounded (see tc_common.cuh).

#include <cuda_bf16.h>

#include "e4m3.cuh"
#include "tc_common.cuh"

namespace rf {
namespace {

constexpr int BM = 128, BN = 512, BK = 128;
constexpr int STAGES = 2;
constexpr int X_BYTES = BM * BK * 2;          // 32 KiB bf16 (two 16 KiB boxes)
constexpr int W_BYTES = BN * BK;              // 64 KiB e4m3 (two 32 KiB boxes)
constexpr int A_BYTES = BM * BK;              // 16 KiB e4m3
constexpr int PARTS = 4;                      // converter threads per row
constexpr int CONV_WARPS = 4 * PARTS;
constexpr int THREADS = (2 + CONV_WARPS) * 32;
constexpr int TMEM_COLS = 512;
constexpr float kRcp448 = 1.0f / 448.0f;      // RN(1/448), folded by the compiler

struct Shared {
  uint64_t x_full[STAGES], x_empty[STAGES];
  uint64_t w_full[STAGES], w_empty[STAGES];
  uint64_t a_full[STAGES], a_empty[STAGES];
  uint64_t pair[4];
  uint64_t pread[4];              // per row quarter: its PARTS warps have read pmax
  uint16_t pmax[PARTS][BM];       // partial abs-max of the current tile (a bf16 value)
  uint32_t tmem_base;
  int abort;
};

constexpr size_t SMEM_BYTES =
    (size_t)STAGES * (X_BYTES + W_BYTES + A_BYTES) + sizeof(Shared) + 1024;
static_assert(SMEM_BYTES <= 232448, "exceeds the 227 KiB of shared memory a CTA may use");

// byte offset of 16-byte chunk `c` of row `r` in a 128-byte-swizzled tile
__device__ __forceinline__ uint32_t sw128(int r, int c) {
  return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

__global__ void __launch_bounds__(THREADS, 1)
fp8_incremental_kernel(const __grid_constant__ CUtensorMap tmX,
                       const __grid_constant__ CUtensorMap tmW, const float* __restrict__ sw,
                       __nv_bfloat16* __restrict__ y, float* __restrict__ sx_out, int M, int N,
                       int K) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sW = smem;                                 // W stages first (32 KiB aligned halves)
  uint8_t* sX = sW + STAGES * W_BYTES;
  uint8_t* sA = sX + STAGES * X_BYTES;
  Shared* sh = reinterpret_cast<Shared*>(sA + STAGES * A_BYTES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nblocks = N / BN;
  const int m0 = (int)(blockIdx.x / nblocks) * BM;
  const int n0 = (int)(blockIdx.x % nblocks) * BN;
  const int T = K / BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      tc::mbar_init(&sh->x_full[s], 1);
      tc::mbar_init(&sh->x_empty[s], CONV_WARPS);
      tc::mbar_init(&sh->w_full[s], 1);
      tc::mbar_init(&sh->w_empty[s], 1);
      tc::mbar_init(&sh->a_full[s], CONV_WARPS);
      tc::mbar_init(&sh->a_empty[s], 1);
    }
    for (int q = 0; q < 4; ++q) {
      tc::mbar_init(&sh->pair[q], PARTS);
      tc::mbar_init(&sh->pread[q], PARTS);
    }
    sh->abort = 0;
    tc::fence_barrier_init();
  }
  if (warp == 1) tc::tmem_alloc(&sh->tmem_base, TMEM_COLS);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = sh->tmem_base;
  volatile int* abort = &sh->abort;

  if (warp == 0) {
    // ------------------------------------------------------ TMA ----
    if (lane == 0) {
      tc::prefetch_tmap(&tmX);
      tc::prefetch_tmap(&tmW);
      for (int t = 0; t < T; ++t) {
        const int s = t % STAGES;
        const uint32_t ph = (uint32_t)(t / STAGES) & 1u;
        if (!tc::mbar_wait(&sh->x_empty[s], ph ^ 1u, abort)) break;
        tc::mbar_arrive_expect_tx(&sh->x_full[s], X_BYTES);
        tc::tma_load_2d(sX + s * X_BYTES, &tmX, &sh->x_full[s], t * BK, m0);
        tc::tma_load_2d(sX + s * X_BYTES + X_BYTES / 2, &tmX, &sh->x_full[s], t * BK + 64, m0);
        if (!tc::mbar_wait(&sh->w_empty[s], ph ^ 1u, abort)) break;
        tc::mbar_arrive_expect_tx(&sh->w_full[s], W_BYTES);
        tc::tma_load_2d(sW + s * W_BYTES, &tmW, &sh->w_full[s], t * BK, n0);
        tc::tma_load_2d(sW + s * W_BYTES + W_BYTES / 2, &tmW, &sh->w_full[s], t * BK, n0 + 256);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------ MMA ----
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_e4m3_f32(BM, 256);
      for (int t = 0; t < T; ++t) {
        const int s = t % STAGES;
        const uint32_t ph = (uint32_t)(t / STAGES) & 1u;
        if (!tc::mbar_wait(&sh->a_full[s], ph, abort)) break;
        if (!tc::mbar_wait(&sh->w_full[s], ph, abort)) break;
        tc::fence_after_sync();
        const uint32_t a_addr = tc::smem_u32(sA + s * A_BYTES);
        const uint32_t w_addr = tc::smem_u32(sW + s * W_BYTES);
#pragma unroll
        for (int kk = 0; kk < BK / 32; ++kk) {
          const uint64_t ad = tc::sdesc_sw128(a_addr + (uint32_t)(kk * 32), 16, 1024);
#pragma unroll
          for (int nh = 0; nh < 2; ++nh)
            tc::mma_f8f6f4_ss(tmem + (uint32_t)(nh * 256), ad,
                              tc::sdesc_sw128(w_addr + (uint32_t)(nh * (W_BYTES / 2) + kk * 32), 16,
                                              1024),
                              idesc, (t | kk) != 0);
        }
        tc::mma_commit(&sh->a_empty[s]);
        tc::mma_commit(&sh->w_empty[s]);
      }
    }
  } else {
    // ------------------------------------------------ quantise + rescale ----
    const int quarter = warp & 3, part = (warp - 2) >> 2;
    const int r = quarter * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    float a = 0.f, s_cur = 0.f, rcp = 0.f;
    bool ok = T > 0;
    for (int t = 0; t < T && ok; ++t) {
      const int s = t % STAGES;
      const uint32_t ph = (uint32_t)(t / STAGES) & 1u;
      if (!tc::mbar_wait(&sh->x_full[s], ph, abort)) {
        ok = false;
        break;
      }
      // this thread's 32 bf16 values of row r: 16-byte chunks 4 (part % 2)
      // to 4 (part % 2) + 3 of box part / 2 of the X tile
      uint4 xv[4];
      const uint8_t* xb = sX + s * X_BYTES + (part >> 1) * (X_BYTES / 2);
#pragma unroll
      for (int c = 0; c < 4; ++c)
        xv[c] = *reinterpret_cast<const uint4*>(xb + sw128(r, (part & 1) * 4 + c));
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&sh->x_empty[s]);
      // partial abs-max (packed bf16 pairs, two chains), then the other parts'
      uint32_t pk0 = 0u, pk1 = 0u;
      const uint32_t mask = 0x7FFF7FFFu;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        asm("max.bf16x2 %0, %0, %1;" : "+r"(pk0) : "r"(xv[c].x & mask));
        asm("max.bf16x2 %0, %0, %1;" : "+r"(pk1) : "r"(xv[c].y & mask));
        asm("max.bf16x2 %0, %0, %1;" : "+r"(pk0) : "r"(xv[c].z & mask));
        asm("max.bf16x2 %0, %0, %1;" : "+r"(pk1) : "r"(xv[c].w & mask));
      }
      asm("max.bf16x2 %0, %0, %1;" : "+r"(pk0) : "r"(pk1));
      const float pm = fmaxf(bf16_lo(pk0), bf16_hi(pk0));  // a bf16 value: exact in 16 bits
      // one pmax buffer: the other parts must have read the previous tile's
      if (t > 0 && !tc::mbar_wait(&sh->pread[quarter], (uint32_t)(t - 1) & 1u, abort)) {
        ok = false;
        break;
      }
      sh->pmax[part][r] = (uint16_t)(__float_as_uint(pm) >> 16);
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&sh->pair[quarter]);
      if (!tc::mbar_wait(&sh->pair[quarter], (uint32_t)t & 1u, abort)) {
        ok = false;
        break;
      }
      float tile_max = pm;
#pragma unroll
      for (int q = 0; q < PARTS; ++q)
        tile_max = fmaxf(tile_max, __uint_as_float((uint32_t)sh->pmax[q][r] << 16));
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&sh->pread[quarter]);
      const float a_new = fmaxf(a, tile_max);
      // running scale; the accumulator is rescaled by s / s' when it grows
      float factor = 1.f;
      const bool grow = a > 0.f && a_new > a;
      if (a_new != a) {
        // fp32(a' / 448) and fp32(s / s'), correctly rounded: the reciprocal
        // and two residual corrections (see e4m3.cuh) where no residual can
        // underflow, IEEE division otherwise
        const float s_new =
            a_new >= 0x1p-80f ? quotient(a_new, 448.f, kRcp448) : __fdiv_rn(a_new, 448.f);
        rcp = fast_scale(s_new) ? __frcp_rn(s_new) : 0.f;
        if (grow)
          factor = fast_scale(s_new) && s_cur >= s_new * 0x1p-64f ? quotient(s_cur, s_new, rcp)
                                                                  : __fdiv_rn(s_cur, s_new);
        s_cur = s_new;
        a = a_new;
      }
      // the A stage is free once the MMAs two tiles back have read it
      if (!tc::mbar_wait(&sh->a_empty[s], ph ^ 1u, abort)) {
        ok = false;
        break;
      }
      uint8_t* ab = sA + s * A_BYTES;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        uint2 lo, hi;
        if (s_cur == 0.f) {
          lo = hi = make_uint2(0u, 0u);
        } else if (fast_scale(s_cur)) {
          lo = encode8_x2(xv[2 * j], s_cur, rcp);
          hi = encode8_x2(xv[2 * j + 1], s_cur, rcp);
        } else {
          lo = encode8_exact(xv[2 * j], s_cur);
          hi = encode8_exact(xv[2 * j + 1], s_cur);
        }
        *reinterpret_cast<uint4*>(ab + sw128(r, 2 * part + j)) = make_uint4(lo.x, lo.y, hi.x, hi.y);
      }
      // make the generic-proxy stores visible to the tensor core
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      // a grown scale rescales the accumulator, which must then hold every
      // earlier tile: wait for the MMAs of tile t-1 (the A stage they read is
      // released when they finish).  Otherwise tile t is handed over at once
      // and its MMAs queue behind those of tile t-1.
      if (t > 0 && __any_sync(0xffffffffu, grow)) {
        const int sp = (t - 1) % STAGES;
        if (!tc::mbar_wait(&sh->a_empty[sp], (uint32_t)((t - 1) / STAGES) & 1u, abort)) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        // this thread's 128 accumulator columns, 32 at a time (two loads in
        // flight cost a register spill)
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          const uint32_t col = lane_base + (uint32_t)(part * 128 + c * 32);
          uint32_t v[32];
          tc::tmem_ld_32x32b_x32(col, v);
          tc::tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * factor);
          tc::tmem_st_32x32b_x32(col, v);
        }
        tc::tmem_st_wait();
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&sh->a_full[s]);
    }
    // epilogue: Y = acc * s_final * sw
    // every MMA has finished once the last tile's A stage is released
    if (ok && tc::mbar_wait(&sh->a_empty[(T - 1) % STAGES], (uint32_t)((T - 1) / STAGES) & 1u,
                            abort)) {
      tc::fence_after_sync();
      const int row = m0 + r;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        tc::tmem_ld_32x32b_x32(lane_base + (uint32_t)(part * 128 + c * 32), v);
        tc::tmem_ld_wait();
        const int col0 = n0 + part * 128 + c * 32;
        if (!RF_SPAN_OK(col0, 32, N) || !RF_SPAN_OK((size_t)row * N + col0, 32, (long long)M * N))
          continue;                            // (checked build) sw and y spans
        uint32_t p[16];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float4 s4 = __ldg(reinterpret_cast<const float4*>(sw + col0) + j);
          p[2 * j] = pack_bf16x2(__uint_as_float(v[4 * j]) * s_cur * s4.x,
                                 __uint_as_float(v[4 * j + 1]) * s_cur * s4.y);
          p[2 * j + 1] = pack_bf16x2(__uint_as_float(v[4 * j + 2]) * s_cur * s4.z,
                                     __uint_as_float(v[4 * j + 3]) * s_cur * s4.w);
        }
        uint4* dst = reinterpret_cast<uint4*>(y + (size_t)row * N + col0);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          dst[j] = make_uint4(p[4 * j], p[4 * j + 1], p[4 * j + 2], p[4 * j + 3]);
      }
      if (part == 0 && n0 == 0 && sx_out != nullptr && RF_IDX_OK(row, M)) sx_out[row] = s_cur;
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace

rf_status launch_fp8_incremental(const void* x, const uint8_t* wq, const float* sw, int M, int N,
                                 int K, void* y, float* sx_final, cudaStream_t st) {
  CUtensorMap tx, tw;
  if (!tc::make_tmap_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, (uint64_t)K, (uint64_t)M,
                        (uint64_t)K * 2, 64, BM, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !tc::make_tmap_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, wq, (uint64_t)K, (uint64_t)N,
                        (uint64_t)K, BK, 256, CU_TENSOR_MAP_SWIZZLE_128B))
    return RF_ERR_CUDA;
  static std::atomic<uint64_t> attr{0};
  if (smem_attr(fp8_incremental_kernel, SMEM_BYTES, attr) != RF_OK) return RF_ERR_CUDA;
  const unsigned grid = (unsigned)(M / BM) * (unsigned)(N / BN);
  fp8_incremental_kernel<<<grid, THREADS, SMEM_BYTES, st>>>(
      tx, tw, sw, static_cast<__nv_bfloat16*>(y), sx_final, M, N, K);
  return launch_status();
}

RF_TIMEOUT_WORD_OF_THIS_FILE

RF_BOUNDS_WORD_OF_THIS_FILE

}  // namespace rf
