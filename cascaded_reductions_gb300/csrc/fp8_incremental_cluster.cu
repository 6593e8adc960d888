// Incremental FP8 quantise-in-GEMM across a thread-block cluster: the same
// cascade as fp8_incremental.cu (RedFuser episode transcript, cue 33: the
// abs-max enters the GEMM as one multiplicative factor, so when the running
// abs-max grows the running accumulator is multiplied by the old abs-max over
// the new one), with the quantisation of X shared by the C CTAs that compute
// the same 128 rows of Y.
//
// Per row and K-tile of 128 columns, in order:
//   a' = max(a, max |x| over the tile),  s' = fp32(a' / 448)
//   if a > 0 and a' > a:  acc *= s / s'
//   codes = e4m3(fp32(x / s'))
//   acc += codes . Wq_tile^T
// and Y = bf16(acc * s_final * sw).
//
// A cluster of C CTAs (C = 8 or 4) covers C consecutive 512-column blocks of
// one 128-row block of Y.  CTA c of the cluster owns rows [c R, c R + R),
// R = 128 / C: it alone reads those rows of X, keeps their running abs-max,
// encodes them into its own A tile, and stores the codes and the rows'
// factors s / s' into the A tile of every other CTA of the cluster too
// (st.async into distributed shared memory, completing as transaction bytes
// on the receiving CTA's A barrier).  Each CTA thus quantises 1/C of the
// tile instead of all of it.
//
// One CTA per 128 x 512 block of Y; 512 TMEM columns hold the accumulator as
// two halves of 256 columns, so that one half is rescaled while the tensor
// core works on the other.
//   warp 0       TMA: e4m3 Wq tiles (two 256-row halves on one barrier,
//                2-tile ring);
//   warp 1       TMEM allocation and the MMAs (128x256x32, one half of the
//                accumulator at a time), committing A stages to every CTA of
//                the cluster;
//   warps 2-9    convert: 2C threads per owned row, each prefetching its own
//                part of the bf16 X band with cp.async several tiles ahead
//                (off the TMA unit, which the W tiles keep busy); running
//                abs-max, encode into a 4-stage ring of A tiles, every
//                thread storing its codes into all C of them; each warp
//                runs on without waiting for the others;
//   warps 10-25  rescale each accumulator half when a row's scale grew (a
//                warp whose 32 rows did not grow skips it), and the epilogue.
// Every barrier wait is bounded (see tc_common.cuh).  The CTAs of a cluster
// meet at a cluster barrier before any of them exits.  A CTA that consumed
// every tile has received every store and commit addressed to it; one whose
// waits gave up holds its shared memory a further 200 us after that barrier,
// so that stores issued before it land in memory that is still its own.

#include <cuda_bf16.h>

#include "e4m3.cuh"
#include "tc_common.cuh"

namespace rf {
namespace {

constexpr int BM = 128, BN = 512, BK = 128;
constexpr int A_STAGES = 4, W_STAGES = 4;
constexpr int W_BYTES = 256 * BK;             // one 256-row half of the Wq tile, e4m3
constexpr int A_BYTES = BM * BK;              // 16 KiB e4m3
constexpr int FIRST_CONV_WARP = 2;
constexpr int CONV_WARPS = 8, RESC_WARPS = 16;
constexpr int CONV_THREADS = CONV_WARPS * 32;
constexpr int FIRST_RESC_WARP = FIRST_CONV_WARP + CONV_WARPS;
constexpr int THREADS = (FIRST_RESC_WARP + RESC_WARPS) * 32;
constexpr int TMEM_COLS = 512;
constexpr float kRcp448 = 1.0f / 448.0f;      // RN(1/448), folded by the compiler

template <int C>
struct Cfg {
  static_assert(C == 4 || C == 8, "clusters of 4 or 8 CTAs");
  static constexpr int R = BM / C;            // rows this CTA converts
  static constexpr int P = CONV_THREADS / R;  // converter threads per row (2C)
  static constexpr int E = BK / P;            // columns per converter thread (64 / C)
  static constexpr int X_BYTES = R * BK * 2;  // one bf16 band (chunk u of thread ct at u * 4 KiB + ct * 16)
  static constexpr int X_STAGES = C == 8 ? 4 : 3;  // tiles of X in flight per thread
};

struct Shared {
  float2 fac[A_STAGES][BM];       // per A stage and row: {s / s' (1 if unchanged), s'}
  uint64_t w_full[W_STAGES / 2], w_empty[W_STAGES / 2];   // per tile slot (two half tiles)
  uint64_t a_full[A_STAGES];      // own band written + the other CTAs' bands stored in
  uint64_t a_empty[A_STAGES];     // one MMA commit from each CTA of the cluster
  uint64_t mma_done[2];           // per accumulator half
  uint64_t resc_done[2];          // per accumulator half: the rescale warps
  uint32_t tmem_base;
  int abort;
};

template <int C>
constexpr size_t smem_bytes() {
  return (size_t)W_STAGES * W_BYTES + (size_t)A_STAGES * A_BYTES +
         (size_t)Cfg<C>::X_STAGES * Cfg<C>::X_BYTES + sizeof(Shared) + 1024;
}
static_assert(smem_bytes<4>() <= 232448 && smem_bytes<8>() <= 232448,
              "exceeds the 227 KiB of shared memory a CTA may use");

// byte offset of 16-byte chunk `c` of row `r` in a 128-byte-swizzled tile
__device__ __forceinline__ uint32_t sw128(int r, int c) {
  return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

// a bounded wait whose outcome is the same for every lane of the warp
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  return __all_sync(0xffffffffu, tc::mbar_wait(bar, parity, abort));
}

// E bf16 values of one row (E / 8 16-byte chunks) -> E e4m3 codes
template <int E>
__device__ __forceinline__ void encode_row_part(const uint4 (&xv)[E / 8], float s, float rcp,
                                                uint2 (&codes)[E / 8]) {
#pragma unroll
  for (int u = 0; u < E / 8; ++u) {
    if (s == 0.f)
      codes[u] = make_uint2(0u, 0u);
    else if (fast_scale(s))
      codes[u] = encode8_x2(xv[u], s, rcp);
    else
      codes[u] = encode8_exact(xv[u], s);
  }
}

template <int C>
__global__ void __launch_bounds__(THREADS, 1)
fp8_incremental_cluster_kernel(const __nv_bfloat16* __restrict__ x,
                               const __grid_constant__ CUtensorMap tmW,
                               const float* __restrict__ sw, __nv_bfloat16* __restrict__ y,
                               float* __restrict__ sx_out, int M, int N, int K) {
  using G = Cfg<C>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sW = smem;
  uint8_t* sA = sW + W_STAGES * W_BYTES;
  uint8_t* sX = sA + A_STAGES * A_BYTES;
  Shared* sh = reinterpret_cast<Shared*>(sX + G::X_STAGES * G::X_BYTES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nblocks = N / BN;
  const int m0 = (int)(blockIdx.x / nblocks) * BM;
  const int n0 = (int)(blockIdx.x % nblocks) * BN;
  const int T = K / BK;
  const uint32_t crank = tc::cluster_ctarank();
  const int band0 = (int)crank * G::R;          // first row this CTA converts

  if (threadIdx.x == 0) {
    for (int s = 0; s < A_STAGES; ++s) {
      tc::mbar_init(&sh->a_full[s], CONV_WARPS);
      tc::mbar_init(&sh->a_empty[s], C);
    }
    for (int q = 0; q < W_STAGES / 2; ++q) {
      tc::mbar_init(&sh->w_full[q], 1);
      tc::mbar_init(&sh->w_empty[q], 1);
    }
    for (int h = 0; h < 2; ++h) {
      tc::mbar_init(&sh->mma_done[h], 1);
      tc::mbar_init(&sh->resc_done[h], RESC_WARPS);
    }
    sh->abort = 0;
    tc::fence_barrier_init();
  }
  if (warp == 1) tc::tmem_alloc(&sh->tmem_base, TMEM_COLS);
  tc::fence_before_sync();
  // every CTA's barriers are initialised before any copy or commit reaches them
  tc::cluster_sync();
  tc::fence_after_sync();
  const uint32_t tmem = sh->tmem_base;
  volatile int* abort = &sh->abort;

  if (warp == 0) {
    // ------------------------------------------------------ TMA ----
    if (lane == 0) {
      tc::prefetch_tmap(&tmW);
      for (int t = 0; t < T; ++t) {            // both 256-row halves of tile t on one barrier
        const int q = t % (W_STAGES / 2);
        if (!tc::mbar_wait(&sh->w_empty[q], ((uint32_t)(t / (W_STAGES / 2)) & 1u) ^ 1u, abort))
          break;
        tc::mbar_arrive_expect_tx(&sh->w_full[q], 2 * W_BYTES);
        tc::tma_load_2d(sW + (2 * q) * W_BYTES, &tmW, &sh->w_full[q], t * BK, n0);
        tc::tma_load_2d(sW + (2 * q + 1) * W_BYTES, &tmW, &sh->w_full[q], t * BK, n0 + 256);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------ MMA ----
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_e4m3_f32(BM, 256);
      constexpr uint16_t all_ctas = (uint16_t)((1u << C) - 1u);
      bool ok = true;
      for (int t = 0; t < T && ok; ++t) {
        const int s = t % A_STAGES;
        const uint32_t ph = (uint32_t)(t / A_STAGES) & 1u;
        if (!(ok = tc::mbar_wait(&sh->a_full[s], ph, abort))) break;
        // the other CTAs' codes were stored into this stage by st.async
        tc::fence_proxy_async_cta();
        const uint64_t a_desc = tc::sdesc_sw128(tc::smem_u32(sA + s * A_BYTES), 16, 1024);
        const int q = t % (W_STAGES / 2);
        if (!(ok = tc::mbar_wait(&sh->w_full[q], (uint32_t)(t / (W_STAGES / 2)) & 1u, abort))) break;
        for (int h = 0; h < 2; ++h) {
          // the rescale warps have brought this half up to the scale of tile t
          if (!(ok = tc::mbar_wait(&sh->resc_done[h], (uint32_t)t & 1u, abort))) break;
          tc::fence_after_sync();
          const uint64_t w_desc = tc::sdesc_sw128(tc::smem_u32(sW + (2 * q + h) * W_BYTES), 16, 1024);
#pragma unroll
          for (int kk = 0; kk < BK / 32; ++kk)
            tc::mma_f8f6f4_ss(tmem + (uint32_t)(h * 256), a_desc + (uint64_t)((kk * 32) >> 4),
                              w_desc + (uint64_t)((kk * 32) >> 4), idesc, (t | kk) != 0);
          tc::mma_commit(&sh->mma_done[h]);
          if (h == 1) tc::mma_commit(&sh->w_empty[q]);
        }
        if (!ok) break;
        // this CTA is done with A stage s: tell every converter of the cluster
        tc::mma_commit_multicast(&sh->a_empty[s], all_ctas);
      }
    }
  } else if (warp < FIRST_RESC_WARP) {
    // -------------------------------------------------------- convert ----
    const int ct = threadIdx.x - FIRST_CONV_WARP * 32;   // 0 .. CONV_THREADS-1
    const int br = ct / G::P;                    // row of this CTA's band
    const int j = ct % G::P;                     // part of the row
    const int col = j * G::E;                    // first column of the part
    const int row = band0 + br;                  // row of the 128-row block
    // this thread's E values of tile t: 16-byte chunk u at u * CONV_THREADS * 16
    // + ct * 16 of the stage (each LDS.128 of the warp reads 512 contiguous bytes)
    const __nv_bfloat16* xrow = x + (size_t)(m0 + row) * K + col;
    constexpr uint32_t BAND_BYTES = G::R * BK, FAC_BYTES = G::R * sizeof(float2);
    // shared::cluster address of this shared memory in the other CTAs, for
    // p = 1 .. C-1 (CTA crank + p mod C)
    const uint32_t base = tc::smem_u32(smem);
    uint32_t peer[C];
#pragma unroll
    for (int p = 1; p < C; ++p) peer[p] = tc::mapa(base, (crank + (uint32_t)p) % (uint32_t)C);
    auto load_x = [&](int t) {
      if (t < T) {
        uint8_t* dst = sX + (t % G::X_STAGES) * G::X_BYTES + ct * 16;
#pragma unroll
        for (int u = 0; u < G::E / 8; ++u)
          asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                           tc::smem_u32(dst + u * CONV_THREADS * 16)),
                       "l"(xrow + (size_t)t * BK + u * 8)
                       : "memory");
      }
      asm volatile("cp.async.commit_group;" ::: "memory");   // (empty past the end)
    };
    for (int t = 0; t < G::X_STAGES; ++t) load_x(t);
    float a = 0.f, s_cur = 0.f, rcp = 0.f;
    bool ok = T > 0;
    for (int t = 0; t < T && ok; ++t) {
      const int s = t % A_STAGES;
      const uint32_t ph = (uint32_t)(t / A_STAGES) & 1u;
      // this thread's copies of tile t are the oldest of X_STAGES groups
      asm volatile("cp.async.wait_group %0;" ::"n"(G::X_STAGES - 1) : "memory");
      bool good = true;
      {
        uint4 xv[G::E / 8];
        const uint8_t* xb = sX + (t % G::X_STAGES) * G::X_BYTES + ct * 16;
#pragma unroll
        for (int u = 0; u < G::E / 8; ++u)
          xv[u] = *reinterpret_cast<const uint4*>(xb + u * CONV_THREADS * 16);
        // abs-max of the part (packed bf16 pairs), then over the row's P threads
        uint32_t pk = 0u;
        const uint32_t mask = 0x7FFF7FFFu;
#pragma unroll
        for (int u = 0; u < G::E / 8; ++u) {
          asm("max.bf16x2 %0, %0, %1;" : "+r"(pk) : "r"(xv[u].x & mask));
          asm("max.bf16x2 %0, %0, %1;" : "+r"(pk) : "r"(xv[u].y & mask));
          asm("max.bf16x2 %0, %0, %1;" : "+r"(pk) : "r"(xv[u].z & mask));
          asm("max.bf16x2 %0, %0, %1;" : "+r"(pk) : "r"(xv[u].w & mask));
        }
        float tile_max = fmaxf(bf16_lo(pk), bf16_hi(pk));
#pragma unroll
        for (int o = G::P / 2; o >= 1; o >>= 1)
          tile_max = fmaxf(tile_max, __shfl_xor_sync(0xffffffffu, tile_max, o));
        const float a_new = fmaxf(a, tile_max);
        float factor = 1.f;
        if (a_new != a) {
          // fp32(a' / 448) and fp32(s / s'), correctly rounded (see e4m3.cuh)
          const float s_new =
              a_new >= 0x1p-80f ? quotient(a_new, 448.f, kRcp448) : __fdiv_rn(a_new, 448.f);
          rcp = fast_scale(s_new) ? __frcp_rn(s_new) : 0.f;
          if (a > 0.f)
            factor = fast_scale(s_new) && s_cur >= s_new * 0x1p-64f
                         ? quotient(s_cur, s_new, rcp)
                         : __fdiv_rn(s_cur, s_new);
          s_cur = s_new;
          a = a_new;
        }
        uint2 codes[G::E / 8];
        encode_row_part<G::E>(xv, s_cur, rcp, codes);
        // the values read from X stage t % X_STAGES are consumed: refill it
        load_x(t + G::X_STAGES);
        // A stage s is free once every CTA's MMAs of tile t - A_STAGES have read it
        good = warp_wait(&sh->a_empty[s], ph ^ 1u, abort);
        if (good) {
          uint8_t* ab = sA + s * A_BYTES;
          if constexpr (G::E == 8) {
            *reinterpret_cast<uint2*>(ab + sw128(row, col / 16) + col % 16) = codes[0];
          } else {
#pragma unroll
            for (int u = 0; u < G::E / 16; ++u)
              *reinterpret_cast<uint4*>(ab + sw128(row, col / 16 + u)) =
                  make_uint4(codes[2 * u].x, codes[2 * u].y, codes[2 * u + 1].x, codes[2 * u + 1].y);
          }
          if (j == 0) sh->fac[s][row] = make_float2(factor, s_cur);
          // the same codes and factors into the other CTAs' stage s
          const uint32_t code_off = tc::smem_u32(ab + sw128(row, col / 16) + col % 16) - base;
          const uint32_t fac_off = tc::smem_u32(&sh->fac[s][row]) - base;
          const uint32_t bar_off = tc::smem_u32(&sh->a_full[s]) - base;
#pragma unroll
          for (int p = 1; p < C; ++p) {
            if constexpr (G::E == 8)
              tc::st_async_v2(peer[p] + code_off, codes[0].x, codes[0].y, peer[p] + bar_off);
            else
              tc::st_async_v4(peer[p] + code_off,
                              make_uint4(codes[0].x, codes[0].y, codes[1].x, codes[1].y),
                              peer[p] + bar_off);
            if (j == 0)
              tc::st_async_v2(peer[p] + fac_off, __float_as_uint(factor), __float_as_uint(s_cur),
                              peer[p] + bar_off);
          }
        }
      }
      // this CTA's tensor core reads the band through the async proxy
      tc::fence_proxy_async_cta();
      __syncwarp();
      if (!(ok = good)) break;
      // one arrival per converter warp; the first also expects the other
      // CTAs' bands
      if (lane == 0) {
        if (warp == FIRST_CONV_WARP)
          tc::mbar_arrive_expect_tx(&sh->a_full[s],
                                    (uint32_t)(C - 1) * (BAND_BYTES + FAC_BYTES));
        else
          tc::mbar_arrive(&sh->a_full[s]);
      }
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");   // no copy outlives the loop
    // the last A_STAGES tiles' MMA commits of every CTA target this CTA's
    // a_empty barriers: let them land before the cluster barrier
    if (ok && ct == 0) {
      for (int t = (T >= A_STAGES ? T - A_STAGES : 0); t < T; ++t)
        if (!tc::mbar_wait(&sh->a_empty[t % A_STAGES], (uint32_t)(t / A_STAGES) & 1u, abort))
          break;
    }
  } else {
    // ------------------------------------------------ rescale + epilogue ----
    const int quarter = warp & 3, part = (warp - FIRST_RESC_WARP) >> 2;
    const int r = quarter * 32 + lane;           // accumulator row (TMEM lane)
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    bool ok = T > 0;
    for (int t = 0; t < T && ok; ++t) {
      const int s = t % A_STAGES;
      if (!(ok = warp_wait(&sh->a_full[s], (uint32_t)(t / A_STAGES) & 1u, abort))) break;
      const float factor = sh->fac[s][r].x;
      const bool grow = __any_sync(0xffffffffu, factor != 1.f);
      for (int h = 0; h < 2; ++h) {
        // the MMAs of tile t-1 on this half are done (waited every tile, so
        // that this arrival never runs two phases ahead of the MMA warp)
        if (t > 0 && !(ok = warp_wait(&sh->mma_done[h], (uint32_t)(t - 1) & 1u, abort)))
          break;
        if (t > 0 && grow) {
          tc::fence_after_sync();
#pragma unroll 1
          for (int c = 0; c < 2; ++c) {
            const uint32_t tcol = lane_base + (uint32_t)(h * 256 + part * 64 + c * 32);
            uint32_t v[32];
            tc::tmem_ld_32x32b_x32(tcol, v);
            tc::tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * factor);
            tc::tmem_st_32x32b_x32(tcol, v);
          }
          tc::tmem_st_wait();
        }
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&sh->resc_done[h]);
      }
    }
    // epilogue: Y = acc * s_final * sw, once both halves of the last tile are done
    if (ok && warp_wait(&sh->mma_done[0], (uint32_t)(T - 1) & 1u, abort) &&
        warp_wait(&sh->mma_done[1], (uint32_t)(T - 1) & 1u, abort)) {
      tc::fence_after_sync();
      const float s_fin = sh->fac[(T - 1) % A_STAGES][r].y;
      const int yrow = m0 + r;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        tc::tmem_ld_32x32b_x32(lane_base + (uint32_t)(part * 128 + c * 32), v);
        tc::tmem_ld_wait();
        const int col0 = n0 + part * 128 + c * 32;
        if (!RF_SPAN_OK(col0, 32, N) ||
            !RF_SPAN_OK((size_t)yrow * N + col0, 32, (long long)M * N))
          continue;                            // (checked build) sw and y spans
        uint32_t pk[16];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float4 s4 = __ldg(reinterpret_cast<const float4*>(sw + col0) + q);
          pk[2 * q] = pack_bf16x2(__uint_as_float(v[4 * q]) * s_fin * s4.x,
                                  __uint_as_float(v[4 * q + 1]) * s_fin * s4.y);
          pk[2 * q + 1] = pack_bf16x2(__uint_as_float(v[4 * q + 2]) * s_fin * s4.z,
                                      __uint_as_float(v[4 * q + 3]) * s_fin * s4.w);
        }
        uint4* dst = reinterpret_cast<uint4*>(y + (size_t)yrow * N + col0);
#pragma unroll
        for (int q = 0; q < 4; ++q)
          dst[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
      }
      if (part == 0 && n0 == 0 && sx_out != nullptr && RF_IDX_OK(yrow, M))
        sx_out[yrow] = s_fin;
    }
  }

  tc::fence_before_sync();
  __syncwarp();
  // no CTA leaves while another may still store into its shared memory
  tc::cluster_sync();
  if (warp == 1) {
    if (*abort) {
      // stores or commits issued before the other CTAs gave up may still be
      // on their way here: hold this CTA's shared memory for 200 us
      const unsigned long long t0 = tc::globaltimer_ns();
      while (tc::globaltimer_ns() - t0 < 200000ull) {
      }
    }
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, TMEM_COLS);
  }
}

template <int C>
cudaLaunchConfig_t cluster_config(cudaLaunchAttribute* attr, unsigned grid, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = smem_bytes<C>();
  cfg.stream = st;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

// How many clusters of C of these CTAs can be resident at once on the current
// device (0: none), queried once per device (up to 64); also sets the
// kernel's shared-memory attribute.
template <int C>
int resident_clusters() {
  static std::atomic<int> count[64];
  static std::atomic<uint64_t> attr_done{0}, known{0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  const uint64_t bit = 1ull << dev;
  if (known.load(std::memory_order_acquire) & bit) return count[dev].load();
  int n = 0;
  if (smem_attr(fp8_incremental_cluster_kernel<C>, smem_bytes<C>(), attr_done) == RF_OK) {
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = cluster_config<C>(attr, (unsigned)C, 0);
    if (cudaOccupancyMaxActiveClusters(&n, fp8_incremental_cluster_kernel<C>, &cfg) !=
        cudaSuccess)
      n = 0;
  }
  cudaGetLastError();
  count[dev].store(n);
  known.fetch_or(bit, std::memory_order_release);
  return n;
}

template <int C>
rf_status launch_c(const void* x, const uint8_t* wq, const float* sw, int M, int N, int K,
                   void* y, float* sx_final, cudaStream_t st) {
  CUtensorMap tw;
  if (!tc::make_tmap_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, wq, (uint64_t)K, (uint64_t)N,
                        (uint64_t)K, BK, 256, CU_TENSOR_MAP_SWIZZLE_128B))
    return RF_ERR_CUDA;
  const unsigned grid = (unsigned)(M / BM) * (unsigned)(N / BN);
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = cluster_config<C>(attr, grid, st);
  if (cudaLaunchKernelEx(&cfg, fp8_incremental_cluster_kernel<C>,
                         static_cast<const __nv_bfloat16*>(x), tw, sw,
                         static_cast<__nv_bfloat16*>(y), sx_final, M, N, K) != cudaSuccess) {
    cudaGetLastError();
    return RF_ERR_CUDA;
  }
  return launch_status();
}

}  // namespace

// Launches the cluster kernel when N / 512 is a multiple of 4 and such
// clusters fit on the device; returns RF_ERR_UNSUPPORTED otherwise, leaving
// the shape to the one-CTA kernel.  Of the cluster sizes that divide N / 512,
// the one whose grid runs in fewer waves of resident CTAs is taken (fewer 8-CTA
// clusters than 4-CTA ones fit on the GPU's processing clusters); on a tie,
// 8, which converts fewer rows per CTA.
rf_status launch_fp8_incremental_cluster(const void* x, const uint8_t* wq, const float* sw, int M,
                                         int N, int K, void* y, float* sx_final,
                                         cudaStream_t st) {
  const long long grid = (long long)(M / BM) * (N / BN);
  const int nblocks = N / BN;
  auto waves = [&](int c, int clusters) {
    return clusters > 0 ? (grid + (long long)c * clusters - 1) / ((long long)c * clusters) : -1;
  };
  const long long w8 = nblocks % 8 == 0 ? waves(8, resident_clusters<8>()) : -1;
  const long long w4 = nblocks % 4 == 0 ? waves(4, resident_clusters<4>()) : -1;
  if (w8 > 0 && (w4 <= 0 || w8 <= w4)) return launch_c<8>(x, wq, sw, M, N, K, y, sx_final, st);
  if (w4 > 0) return launch_c<4>(x, wq, sw, M, N, K, y, sx_final, st);
  return RF_ERR_UNSUPPORTED;
}

RF_TIMEOUT_WORD_OF_THIS_FILE

RF_BOUNDS_WORD_OF_THIS_FILE

}  // namespace rf
