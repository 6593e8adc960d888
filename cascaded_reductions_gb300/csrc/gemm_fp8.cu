// FP8 GEMM with a per-row x per-column scale epilogue: phase 2 of the
// abs-max -> quantise -> GEMM cascade (RedFuser episode transcript, cue 33;
// cue 5: every GEMM output is a sum reduction along K).
//
//   Y[m, n] = bf16( (sum_k dec(Xq[m,k]) dec(Wq[n,k])) * sx[m] * sw[n] )
//
// Persistent, warp-specialised tcgen05 kernel, one CTA per SM:
//   warp 0      TMA producer: 128x128-byte tiles of Xq and 256x128-byte tiles
//               of Wq (128-byte swizzle) into a 4-stage shared-memory ring;
//   warp 1      allocates 512 TMEM columns (two 128x256 fp32 accumulators)
//               and issues tcgen05.mma kind::f8f6f4 (M=128, N=256, K=32) from
//               one thread, committing each stage back to the producer and
//               each finished accumulator to the epilogue;
//   warps 2-5   epilogue: tcgen05.ld of the accumulator (each thread one
//               row, 32 columns at a time), scale by sx[row] * sw[col],
//               round to bf16, store; then hand the accumulator back, so the
//               next tile's MMAs overlap this tile's epilogue.
// Output tiles are 128 x 256; CTAs walk work items t = blockIdx.x + i*gridDim.x.
// When the tiles left after the whole waves fit into one wave as halves,
// those tiles run as 128 x 128 halves (N = 128 MMAs), so the last wave is a
// half-tile wave rather than a sparse whole-tile one.
// Every barrier wait is bounded (see tc_common.cuh).

#include <cuda_bf16.h>

#include "tc_common.cuh"

namespace rf {
namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 128;                       // bytes = e4m3 elements per stage
constexpr int UMMA_K = 32;                    // K of one kind::f8f6f4 MMA
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK;              // 16 KiB
constexpr int B_BYTES = BN * BK;              // 32 KiB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int TMEM_COLS = 2 * BN;             // two accumulators
constexpr int THREADS = 192;

struct Shared {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint32_t tmem_base;
  int abort;
};

constexpr size_t SMEM_BYTES = (size_t)STAGES * STAGE_BYTES + sizeof(Shared) + 1024;
static_assert(SMEM_BYTES <= 232448, "exceeds the 227 KiB of shared memory a CTA may use");

__global__ void __launch_bounds__(THREADS, 1)
fp8_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmBh, const float* __restrict__ sx,
                const float* __restrict__ sw, __nv_bfloat16* __restrict__ y, int M, int N, int K,
                int full_items, int num_items) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  Shared* sh = reinterpret_cast<Shared*>(smem + (size_t)STAGES * STAGE_BYTES);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // ragged edges: the tensor maps zero-fill rows past M / N and columns past
  // K (an e4m3 zero adds nothing), the epilogue masks what it stores
  const int tiles_n = (N + BN - 1) / BN;
  const int num_k = (K + BK - 1) / BK;
  // work item i: a 128 x 256 tile for i < full_items, else half of one of
  // the remaining tiles (128 x 128), so the last wave is a half-tile wave
  auto item = [&](int i, int& tm, int& col0, int& width) {
    int tile = i, half = 0;
    width = BN;
    if (i >= full_items) {
      tile = full_items + ((i - full_items) >> 1);
      half = (i - full_items) & 1;
      width = BN / 2;
    }
    tm = tile / tiles_n;
    col0 = (tile - tm * tiles_n) * BN + half * (BN / 2);
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      tc::mbar_init(&sh->full[s], 1);
      tc::mbar_init(&sh->empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&sh->acc_full[b], 1);
      tc::mbar_init(&sh->acc_empty[b], 4);
    }
    sh->abort = 0;
    tc::fence_barrier_init();
    tc::prefetch_tmap(&tmA);
    tc::prefetch_tmap(&tmB);
    tc::prefetch_tmap(&tmBh);
  }
  if (warp == 1) tc::tmem_alloc(&sh->tmem_base, TMEM_COLS);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = sh->tmem_base;
  volatile int* abort = &sh->abort;

  if (warp == 0) {
    // ------------------------------------------------ TMA producer ----
    if (lane == 0) {
      uint32_t it = 0;
      for (int i = blockIdx.x; i < num_items && !*abort; i += gridDim.x) {
        int tm, col0, width;
        item(i, tm, col0, width);
        const bool half = width != BN;
        for (int kb = 0; kb < num_k; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1u;
          if (!tc::mbar_wait(&sh->empty[s], ph ^ 1u, abort)) break;
          uint8_t* a = smem + (size_t)s * STAGE_BYTES;
          tc::mbar_arrive_expect_tx(&sh->full[s], half ? A_BYTES + B_BYTES / 2 : STAGE_BYTES);
          tc::tma_load_2d(a, &tmA, &sh->full[s], kb * BK, tm * BM);
          tc::tma_load_2d(a + A_BYTES, half ? &tmBh : &tmB, &sh->full[s], kb * BK, col0);
        }
      }
      // On an abort, let the copies already issued land before the CTA exits.
      if (*abort) {
        for (int s = 0; s < STAGES; ++s) {
          const unsigned long long t0 = tc::globaltimer_ns();
          while (!tc::mbar_try_wait(&sh->full[s], 0) && !tc::mbar_try_wait(&sh->full[s], 1) &&
                 tc::globaltimer_ns() - t0 < tc::kWaitLimitNs) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer ----
    if (lane == 0) {
      constexpr uint32_t idesc_full = tc::idesc_e4m3_f32(BM, BN);
      constexpr uint32_t idesc_half = tc::idesc_e4m3_f32(BM, BN / 2);
      uint32_t it = 0, t = 0;
      for (int i = blockIdx.x; i < num_items && !*abort; i += gridDim.x, ++t) {
        const uint32_t idesc = i < full_items ? idesc_full : idesc_half;
        const int buf = t & 1;
        const uint32_t bph = (t >> 1) & 1u;
        if (!tc::mbar_wait(&sh->acc_empty[buf], bph ^ 1u, abort)) break;
        tc::fence_after_sync();
        const uint32_t d = tmem + (uint32_t)(buf * BN);
        bool ok = true;
        for (int kb = 0; kb < num_k; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1u;
          if (!tc::mbar_wait(&sh->full[s], ph, abort)) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint32_t a = tc::smem_u32(smem + (size_t)s * STAGE_BYTES);
          const uint64_t adesc = tc::sdesc_sw128(a, 16, 1024);
          const uint64_t bdesc = tc::sdesc_sw128(a + A_BYTES, 16, 1024);
#pragma unroll
          for (int k = 0; k < BK / UMMA_K; ++k) {
            // advance the start address by k*32 bytes inside the swizzle atom
            tc::mma_f8f6f4_ss(d, adesc + (uint64_t)(k * UMMA_K / 16), bdesc + (uint64_t)(k * UMMA_K / 16),
                              idesc, (kb | k) != 0);
          }
          tc::mma_commit(&sh->empty[s]);
        }
        if (!ok) break;
        tc::mma_commit(&sh->acc_full[buf]);
      }
    }
  } else {
    // ------------------------------------------------ epilogue ----
    const int quarter = warp & 3;              // TMEM lanes this warp may access
    const int r = quarter * 32 + lane;         // row within the tile
    uint32_t t = 0;
    for (int i = blockIdx.x; i < num_items; i += gridDim.x, ++t) {
      const int buf = t & 1;
      const uint32_t bph = (t >> 1) & 1u;
      if (!tc::mbar_wait(&sh->acc_full[buf], bph, abort)) break;
      tc::fence_after_sync();
      int tm, tcol0, width;
      item(i, tm, tcol0, width);
      const int row = tm * BM + r;
      const bool row_in = row < M;
      const float srow = row_in && RF_IDX_OK(row, M) ? sx[row] : 0.f;
      __nv_bfloat16* yrow = y + (size_t)(row_in ? row : 0) * N;
      const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(buf * BN);
#pragma unroll 1
      for (int c = 0; c < width / 32; ++c) {
        const int col0 = tcol0 + c * 32;
        uint32_t v[32];
        tc::tmem_ld_32x32b_x32(taddr + (uint32_t)(c * 32), v);   // whole warp, every row
        tc::tmem_ld_wait();
        if (!row_in || col0 >= N) continue;
        if (col0 + 32 <= N && (N & 7) == 0) {
          // whole 32-column chunk, 16-byte aligned row: vector loads and stores
          if (!RF_SPAN_OK(col0, 32, N) || !RF_SPAN_OK((size_t)row * N + col0, 32, (long long)M * N))
            continue;                          // (checked build) sw and y spans
          const float4* swv = reinterpret_cast<const float4*>(sw + col0);
          uint32_t p[16];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float4 s4 = __ldg(swv + j);
            p[2 * j] = pack_bf16x2(__uint_as_float(v[4 * j]) * srow * s4.x,
                                   __uint_as_float(v[4 * j + 1]) * srow * s4.y);
            p[2 * j + 1] = pack_bf16x2(__uint_as_float(v[4 * j + 2]) * srow * s4.z,
                                       __uint_as_float(v[4 * j + 3]) * srow * s4.w);
          }
          uint4* dst = reinterpret_cast<uint4*>(yrow + col0);
#pragma unroll
          for (int j = 0; j < 4; ++j)
            dst[j] = make_uint4(p[4 * j], p[4 * j + 1], p[4 * j + 2], p[4 * j + 3]);
        } else {
          // the ragged edge: one element at a time
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int col = col0 + j;
            if (col < N && RF_IDX_OK((size_t)row * N + col, (long long)M * N))
              yrow[col] = __float2bfloat16_rn(__uint_as_float(v[j]) * srow * __ldg(sw + col));
          }
        }
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&sh->acc_empty[buf]);
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

rf_status launch_fp8_gemm(const uint8_t* xq, const float* sx, const uint8_t* wq, const float* sw,
                          int M, int N, int K, void* y, cudaStream_t st) {
  // CTA pairs (gemm_fp8_2sm.cu) wherever they apply; this kernel otherwise
  const rf_status pair = launch_fp8_gemm_2sm(xq, sx, wq, sw, M, N, K, y, st);
  if (pair != RF_ERR_UNSUPPORTED) return pair;
  CUtensorMap ta, tb, tbh;
  if (!tc::make_tmap_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, xq, (uint64_t)K, (uint64_t)M,
                        (uint64_t)K, BK, BM, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !tc::make_tmap_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, wq, (uint64_t)K, (uint64_t)N,
                        (uint64_t)K, BK, BN, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !tc::make_tmap_2d(&tbh, CU_TENSOR_MAP_DATA_TYPE_UINT8, wq, (uint64_t)K, (uint64_t)N,
                        (uint64_t)K, BK, BN / 2, CU_TENSOR_MAP_SWIZZLE_128B))
    return RF_ERR_CUDA;
  static std::atomic<uint64_t> attr{0};
  if (smem_attr(fp8_gemm_kernel, SMEM_BYTES, attr) != RF_OK) return RF_ERR_CUDA;
  const int tiles = ((M + BM - 1) / BM) * ((N + BN - 1) / BN);
  const int sms = tc::sm_count();
  const int grid = sms > 0 && sms < tiles ? sms : tiles;
  // Wave shaping: when the tiles left after the full waves fit into one wave
  // as halves, run them as 128 x 128 halves (e.g. 512 tiles on 152 SMs: 3
  // waves of whole tiles + one wave of 112 halves instead of a fourth wave of
  // 56 whole tiles).
  const int waves = tiles / grid, rem = tiles - waves * grid;
  int full_items = tiles, num_items = tiles;
  if (waves >= 1 && rem > 0 && 2 * rem <= grid) {
    full_items = waves * grid;
    num_items = full_items + 2 * rem;
  }
  fp8_gemm_kernel<<<grid, THREADS, SMEM_BYTES, st>>>(ta, tb, tbh, sx, sw,
                                                     static_cast<__nv_bfloat16*>(y), M, N, K,
                                                     full_items, num_items);
  return launch_status();
}

RF_TIMEOUT_WORD_OF_THIS_FILE

RF_BOUNDS_WORD_OF_THIS_FILE

}  // namespace rf
