// FP8 GEMM with the per-row x per-column scale epilogue on CTA pairs: the
// same product as gemm_fp8.cu (phase 2 of the abs-max -> quantise -> GEMM
// cascade, RedFuser episode transcript, cue 33), with every MMA issued across
// the two SMs of a cluster of two CTAs (tcgen05 cta_group::2).
//
//   Y[m, n] = bf16( (sum_k dec(Xq[m,k]) dec(Wq[n,k])) * sx[m] * sw[n] )
//
// A pair computes a 256 x 256 tile of Y.  CTA r of the pair holds rows
// [128 r, 128 r + 128) of the tile's Xq and rows [128 r, 128 r + 128) of its
// Wq tile (half of B) in its own shared memory, and its 128 rows of the
// accumulator in its own TMEM.  One thread of CTA 0 issues M = 256, N = 256,
// K = 32 MMAs that read A and B from both CTAs' shared memory at the same
// offsets.  Against one 128 x 256 tile per SM (gemm_fp8.cu) each SM loads
// half the Wq bytes, its tensor core reads 8 KiB of operands per 128-cycle
// MMA instead of 12 KiB, and a single issued instruction covers two SMs.
//
// Persistent, one CTA per SM, warp-specialised (both CTAs of a pair run the
// same roles):
//   warp 0      TMA producer: this CTA's 128 x 256-byte Xq rows and 128 x
//               256-byte Wq rows (each as two 128-byte-swizzled sub-tiles)
//               into a 3-stage ring; the copies of both CTAs complete on CTA
//               0's stage barrier.  256 bytes of K per stage: the issuing
//               thread's wait, fence and commit per stage cost the tensor pipe
//               idle time, so a stage carries eight MMAs rather than four;
//   warp 1      TMEM allocation for the pair (512 columns: two 256-column
//               accumulators); in CTA 0 one thread issues the MMAs, commits
//               each stage to both CTAs' producers and each finished
//               accumulator to both CTAs' epilogues;
//   warps 2-5   epilogue: tcgen05.ld of this CTA's 128 accumulator rows,
//               scale by sx[row] * sw[col], round to bf16, store; then tell
//               CTA 0 that the accumulator may be reused.
// Work items are pair tiles i = cluster + j * clusters.  When the tiles left
// after the whole waves fit into one wave as halves, they run as 256 x 128
// halves (N = 128 MMAs; each CTA holds 64 rows of B).  Every barrier wait is
// bounded (see tc_common.cuh); the two CTAs meet at a cluster barrier before
// either exits, and hold their shared memory 200 us longer after a timeout.

#include <cuda_bf16.h>

#include "tc_common.cuh"

namespace rf {
namespace {

constexpr int BM = 128;                       // rows per CTA (256 per pair)
constexpr int BN = 256;                       // columns per pair tile
constexpr int NSUB = 2;                       // 128-byte-swizzled sub-tiles per operand and stage
constexpr int SUB = 128;                      // K bytes per sub-tile
constexpr int BK = NSUB * SUB;                // bytes = e4m3 elements per stage
constexpr int UMMA_K = 32;
constexpr int STAGES = 3;
constexpr int A_SUB = BM * SUB;               // 16 KiB: this CTA's Xq rows, one sub-tile
constexpr int B_SUB = (BN / 2) * SUB;         // 16 KiB: this CTA's half of the Wq tile, one sub-tile
constexpr int A_BYTES = NSUB * A_SUB;
constexpr int B_BYTES = NSUB * B_SUB;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int TMEM_COLS = 2 * BN;
constexpr int THREADS = 192;

struct Shared {
  uint64_t full[STAGES];         // CTA 0: both CTAs' copies of a stage
  uint64_t empty[STAGES];        // each CTA: the pair's MMAs done with the stage
  uint64_t acc_full[2];          // each CTA: the accumulator is complete
  uint64_t acc_empty[2];         // CTA 0: both CTAs' epilogues are done with it
  uint32_t tmem_base;
  int abort;
};

constexpr size_t SMEM_BYTES = (size_t)STAGES * STAGE_BYTES + sizeof(Shared) + 1024;
static_assert(SMEM_BYTES <= 232448, "exceeds the 227 KiB of shared memory a CTA may use");

__global__ void __launch_bounds__(THREADS, 1)
fp8_gemm_2sm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmBh, const float* __restrict__ sx,
                    const float* __restrict__ sw, __nv_bfloat16* __restrict__ y, int M, int N,
                    int K, int full_items, int num_items) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  Shared* sh = reinterpret_cast<Shared*>(smem + (size_t)STAGES * STAGE_BYTES);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rank = (int)tc::cluster_ctarank();          // 0 or 1
  const int cluster = (int)(blockIdx.x >> 1), nclusters = (int)(gridDim.x >> 1);
  const int tiles_n = (N + BN - 1) / BN;
  const int num_k = (K + BK - 1) / BK;
  // work item i: a 256 x 256 pair tile for i < full_items, else half of one
  // of the remaining tiles (256 x 128)
  auto item = [&](int i, int& tm2, int& col0, int& width) {
    int tile = i, half = 0;
    width = BN;
    if (i >= full_items) {
      tile = full_items + ((i - full_items) >> 1);
      half = (i - full_items) & 1;
      width = BN / 2;
    }
    tm2 = tile / tiles_n;
    col0 = (tile - tm2 * tiles_n) * BN + half * (BN / 2);
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      tc::mbar_init(&sh->full[s], 1);
      tc::mbar_init(&sh->empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&sh->acc_full[b], 1);
      tc::mbar_init(&sh->acc_empty[b], 8);    // 4 epilogue warps in each CTA
    }
    sh->abort = 0;
    tc::fence_barrier_init();
    tc::prefetch_tmap(&tmA);
    tc::prefetch_tmap(&tmB);
    tc::prefetch_tmap(&tmBh);
  }
  if (warp == 1) tc::tmem_alloc_pair(&sh->tmem_base, TMEM_COLS);
  tc::fence_before_sync();
  // both CTAs' barriers are initialised before any copy, commit or arrival
  // reaches them
  tc::cluster_sync();
  tc::fence_after_sync();
  const uint32_t tmem = sh->tmem_base;
  volatile int* abort = &sh->abort;

  if (warp == 0) {
    // ------------------------------------------------ TMA producer ----
    if (lane == 0) {
      uint32_t it = 0;
      for (int i = cluster; i < num_items && !*abort; i += nclusters) {
        int tm2, col0, width;
        item(i, tm2, col0, width);
        const bool half = width != BN;
        const uint32_t bytes = 2u * (uint32_t)(A_BYTES + (half ? B_BYTES / 2 : B_BYTES));
        const int bw = width / 2;                   // rows of B this CTA loads
        for (int kb = 0; kb < num_k; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1u;
          if (!tc::mbar_wait(&sh->empty[s], ph ^ 1u, abort)) break;
          const uint32_t full0 = tc::mapa(tc::smem_u32(&sh->full[s]), 0);
          if (rank == 0) tc::mbar_arrive_expect_tx(&sh->full[s], bytes);
          uint8_t* a = smem + (size_t)s * STAGE_BYTES;
          uint8_t* b = a + A_BYTES;
#pragma unroll
          for (int h = 0; h < NSUB; ++h) {
            tc::tma_load_2d_pair(a + h * A_SUB, &tmA, full0, kb * BK + h * SUB, tm2 * 2 * BM + rank * BM);
            tc::tma_load_2d_pair(b + h * (half ? B_SUB / 2 : B_SUB), half ? &tmBh : &tmB, full0,
                             kb * BK + h * SUB, col0 + rank * bw);
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer (CTA 0) ----
    if (lane == 0 && rank == 0) {
      constexpr uint32_t idesc_full = tc::idesc_e4m3_f32(2 * BM, BN);
      constexpr uint32_t idesc_half = tc::idesc_e4m3_f32(2 * BM, BN / 2);
      uint32_t it = 0, t = 0;
      for (int i = cluster; i < num_items && !*abort; i += nclusters, ++t) {
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
          // the B sub-tiles of a half-width item are half as tall
          const uint64_t b_sub = (uint64_t)((i < full_items ? B_SUB : B_SUB / 2) >> 4);
#pragma unroll
          for (int k = 0; k < BK / UMMA_K; ++k) {
            const int h = k / (SUB / UMMA_K), kk = k % (SUB / UMMA_K);
            tc::mma_pair_f8f6f4(d, adesc + (uint64_t)((h * A_SUB + kk * UMMA_K) >> 4),
                     bdesc + (uint64_t)h * b_sub + (uint64_t)((kk * UMMA_K) >> 4), idesc,
                     (kb | k) != 0);
          }
          tc::commit_pair_both(&sh->empty[s]);
        }
        if (!ok) break;
        tc::commit_pair_both(&sh->acc_full[buf]);
      }
    }
  } else {
    // ------------------------------------------------ epilogue ----
    const int quarter = warp & 3;              // TMEM lanes this warp may access
    const int r = quarter * 32 + lane;         // row within this CTA's half of the tile
    const uint32_t acc_empty0_0 = tc::mapa(tc::smem_u32(&sh->acc_empty[0]), 0);
    const uint32_t acc_empty0_1 = tc::mapa(tc::smem_u32(&sh->acc_empty[1]), 0);
    uint32_t t = 0;
    for (int i = cluster; i < num_items; i += nclusters, ++t) {
      const int buf = t & 1;
      const uint32_t bph = (t >> 1) & 1u;
      if (!tc::mbar_wait(&sh->acc_full[buf], bph, abort)) break;
      tc::fence_after_sync();
      int tm2, tcol0, width;
      item(i, tm2, tcol0, width);
      const int row = tm2 * 2 * BM + rank * BM + r;
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
      if (lane == 0) tc::arrive_cluster(buf ? acc_empty0_1 : acc_empty0_0);
    }
  }

  tc::fence_before_sync();
  __syncwarp();
  // neither CTA leaves while the other may still copy, commit or arrive into it
  tc::cluster_sync();
  if (warp == 1) {
    if (*abort) {
      const unsigned long long t0 = tc::globaltimer_ns();
      while (tc::globaltimer_ns() - t0 < 200000ull) {
      }
    }
    tc::fence_after_sync();
    tc::tmem_dealloc_pair(tmem, TMEM_COLS);
  }
}

cudaLaunchConfig_t pair_config(cudaLaunchAttribute* attr, unsigned grid, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = st;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

// resident clusters of two on the current device (0: none), queried once per
// device (up to 64); also sets the kernel's shared-memory attribute
int resident_pairs() {
  static std::atomic<int> count[64];
  static std::atomic<uint64_t> attr_done{0}, known{0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  const uint64_t bit = 1ull << dev;
  if (known.load(std::memory_order_acquire) & bit) return count[dev].load();
  int n = 0;
  if (smem_attr(fp8_gemm_2sm_kernel, SMEM_BYTES, attr_done) == RF_OK) {
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = pair_config(attr, 2u, 0);
    if (cudaOccupancyMaxActiveClusters(&n, fp8_gemm_2sm_kernel, &cfg) != cudaSuccess) n = 0;
  }
  cudaGetLastError();
  count[dev].store(n);
  known.fetch_or(bit, std::memory_order_release);
  return n;
}

}  // namespace

// The pair kernel for M > 128 when clusters of two fit on the device;
// RF_ERR_UNSUPPORTED otherwise (the one-SM kernel takes the shape).
rf_status launch_fp8_gemm_2sm(const uint8_t* xq, const float* sx, const uint8_t* wq,
                              const float* sw, int M, int N, int K, void* y, cudaStream_t st) {
  if (M <= BM) return RF_ERR_UNSUPPORTED;
  const int pairs = resident_pairs();
  if (pairs <= 0) return RF_ERR_UNSUPPORTED;
  CUtensorMap ta, tb, tbh;
  if (!tc::make_tmap_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, xq, (uint64_t)K, (uint64_t)M,
                        (uint64_t)K, SUB, BM, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !tc::make_tmap_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, wq, (uint64_t)K, (uint64_t)N,
                        (uint64_t)K, SUB, BN / 2, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !tc::make_tmap_2d(&tbh, CU_TENSOR_MAP_DATA_TYPE_UINT8, wq, (uint64_t)K, (uint64_t)N,
                        (uint64_t)K, SUB, BN / 4, CU_TENSOR_MAP_SWIZZLE_128B))
    return RF_ERR_CUDA;
  const int tiles = ((M + 2 * BM - 1) / (2 * BM)) * ((N + BN - 1) / BN);
  const int clusters = pairs < tiles ? pairs : tiles;
  // wave shaping as in the one-SM kernel: leftover tiles that fit into one
  // wave as halves run as 256 x 128 halves
  const int waves = tiles / clusters, rem = tiles - waves * clusters;
  int full_items = tiles, num_items = tiles;
  if (waves >= 1 && rem > 0 && 2 * rem <= clusters) {
    full_items = waves * clusters;
    num_items = full_items + 2 * rem;
  }
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pair_config(attr, (unsigned)(2 * clusters), st);
  if (cudaLaunchKernelEx(&cfg, fp8_gemm_2sm_kernel, ta, tb, tbh, sx, sw,
                         static_cast<__nv_bfloat16*>(y), M, N, K, full_items, num_items) !=
      cudaSuccess) {
    cudaGetLastError();
    return RF_ERR_CUDA;
  }
  return launch_status();
}

RF_TIMEOUT_WORD_OF_THIS_FILE

RF_BOUNDS_WORD_OF_THIS_FILE

}  // namespace rf
