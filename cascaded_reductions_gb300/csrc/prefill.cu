// Causal prefill attention: GEMM -> online softmax -> GEMM on tcgen05.
//
// The cascade (RedFuser episode transcript, cue 9): S = Q K^T, then the row
// max, the exp-sum and the weighted sum with V.  Fused form (cues 15-19, 31):
// every 128-row query tile streams its 128-key K/V tiles once and keeps the
// running state per row; the state lives at the block level of the reduction
// tree (cue 31), one thread per query row.
//
// One CTA per (batch*head, 128-row query tile), head-major, heaviest causal
// tile of each head first.
//   warp 8      TMA: Q tile once, then K_j and V_j tiles (two 64-column
//               boxes each, 128-byte swizzle) into a 3-stage ring;
//   warp 9      allocates 512 TMEM columns and issues the MMAs from one
//               thread: S_j = Q K_j^T (kind::f16, 128x128x16, both operands
//               K-major in shared memory) into one of two S buffers, and
//               O += P_j V_j with P_j read from TMEM (it overwrites the first
//               64 columns of S_j as bf16 pairs) and V_j MN-major in shared
//               memory.  S_{j+1} is issued before P_j is ready, so the tensor
//               core computes the next scores while the softmax runs;
//   warps 0-7   softmax, two threads per query row (TMEM lane), one per
//               64-key half: load S_j, mask the diagonal tile, tile max in
//               the log2 domain (scores times scale*log2(e)), p = exp2(s -
//               m_ref), partial row sum, P_j back to TMEM; then the epilogue
//               out = O / l (l = the two partial sums), lse.
// Rescaling is lazy: the reference max m_ref of a row moves (and O and l are
// multiplied by exp2(m_ref_old - m_ref_new)) only when the tile max exceeds
// it by more than 8, so p <= 2^8.  The result is the same mathematics (O and
// l share the reference), with far fewer passes over O.
// Every barrier wait is bounded (see tc_common.cuh).

#include <cuda_bf16.h>

#include "tc_common.cuh"

namespace rf {
namespace {

constexpr int BM = 128;            // query rows per tile
constexpr int BN = 128;            // keys per tile
constexpr int HD = 128;            // head dim
constexpr int STAGES = 3;
constexpr int TILE_BYTES = BM * HD * 2;      // 32 KiB (two 16 KiB swizzled halves)
constexpr int HALF_BYTES = TILE_BYTES / 2;
constexpr int THREADS = 320;
constexpr int TMEM_COLS = 512;
constexpr uint32_t O_COL = 256;           // S buffers at columns 0 and 128
__device__ __forceinline__ uint32_t s_col(int j) { return (uint32_t)(j & 1) * 128u; }
constexpr float RESCALE_THRESHOLD = 8.0f;    // log2 units

struct Shared {
  uint64_t q_full;
  uint64_t k_full[STAGES];
  uint64_t v_full[STAGES];
  uint64_t kv_empty[STAGES];
  uint64_t s_full[2];
  uint64_t p_ready[2];
  uint64_t o_done;
  uint64_t l_ready;
  float l_part[2][BM];
  uint32_t tmem_base;
  int abort;
};

// layout: Q | K[STAGES] | V[STAGES] | Shared
constexpr size_t SMEM_BYTES = (size_t)(1 + 2 * STAGES) * TILE_BYTES + sizeof(Shared) + 1024;
static_assert(SMEM_BYTES <= 232448, "exceeds the 227 KiB of shared memory a CTA may use");

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// load a 128x128 bf16 tile as two 128-byte-wide boxes
__device__ __forceinline__ void load_tile(uint8_t* dst, const CUtensorMap* map, uint64_t* bar,
                                          int row) {
  tc::tma_load_2d(dst, map, bar, 0, row);
  tc::tma_load_2d(dst + HALF_BYTES, map, bar, 64, row);
}

__global__ void __launch_bounds__(THREADS, 1)
prefill_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, __nv_bfloat16* __restrict__ out,
               float* __restrict__ lse, int BH, int N, int causal, float scale_log2) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;
  uint8_t* sK = smem + TILE_BYTES;
  uint8_t* sV = sK + STAGES * TILE_BYTES;
  Shared* sh = reinterpret_cast<Shared*>(sV + STAGES * TILE_BYTES);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int NB = N / BM;
  // head-major order, heaviest causal tile of each head first: the CTAs that
  // run at the same time share a head's K and V through L2
  const int bh = (int)(blockIdx.x / NB);
  const int mblk = NB - 1 - (int)(blockIdx.x % NB);
  const int nblocks = causal ? mblk + 1 : NB;
  const int row0 = bh * N + mblk * BM;        // first global row of this Q tile
  const int key0 = bh * N;

  if (threadIdx.x == 0) {
    tc::mbar_init(&sh->q_full, 1);
    for (int s = 0; s < STAGES; ++s) {
      tc::mbar_init(&sh->k_full[s], 1);
      tc::mbar_init(&sh->v_full[s], 1);
      tc::mbar_init(&sh->kv_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&sh->s_full[b], 1);
      tc::mbar_init(&sh->p_ready[b], 8);
    }
    tc::mbar_init(&sh->o_done, 1);
    tc::mbar_init(&sh->l_ready, 8);
    sh->abort = 0;
    tc::fence_barrier_init();
  }
  if (warp == 9) tc::tmem_alloc(&sh->tmem_base, TMEM_COLS);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = sh->tmem_base;
  volatile int* abort = &sh->abort;

  if (warp == 8) {
    // ------------------------------------------------------ TMA ----
    if (lane == 0) {
      tc::prefetch_tmap(&tmQ);
      tc::prefetch_tmap(&tmK);
      tc::prefetch_tmap(&tmV);
      tc::mbar_arrive_expect_tx(&sh->q_full, TILE_BYTES);
      load_tile(sQ, &tmQ, &sh->q_full, row0);
      for (int j = 0; j < nblocks; ++j) {
        const int s = j % STAGES;
        const uint32_t ph = (uint32_t)(j / STAGES) & 1u;
        if (!tc::mbar_wait(&sh->kv_empty[s], ph ^ 1u, abort)) break;
        tc::mbar_arrive_expect_tx(&sh->k_full[s], TILE_BYTES);
        load_tile(sK + s * TILE_BYTES, &tmK, &sh->k_full[s], key0 + j * BN);
        tc::mbar_arrive_expect_tx(&sh->v_full[s], TILE_BYTES);
        load_tile(sV + s * TILE_BYTES, &tmV, &sh->v_full[s], key0 + j * BN);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------ MMA ----
    if (lane == 0) {
      constexpr uint32_t idesc_s = tc::idesc_bf16_f32(BM, BN, false);
      constexpr uint32_t idesc_o = tc::idesc_bf16_f32(BM, HD, true);
      const uint32_t q_addr = tc::smem_u32(sQ);
      bool ok = tc::mbar_wait(&sh->q_full, 0, abort);
      // S_j = Q K_j^T into S buffer j % 2
      auto issue_s = [&](int j) -> bool {
        const int s = j % STAGES;
        if (!tc::mbar_wait(&sh->k_full[s], (uint32_t)(j / STAGES) & 1u, abort)) return false;
        tc::fence_after_sync();
        const uint32_t k_addr = tc::smem_u32(sK + s * TILE_BYTES);
        const uint32_t d = tmem + s_col(j);
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          // K-steps of 16 elements (32 bytes); the second 64 columns sit in
          // the second swizzled half
          const uint32_t off = (uint32_t)((kk >> 2) * HALF_BYTES + (kk & 3) * 32);
          tc::mma_f16_ss(d, tc::sdesc_sw128(q_addr + off, 16, 1024),
                         tc::sdesc_sw128(k_addr + off, 16, 1024), idesc_s, kk != 0);
        }
        tc::mma_commit(&sh->s_full[j & 1]);
        return true;
      };
      if (ok) ok = issue_s(0);
      for (int j = 0; ok && j < nblocks; ++j) {
        if (j + 1 < nblocks && !issue_s(j + 1)) break;
        // O += P_j V_j once the softmax has written P_j (and rescaled O)
        const int s = j % STAGES;
        if (!tc::mbar_wait(&sh->p_ready[j & 1], (uint32_t)(j >> 1) & 1u, abort)) break;
        if (!tc::mbar_wait(&sh->v_full[s], (uint32_t)(j / STAGES) & 1u, abort)) break;
        tc::fence_after_sync();
        const uint32_t v_addr = tc::smem_u32(sV + s * TILE_BYTES);
        const uint32_t p_tmem = tmem + s_col(j);
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          // A = P (TMEM, 16 keys = 8 columns per step); B = V rows kk*16..,
          // MN-major: 64-column halves 16 KiB apart (LBO), 8-key groups
          // 1 KiB apart (SBO)
          tc::mma_f16_ts(tmem + O_COL, p_tmem + (uint32_t)(kk * 8),
                         tc::sdesc_sw128(v_addr + (uint32_t)(kk * 2048), HALF_BYTES, 1024),
                         idesc_o, (j | kk) != 0);
        }
        tc::mma_commit(&sh->kv_empty[s]);
        tc::mma_commit(&sh->o_done);
      }
    }
  } else {
    // --------------------------------------------------- softmax ----
    // warp w: TMEM lane quarter w & 3 (query rows), column half w >> 2.  Both
    // threads of a row read all 128 scores of S_j and compute the same tile
    // max (same values, same order), then each exponentiates its own 64 keys
    // and, later, rescales and stores its own 64 columns of O.
    const int quarter = warp & 3, half = warp >> 2;
    const int r = quarter * 32 + lane;              // query row in the tile (TMEM lane)
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    const int col0 = half * 64;
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nblocks && ok; ++j) {
      if (!tc::mbar_wait(&sh->s_full[j & 1], (uint32_t)(j >> 1) & 1u, abort)) {
        ok = false;
        break;
      }
      tc::fence_after_sync();
      // own 64 keys (columns col0..col0+63) and the other half's 64
      float so[64], sx[64];
      {
        uint32_t v0[32], v1[32], v2[32], v3[32];
        const uint32_t sb = lane_base + s_col(j);
        tc::tmem_ld_32x32b_x32(sb + (uint32_t)col0, v0);
        tc::tmem_ld_32x32b_x32(sb + (uint32_t)col0 + 32u, v1);
        tc::tmem_ld_32x32b_x32(sb + (uint32_t)(64 - col0), v2);
        tc::tmem_ld_32x32b_x32(sb + (uint32_t)(64 - col0) + 32u, v3);
        tc::tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          so[i] = __uint_as_float(v0[i]);
          so[32 + i] = __uint_as_float(v1[i]);
          sx[i] = __uint_as_float(v2[i]);
          sx[32 + i] = __uint_as_float(v3[i]);
        }
      }
      if (causal && j == mblk) {
        // key index of so[i] is col0 + i, of sx[i] is (64 - col0) + i
#pragma unroll
        for (int i = 0; i < 64; ++i) {
          if (col0 + i > r) so[i] = -INFINITY;
          if (64 - col0 + i > r) sx[i] = -INFINITY;
        }
      }
      // raw scores here; scale_log2 > 0 is applied inside the exponent.
      // Independent maxima shorten the dependency chain; both threads of a
      // row reduce the same 128 values in the same order, so they agree.
      float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
      if (half == 0) {
#pragma unroll
        for (int i = 0; i < 64; ++i) mx[i & 3] = fmaxf(mx[i & 3], so[i]);
#pragma unroll
        for (int i = 0; i < 64; ++i) mx[i & 3] = fmaxf(mx[i & 3], sx[i]);
      } else {
#pragma unroll
        for (int i = 0; i < 64; ++i) mx[i & 3] = fmaxf(mx[i & 3], sx[i]);
#pragma unroll
        for (int i = 0; i < 64; ++i) mx[i & 3] = fmaxf(mx[i & 3], so[i]);
      }
      const float mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * scale_log2;
      // move the reference max only when it has grown by more than the threshold
      const bool move = mt > m_ref + RESCALE_THRESHOLD;
      const float m_new = move ? mt : m_ref;
      const float alpha = ex2(m_ref - m_new);       // 0 on the first tile, 1 when not moved
      l *= alpha;
      // this thread's 64 keys of P_j into its 32 columns of S_j (two bf16 per column)
      float sum[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float p0 = ex2(fmaf(so[c * 32 + 2 * i], scale_log2, -m_new));
          const float p1 = ex2(fmaf(so[c * 32 + 2 * i + 1], scale_log2, -m_new));
          sum[i & 3] += p0 + p1;
          w[i] = pack_bf16x2(p0, p1);
        }
        tc::tmem_st_32x32b_x16(lane_base + s_col(j) + (uint32_t)(half * 32 + c * 16), w);
      }
      l += (sum[0] + sum[1]) + (sum[2] + sum[3]);
      m_ref = m_new;
      // O must hold every earlier P V before it is rescaled
      if (j > 0) {
        if (!tc::mbar_wait(&sh->o_done, (uint32_t)(j - 1) & 1u, abort)) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        if (__any_sync(0xffffffffu, move)) {
#pragma unroll 1
          for (int c = 0; c < 2; ++c) {
            const uint32_t oc = lane_base + O_COL + (uint32_t)(col0 + c * 32);
            uint32_t v[32];
            tc::tmem_ld_32x32b_x32(oc, v);
            tc::tmem_ld_wait();
            uint32_t w0[16], w1[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              w0[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
              w1[i] = __float_as_uint(__uint_as_float(v[16 + i]) * alpha);
            }
            tc::tmem_st_32x32b_x16(oc, w0);
            tc::tmem_st_32x32b_x16(oc + 16u, w1);
          }
        }
      }
      tc::tmem_st_wait();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&sh->p_ready[j & 1]);
    }
    // the two halves of each row add their partial sums
    sh->l_part[half][r] = l;
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(&sh->l_ready);
    // epilogue: out = O / l, lse = (m_ref + log2 l) * ln 2
    if (ok && tc::mbar_wait(&sh->l_ready, 0, abort) &&
        tc::mbar_wait(&sh->o_done, (uint32_t)(nblocks - 1) & 1u, abort)) {
      tc::fence_after_sync();
      const float lt = sh->l_part[0][r] + sh->l_part[1][r];
      const float inv = 1.f / lt;
      __nv_bfloat16* orow = out + (size_t)(row0 + r) * HD + col0;
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        uint32_t v[32];
        tc::tmem_ld_32x32b_x32(lane_base + O_COL + (uint32_t)(col0 + c * 32), v);
        tc::tmem_ld_wait();
        uint32_t pkd[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          pkd[i] = pack_bf16x2(__uint_as_float(v[2 * i]) * inv, __uint_as_float(v[2 * i + 1]) * inv);
        uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
        for (int i = 0; i < 4; ++i) dst[i] = make_uint4(pkd[4 * i], pkd[4 * i + 1], pkd[4 * i + 2], pkd[4 * i + 3]);
      }
      if (lse != nullptr && half == 0) lse[row0 + r] = (m_ref + log2f(lt)) * kLn2;
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 9) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace

rf_status launch_prefill(const void* q, const void* k, const void* v, int B, int H, int N, int D,
                         int causal, float scale, void* out, float* lse, cudaStream_t st) {
  (void)D;
  const uint64_t rows = (uint64_t)B * H * N;
  CUtensorMap tq, tk, tv;
  const uint64_t stride = HD * 2;
  if (!tc::make_tmap_2d(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, q, HD, rows, stride, 64, BM,
                        CU_TENSOR_MAP_SWIZZLE_128B) ||
      !tc::make_tmap_2d(&tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, k, HD, rows, stride, 64, BN,
                        CU_TENSOR_MAP_SWIZZLE_128B) ||
      !tc::make_tmap_2d(&tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, v, HD, rows, stride, 64, BN,
                        CU_TENSOR_MAP_SWIZZLE_128B))
    return RF_ERR_CUDA;
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)SMEM_BYTES) != cudaSuccess)
      return RF_ERR_CUDA;
    attr_set = true;
  }
  const int BH = B * H;
  const unsigned grid = (unsigned)BH * (unsigned)(N / BM);
  prefill_kernel<<<grid, THREADS, SMEM_BYTES, st>>>(tq, tk, tv, static_cast<__nv_bfloat16*>(out),
                                                   lse, BH, N, causal, scale * kLog2e);
  return launch_status();
}

rf_status prefill_take_status(int* status) {
  int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, tc::g_timeout_status, sizeof(int)) != cudaSuccess) return RF_ERR_CUDA;
  if (cudaMemcpyToSymbol(tc::g_timeout_status, &zero, sizeof(int)) != cudaSuccess) return RF_ERR_CUDA;
  *status = v;
  return RF_OK;
}

}  // namespace rf
