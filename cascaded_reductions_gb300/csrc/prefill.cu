// Causal prefill attention: GEMM -> online softmax -> GEMM on tcgen05.
//
// The cascade (RedFuser episode transcript, cue 9): S = Q K^T, then the row
// max, the exp-sum and the weighted sum with V.  Fused form (cues 15-19, 31):
// every 128-row query tile streams its 128-key K/V tiles once and keeps the
// running state per row; the state lives at the block level of the reduction
// tree (cue 31).
//
// One CTA per (batch*head, pair of adjacent 128-row query tiles A and B),
// head-major, heaviest pair of each head first.  The two tiles share every
// K/V tile loaded into shared memory, and their softmaxes run on separate
// warp groups, so while one group works on its scores the tensor core runs
// the other tile's MMAs.
//   warp 16     TMA: both Q tiles once, then K_j and V_j tiles (two 64-column
//               boxes each, 128-byte swizzle) into a 2-stage ring;
//   warp 17     allocates 512 TMEM columns (S_A, S_B, O_A, O_B, 128 each)
//               and issues every MMA from one thread, in the order
//               S_A(0) S_B(0) | PV_A(j) S_A(j+1) PV_B(j) S_B(j+1) | ...
//               S = Q K^T is kind::f16 128x128x16 with both operands K-major
//               in shared memory; O += P V reads P from TMEM (the softmax
//               writes it as bf16 pairs over the first 64 columns of S) and V
//               MN-major from shared memory;
//   warps 0-7   softmax of tile A, warps 8-15 softmax of tile B: each warp
//               reads 16 query rows (TMEM lanes) of S with the 16x256b shape,
//               which gives every thread 32 keys of two rows and puts the
//               four threads of a row in adjacent lanes: the row max is two
//               xor shuffles.  Each thread exponentiates its keys in the log2
//               domain (scores times scale*log2(e)), writes its bf16 pairs of
//               P with the matching 16x128b store, and rescales its part of O
//               when needed.
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
constexpr int STAGES = 2;
constexpr int TILE_BYTES = BM * HD * 2;      // 32 KiB (two 16 KiB swizzled halves)
constexpr int HALF_BYTES = TILE_BYTES / 2;
constexpr int TMA_WARP = 16, MMA_WARP = 17;
constexpr int THREADS = 18 * 32;
constexpr int TMEM_COLS = 512;
constexpr float RESCALE_THRESHOLD = 8.0f;    // log2 units

__device__ __forceinline__ uint32_t s_col(int x) { return (uint32_t)x * 128u; }
__device__ __forceinline__ uint32_t o_col(int x) { return 256u + (uint32_t)x * 128u; }

struct Shared {
  uint64_t q_full;
  uint64_t k_full[STAGES];
  uint64_t v_full[STAGES];
  uint64_t kv_empty[STAGES];
  uint64_t s_full[2];          // per tile
  uint64_t p_ready[2];         // per tile, 8 softmax warps
  uint64_t o_done[2];          // per tile: the last P V done (one phase)
  uint64_t l_ready[2];         // per tile, 8 softmax warps
  float row_l[2][BM];          // [tile][row]: the row's sum, for the epilogue
  float row_m[2][BM];          // [tile][row]: the row's reference max (log2 units)
  uint32_t tmem_base;
  int abort;
};

// layout: Q_A | Q_B | K[STAGES] | V[STAGES] | Shared
constexpr size_t SMEM_BYTES = (size_t)(2 + 2 * STAGES) * TILE_BYTES + sizeof(Shared) + 1024;
static_assert(SMEM_BYTES <= 232448, "exceeds the 227 KiB of shared memory a CTA may use");

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// fp32 pairs in one 64-bit register for the packed FMA / add of sm_100+
__device__ __forceinline__ uint64_t pack_f32x2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float lo_f32(uint64_t v) {
  float lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
  return lo;
}
__device__ __forceinline__ float hi_f32(uint64_t v) {
  float lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
  return hi;
}
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t add_f32x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// load a 128x128 bf16 tile as two 128-byte-wide boxes
__device__ __forceinline__ void load_tile(uint8_t* dst, const CUtensorMap* map, uint64_t* bar,
                                          int row) {
  tc::tma_load_2d(dst, map, bar, 0, row);
  tc::tma_load_2d(dst + HALF_BYTES, map, bar, 64, row);
}

// S (TMEM) = Q (smem) K^T (smem): eight K-steps of 16 columns; the second 64
// columns of each tile sit in the second swizzled half.  The descriptors of
// the tiles' first K-step are built once by the caller; a K-step's descriptor
// is that plus its byte offset >> 4 (a compile-time constant), so each MMA
// costs the issuing thread one 64-bit add instead of a descriptor build.
__device__ __forceinline__ void mma_qk(uint32_t d, uint64_t q_desc, uint64_t k_desc) {
  constexpr uint32_t idesc = tc::idesc_bf16_f32(BM, BN, false);
#pragma unroll
  for (int kk = 0; kk < HD / 16; ++kk) {
    const uint64_t off = (uint64_t)(((kk >> 2) * HALF_BYTES + (kk & 3) * 32) >> 4);
    tc::mma_f16_ss(d, q_desc + off, k_desc + off, idesc, kk != 0);
  }
}

// O (TMEM) [+]= P (TMEM, 16 keys = 8 columns per step) V (smem, MN-major:
// 64-column halves 16 KiB apart, 8-key groups 1 KiB apart; v_desc is the
// descriptor of the first 16-key group)
__device__ __forceinline__ void mma_pv(uint32_t o, uint32_t p, uint64_t v_desc, bool acc) {
  constexpr uint32_t idesc = tc::idesc_bf16_f32(BM, HD, true);
#pragma unroll
  for (int kk = 0; kk < BN / 16; ++kk)
    tc::mma_f16_ts(o, p + (uint32_t)(kk * 8), v_desc + (uint64_t)((kk * 2048) >> 4), idesc,
                   (acc || kk != 0) ? 1u : 0u);
}

__global__ void __launch_bounds__(THREADS, 1)
prefill_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, __nv_bfloat16* __restrict__ out,
               float* __restrict__ lse, int N, int causal, float scale_log2) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;                                 // Q_A, then Q_B
  uint8_t* sK = smem + 2 * TILE_BYTES;
  uint8_t* sV = sK + STAGES * TILE_BYTES;
  Shared* sh = reinterpret_cast<Shared*>(sV + STAGES * TILE_BYTES);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int NB = (N + BM - 1) / BM;                   // query (and key) tiles per head
  const int NP = (NB + 1) / 2;                        // tile pairs per head
  // head-major order, heaviest pair of each head first
  const int bh = (int)(blockIdx.x / NP);
  const int pair = NP - 1 - (int)(blockIdx.x % NP);
  const int m_tile0 = 2 * pair, m_tile1 = 2 * pair + 1;
  const bool has_b = m_tile1 < NB;
  const int nblk0 = causal ? m_tile0 + 1 : NB;
  const int nblk1 = has_b ? (causal ? m_tile1 + 1 : NB) : 0;
  const int nmax = nblk0 > nblk1 ? nblk0 : nblk1;
  const int key0 = bh * N;

  if (threadIdx.x == 0) {
    tc::mbar_init(&sh->q_full, 1);
    for (int s = 0; s < STAGES; ++s) {
      tc::mbar_init(&sh->k_full[s], 1);
      tc::mbar_init(&sh->v_full[s], 1);
      tc::mbar_init(&sh->kv_empty[s], 1);
    }
    for (int x = 0; x < 2; ++x) {
      tc::mbar_init(&sh->s_full[x], 1);
      tc::mbar_init(&sh->p_ready[x], 8);
      tc::mbar_init(&sh->o_done[x], 1);
      tc::mbar_init(&sh->l_ready[x], 8);
    }
    sh->abort = 0;
    tc::fence_barrier_init();
  }
  if (warp == MMA_WARP) tc::tmem_alloc(&sh->tmem_base, TMEM_COLS);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = sh->tmem_base;
  volatile int* abort = &sh->abort;

  if (warp == TMA_WARP) {
    // ------------------------------------------------------ TMA ----
    if (lane == 0) {
      tc::prefetch_tmap(&tmQ);
      tc::prefetch_tmap(&tmK);
      tc::prefetch_tmap(&tmV);
      tc::mbar_arrive_expect_tx(&sh->q_full, (has_b ? 2 : 1) * TILE_BYTES);
      load_tile(sQ, &tmQ, &sh->q_full, key0 + m_tile0 * BM);
      if (has_b) load_tile(sQ + TILE_BYTES, &tmQ, &sh->q_full, key0 + m_tile1 * BM);
      for (int j = 0; j < nmax; ++j) {
        const int s = j % STAGES;
        const uint32_t ph = (uint32_t)(j / STAGES) & 1u;
        if (!tc::mbar_wait(&sh->kv_empty[s], ph ^ 1u, abort)) break;
        tc::mbar_arrive_expect_tx(&sh->k_full[s], TILE_BYTES);
        load_tile(sK + s * TILE_BYTES, &tmK, &sh->k_full[s], key0 + j * BN);
        tc::mbar_arrive_expect_tx(&sh->v_full[s], TILE_BYTES);
        load_tile(sV + s * TILE_BYTES, &tmV, &sh->v_full[s], key0 + j * BN);
      }
    }
  } else if (warp == MMA_WARP) {
    // ------------------------------------------------------ MMA ----
    if (lane == 0) {
      // the first K-step's descriptors of Q_A, Q_B and of each K and V stage
      const uint64_t q_desc0 = tc::sdesc_sw128(tc::smem_u32(sQ), 16, 1024);
      const uint64_t q_desc1 = tc::sdesc_sw128(tc::smem_u32(sQ + TILE_BYTES), 16, 1024);
      static_assert(STAGES == 2, "one descriptor per stage, picked by j & 1");
      const uint64_t k_desc0 = tc::sdesc_sw128(tc::smem_u32(sK), 16, 1024);
      const uint64_t k_desc1 = tc::sdesc_sw128(tc::smem_u32(sK + TILE_BYTES), 16, 1024);
      const uint64_t v_desc0 = tc::sdesc_sw128(tc::smem_u32(sV), HALF_BYTES, 1024);
      const uint64_t v_desc1 = tc::sdesc_sw128(tc::smem_u32(sV + TILE_BYTES), HALF_BYTES, 1024);
      bool ok = tc::mbar_wait(&sh->q_full, 0, abort);
      // S_x(j) needs K_j; the wait is done once per j
      int k_waited = -1;
      auto issue_s = [&](int x, int j) -> bool {
        if (k_waited < j) {
          k_waited = j;
          if (!tc::mbar_wait(&sh->k_full[j % STAGES], (uint32_t)(j / STAGES) & 1u, abort))
            return false;
        }
        tc::fence_after_sync();
        mma_qk(tmem + s_col(x), x ? q_desc1 : q_desc0, (j & 1) ? k_desc1 : k_desc0);
        tc::mma_commit(&sh->s_full[x]);
        return true;
      };
      int v_waited = -1;
      auto issue_pv = [&](int x, int j) -> bool {
        if (!tc::mbar_wait(&sh->p_ready[x], (uint32_t)j & 1u, abort)) return false;
        if (v_waited < j) {
          v_waited = j;
          if (!tc::mbar_wait(&sh->v_full[j % STAGES], (uint32_t)(j / STAGES) & 1u, abort))
            return false;
        }
        tc::fence_after_sync();
        mma_pv(tmem + o_col(x), tmem + s_col(x), (j & 1) ? v_desc1 : v_desc0, j > 0);
        // a tile's softmax learns that P V(j) is done from S(j + 1)'s commit
        // (every commit covers all earlier MMAs of this thread); only the last
        // P V needs a commit of its own, for the epilogue
        if (j == (x ? nblk1 : nblk0) - 1) tc::mma_commit(&sh->o_done[x]);
        return true;
      };
      if (ok) ok = issue_s(0, 0);
      if (ok && nblk1 > 0) ok = issue_s(1, 0);
      for (int j = 0; ok && j < nmax; ++j) {
        if (j < nblk0) {
          if (!(ok = issue_pv(0, j))) break;
          if (j + 1 < nblk0 && !(ok = issue_s(0, j + 1))) break;
        }
        if (j < nblk1) {
          if (!(ok = issue_pv(1, j))) break;
          if (j + 1 < nblk1 && !(ok = issue_s(1, j + 1))) break;
        }
        tc::mma_commit(&sh->kv_empty[j % STAGES]);   // K_j and V_j fully consumed
      }
    }
  } else {
    // --------------------------------------------------- softmax ----
    // Warp (quarter, sub) of a tile owns TMEM lanes 32 quarter + 16 sub ..
    // + 15 and reads them with the 16x256b shape: thread t holds rows
    // r0 = t / 4 and r0 + 8 of those 16, keys 8k + 2 (t % 4) + {0, 1} for
    // k = 0..15.  The four threads of a row are adjacent lanes, so its max is
    // two xor shuffles.
    const int x = warp >> 3;                        // tile A (0) or B (1)
    const int quarter = warp & 3, sub = (warp >> 2) & 1;
    const int cq = lane & 3;                        // key pair within each group of 8 keys
    const int r0 = quarter * 32 + sub * 16 + (lane >> 2);   // rows r0 and r0 + 8 of the tile
    const uint32_t lane16 = tmem + ((uint32_t)(quarter * 32 + sub * 16) << 16);
    const int n = x ? nblk1 : nblk0;
    const int m_tile = x ? m_tile1 : m_tile0;
    float m_ref[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
    bool ok = n > 0;
    const uint64_t sl2 = pack_f32x2(scale_log2, scale_log2);
    for (int j = 0; j < n && ok; ++j) {
      if (!tc::mbar_wait(&sh->s_full[x], (uint32_t)j & 1u, abort)) {
        ok = false;
        break;
      }
      tc::fence_after_sync();
      float s[2][32];                               // s[row][2k + e] = key 8k + 2 cq + e
      {
        uint32_t v[64];
        tc::tmem_ld_16x256b_x16(lane16 + s_col(x), v);
        tc::tmem_ld_wait();
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          s[0][2 * k] = __uint_as_float(v[4 * k]);
          s[0][2 * k + 1] = __uint_as_float(v[4 * k + 1]);
          s[1][2 * k] = __uint_as_float(v[4 * k + 2]);
          s[1][2 * k + 1] = __uint_as_float(v[4 * k + 3]);
        }
      }
      if (causal && j == m_tile) {
#pragma unroll
        for (int k = 0; k < 16; ++k)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int key = 8 * k + 2 * cq + e;
            if (key > r0) s[0][2 * k + e] = -INFINITY;
            if (key > r0 + 8) s[1][2 * k + e] = -INFINITY;
          }
      } else if (!causal && j == NB - 1 && N % BN != 0) {
        // keys past N in the last tile are the next head's rows (or TMA's
        // zero fill): leave them out.  Under the causal mask they never count
        // for a row that is stored.
        const int kmax = N - j * BN;
#pragma unroll
        for (int k = 0; k < 16; ++k)
#pragma unroll
          for (int e = 0; e < 2; ++e)
            if (8 * k + 2 * cq + e >= kmax) {
              s[0][2 * k + e] = -INFINITY;
              s[1][2 * k + e] = -INFINITY;
            }
      }
      float m_new[2], alpha[2];
      bool move_any = false;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        // row max over this thread's 32 keys (three-input max), then over the
        // row's four threads; raw scores (scale_log2 > 0 is applied after)
        float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int i = 0; i < 32; i += 2) mx[(i >> 1) & 3] = max3(mx[(i >> 1) & 3], s[h][i], s[h][i + 1]);
        float pm = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
        pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 1));
        pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 2));
        const float mt = pm * scale_log2;
        // move the reference max only when it has grown by more than the threshold
        const bool move = mt > m_ref[h] + RESCALE_THRESHOLD;
        m_new[h] = move ? mt : m_ref[h];
        alpha[h] = ex2(m_ref[h] - m_new[h]);        // 0 on the first tile, 1 when not moved
        l[h] *= alpha[h];
        m_ref[h] = m_new[h];
        move_any |= move;
      }
      // P = exp2(s * scale_log2 - m) as bf16 pairs over the first 64 columns
      // of S (key pair (8k + 2 cq, + 1) -> column 4k + cq), row sums on pairs
      // (packed fp32x2 FMA and add)
      {
        uint32_t w[32];
        uint64_t sum2[2] = {0ull, 0ull};
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint64_t nm2 = pack_f32x2(-m_new[h], -m_new[h]);
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const uint64_t a = fma_f32x2(pack_f32x2(s[h][2 * k], s[h][2 * k + 1]), sl2, nm2);
            const float p0 = ex2(lo_f32(a));
            const float p1 = ex2(hi_f32(a));
            sum2[h] = add_f32x2(sum2[h], pack_f32x2(p0, p1));
            w[2 * k + h] = pack_bf16x2(p0, p1);
          }
        }
        tc::tmem_st_16x128b_x16(lane16 + s_col(x), w);
        l[0] += lo_f32(sum2[0]) + hi_f32(sum2[0]);
        l[1] += lo_f32(sum2[1]) + hi_f32(sum2[1]);
      }
      // O holds every earlier P V before it is rescaled: S(j) was issued after
      // P V(j - 1), and its completion (waited above) covers it
      if (j > 0) {
        if (__any_sync(0xffffffffu, move_any)) {
#pragma unroll 1
          for (int c = 0; c < 2; ++c) {
            const uint32_t oc = lane16 + o_col(x) + (uint32_t)(c * 64);
            uint32_t v[32];
            tc::tmem_ld_16x256b_x8(oc, v);
            tc::tmem_ld_wait();
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              v[4 * k] = __float_as_uint(__uint_as_float(v[4 * k]) * alpha[0]);
              v[4 * k + 1] = __float_as_uint(__uint_as_float(v[4 * k + 1]) * alpha[0]);
              v[4 * k + 2] = __float_as_uint(__uint_as_float(v[4 * k + 2]) * alpha[1]);
              v[4 * k + 3] = __float_as_uint(__uint_as_float(v[4 * k + 3]) * alpha[1]);
            }
            tc::tmem_st_16x256b_x8(oc, v);
          }
        }
      }
      tc::tmem_st_wait();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&sh->p_ready[x]);
    }
    if (n > 0) {
      // each row's sum over its four threads; one thread per row publishes
      // the row's sum and reference for the epilogue
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        l[h] += __shfl_xor_sync(0xffffffffu, l[h], 1);
        l[h] += __shfl_xor_sync(0xffffffffu, l[h], 2);
      }
      if (cq == 0) {
        sh->row_l[x][r0] = l[0];
        sh->row_l[x][r0 + 8] = l[1];
        sh->row_m[x][r0] = m_ref[0];
        sh->row_m[x][r0 + 8] = m_ref[1];
      }
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&sh->l_ready[x]);
      // epilogue, one thread per row (32x32b shape): warp (quarter, sub)
      // writes columns 64 sub .. 64 sub + 63 of rows 32 quarter .. + 31.
      // out = O / l, lse = (m_ref + log2 l) * ln 2
      if (ok && tc::mbar_wait(&sh->l_ready[x], 0, abort) &&
          tc::mbar_wait(&sh->o_done[x], 0, abort)) {
        tc::fence_after_sync();
        const int r = quarter * 32 + lane;
        const int col0 = sub * 64;
        const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
        const float lt = sh->row_l[x][r];
        const float inv = 1.f / lt;
        const int grow = key0 + m_tile * BM + r;      // global query row
        const bool row_in = m_tile * BM + r < N;      // rows past N belong to no query
        __nv_bfloat16* orow = out + (size_t)(row_in ? grow : key0) * HD + col0;
#pragma unroll 1
        for (int c = 0; c < 2; ++c) {
          uint32_t v[32];
          tc::tmem_ld_32x32b_x32(lane_base + o_col(x) + (uint32_t)(col0 + c * 32), v);
          tc::tmem_ld_wait();
          uint32_t pkd[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            pkd[i] = pack_bf16x2(__uint_as_float(v[2 * i]) * inv,
                                 __uint_as_float(v[2 * i + 1]) * inv);
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
          // (checked build) 32 outputs inside out[B*H = gridDim.x / NP][N][HD]
          if (row_in && RF_SPAN_OK((size_t)grow * HD + col0 + c * 32, 32,
                                   (long long)(gridDim.x / NP) * N * HD)) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
              dst[i] = make_uint4(pkd[4 * i], pkd[4 * i + 1], pkd[4 * i + 2], pkd[4 * i + 3]);
          }
        }
        if (lse != nullptr && sub == 0 && row_in &&
            RF_IDX_OK(grow, (long long)(gridDim.x / NP) * N))
          lse[grow] = (sh->row_m[x][r] + log2f(lt)) * kLn2;
      }
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == MMA_WARP) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace

rf_status launch_prefill(const void* q, const void* k, const void* v, int B, int H, int N, int D,
                         int causal, float scale, void* out, float* lse, cudaStream_t st) {
  (void)D;
  const rf_status pair = launch_prefill_2sm(q, k, v, B, H, N, causal, scale, out, lse, st);
  if (pair != RF_ERR_UNSUPPORTED) return pair;
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
  static std::atomic<uint64_t> attr{0};
  if (smem_attr(prefill_kernel, SMEM_BYTES, attr) != RF_OK) return RF_ERR_CUDA;
  const int NB = (N + BM - 1) / BM;
  const unsigned grid = (unsigned)(B * H) * (unsigned)((NB + 1) / 2);
  prefill_kernel<<<grid, THREADS, SMEM_BYTES, st>>>(tq, tk, tv, static_cast<__nv_bfloat16*>(out),
                                                   lse, N, causal, scale * kLog2e);
  return launch_status();
}

RF_TIMEOUT_WORD_OF_THIS_FILE

RF_BOUNDS_WORD_OF_THIS_FILE

}  // namespace rf
