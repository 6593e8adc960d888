// Causal prefill attention on CTA pairs: GEMM -> online softmax -> GEMM with
// every MMA issued across the two SMs of a cluster (tcgen05 cta_group::2).
//
// The cascade (RedFuser episode transcript, cue 9): S = Q K^T, then the row
// max, the exp-sum and the weighted sum with V.  Fused form (cues 15-19, 31):
// each 128-row query tile streams its key blocks once and keeps the running
// state per row; the state lives at the block level of the reduction tree.
//
// A work item is 256 adjacent query rows of one head: CTA r of the cluster
// takes the 128-row tile 2 p + r.  Key blocks are 256 keys wide.  Per block j:
//   S(j)  = Q K_j^T, one M = 256, N = 256 MMA per 16 columns of the head
//           dimension: CTA r supplies its Q tile (A) and keys [128 r, 128 r +
//           128) of the block (its half of B); each CTA's TMEM receives its
//           own 128 rows x 256 keys;
//   P(j)  = exp2(S scale log2(e) - m) in bf16, written by the softmax warps
//           into TMEM columns of its own (not over S);
//   O    += P(j) V_j, M = 256, N = 128 MMAs with A = P read from each CTA's
//           TMEM and B = V_j split by columns: CTA r holds head-dimension
//           columns [64 r, 64 r + 64) of all 256 keys.
// Because P does not overwrite S, S(j + 1) is issued as soon as the softmax
// has read S(j) into registers, and runs on the tensor pipe while the
// softmax of block j is still exponentiating: the pipe order is
// S(0) S(1) PV(0) S(2) PV(1) ...  The kernel is persistent (one cluster per
// pair of SMs, items head-major and heaviest first within a head, taken
// in snake order), and the numbering of blocks runs on across items, so the
// first S of the next item is computed while the softmax warps write the
// current item's output.
//
// TMEM (512 columns, allocated for the pair): S 0-255, P 256-383 (bf16 pairs,
// key pair (2c, 2c + 1) in column c), O 384-511.
// Shared memory per CTA: Q tiles (two buffers), K halves and V halves in
// 2-stage rings, 32 KiB each, all 128-byte swizzled.
// Roles, both CTAs:
//   warp 8      TMA: this CTA's Q tile, then its halves of K_j and V_j; the
//               copies of both CTAs complete on CTA 0's barriers;
//   warp 9      TMEM allocation; in CTA 0 one thread issues every MMA and
//               commits to both CTAs' barriers;
//   warps 0-7   softmax of this CTA's 128 rows: warp w reads TMEM lanes
//               32 (w % 4) .. + 31 (thread = row) and keys 128 (w / 4) .. + 127
//               of the block into registers; the two warps of a row exchange
//               their partial maxima through shared memory.
// Two softmax warps per SM sub-partition (not four) leave the MMA-issuing
// thread, which shares a sub-partition with two of them, enough issue slots
// for the 64-cycle P V MMAs; with ten warps a thread may hold 168 registers,
// enough for its 128 scores.
// Rescaling is lazy: the reference max m_ref of a row moves (and O and l are
// multiplied by exp2(m_ref_old - m_ref_new)) only when the block max exceeds
// it by more than 8, so p <= 2^8.
//
// The softmax warps tell CTA 0's MMA thread that S was read, that P was
// written and that O was read with relaxed arrivals: each follows the
// tcgen05.wait that completes those TMEM accesses, so it needs no release
// (a release at cluster scope costs the arriving warp about 1000 cycles).
// For the same reason the MMA thread waits at CTA scope: what it orders
// after a wait are MMAs, whose operands were completed by the TMA
// transaction count or by the softmax warps' tcgen05.wait (an acquire at
// cluster scope idles the tensor pipe about 160 cycles per wait).
// An item's epilogue is deferred into the first block of the next item (see
// the softmax role).
// Every barrier wait is bounded (see tc_common.cuh); the two CTAs meet at a
// cluster barrier before either exits.

#include <cuda_bf16.h>

#include "tc_common.cuh"

namespace rf {
namespace {

constexpr int BM = 128;                      // query rows per CTA (256 per pair)
constexpr int BN = 256;                      // keys per block
constexpr int HD = 128;                      // head dim
constexpr int STAGES = 2;
constexpr int TILE_BYTES = 32768;            // Q tile, K half or V half
constexpr int HALF_BYTES = 16384;            // one 64-column swizzled box of a 128-row tile
constexpr int SM_WARPS = 8;                // softmax warps: two per TMEM lane quarter
constexpr int TMA_WARP = 8, MMA_WARP = 9;
constexpr int THREADS = 10 * 32;
constexpr int TMEM_COLS = 512;
constexpr uint32_t S_COL = 0, P_COL = 256, O_COL = 384;
constexpr float RESCALE_THRESHOLD = 8.0f;    // log2 units

struct Shared {
  uint64_t q_full[2];           // CTA 0: both Q tiles of a buffer
  uint64_t q_empty[2];          // each CTA: the item's S MMAs are done with the buffer
  uint64_t k_full[STAGES];      // CTA 0: both K halves of a stage
  uint64_t v_full[STAGES];      // CTA 0: both V halves of a stage
  uint64_t k_empty[STAGES];     // each CTA: S of that block done
  uint64_t v_empty[STAGES];     // each CTA: P V of that block done
  uint64_t s_full;              // each CTA: S(g) complete
  uint64_t pv_done;             // each CTA: P V(g) complete
  uint64_t s_free;              // CTA 0: both CTAs' softmax warps have read S(g) (32 warps)
  uint64_t p_ready;             // CTA 0: both CTAs' P(g) and O rescale written (32 warps)
  uint64_t o_free;              // CTA 0: both CTAs' epilogues have read O (32 warps)
  uint64_t red_bar[4];          // each CTA, per lane quarter: its four warps' maxima / sums
  float red[2][2][BM];          // [exchange & 1][key half][row]: partial row maxima
  float part_l[2][BM];          // [key half][row]: partial row sums of an item
  uint32_t tmem_base;
  int abort;
};

// layout: Q[2] | K[STAGES] | V[STAGES] | Shared
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
__device__ __forceinline__ void unpack_f32x2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
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

// one 32-byte global store (sm_100+); `dst` 32-byte aligned
__device__ __forceinline__ void st_global_v8(void* dst, const uint32_t* w) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst), "r"(w[0]),
               "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}

// arrival on a barrier of CTA 0 without release semantics (see the file
// comment for why none is needed)
__device__ __forceinline__ void arrive_cluster_relaxed(uint32_t bar) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar)
               : "memory");
}

// A work item: 256 query rows (two 128-row tiles) of one head.  Items are
// numbered head-major, the heaviest pair of tiles of each head first.
struct Item {
  int key0;     // first row of the head in Q, K, V and out
  int pair;     // tiles 2 pair and 2 pair + 1 of the head
  int n;        // key blocks (the same for both CTAs)
};

// Cluster c takes the item c of every even round of nclusters items and
// item nclusters - 1 - c of every odd round: with items weighted p + 1 under
// the causal mask, the snake evens out the clusters' totals (plain
// round-robin leaves some clusters a tenth more work than the mean).
__device__ __forceinline__ int item_index(int t, int cluster, int nclusters) {
  return t * nclusters + ((t & 1) ? nclusters - 1 - cluster : cluster);
}
__device__ __forceinline__ Item item_of(int i, int N, int causal) {
  const int NB = (N + BM - 1) / BM;                   // 128-row query tiles per head
  const int NP = (NB + 1) / 2;                        // pairs of tiles per head
  const int NKB = (N + BN - 1) / BN;                  // 256-key blocks per head
  Item it;
  it.key0 = (i / NP) * N;
  it.pair = NP - 1 - i % NP;
  it.n = causal ? it.pair + 1 : NKB;
  return it;
}

__global__ void __launch_bounds__(THREADS, 1)
prefill_2sm_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, __nv_bfloat16* __restrict__ out,
                   float* __restrict__ lse, int N, int causal, float scale_log2, int num_items) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;                                 // two buffers
  uint8_t* sK = smem + 2 * TILE_BYTES;
  uint8_t* sV = sK + STAGES * TILE_BYTES;
  Shared* sh = reinterpret_cast<Shared*>(sV + STAGES * TILE_BYTES);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rank = (int)tc::cluster_ctarank();        // 0 or 1
  const int cluster = (int)(blockIdx.x >> 1), nclusters = (int)(gridDim.x >> 1);
  const int NKB = (N + BN - 1) / BN;

  if (threadIdx.x == 0) {
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&sh->q_full[b], 1);
      tc::mbar_init(&sh->q_empty[b], 1);
    }
    for (int s = 0; s < STAGES; ++s) {
      tc::mbar_init(&sh->k_full[s], 1);
      tc::mbar_init(&sh->v_full[s], 1);
      tc::mbar_init(&sh->k_empty[s], 1);
      tc::mbar_init(&sh->v_empty[s], 1);
    }
    tc::mbar_init(&sh->s_full, 1);
    tc::mbar_init(&sh->pv_done, 1);
    tc::mbar_init(&sh->s_free, 2 * SM_WARPS);
    tc::mbar_init(&sh->p_ready, 2 * SM_WARPS);
    tc::mbar_init(&sh->o_free, 2 * SM_WARPS);
    for (int q = 0; q < 4; ++q) tc::mbar_init(&sh->red_bar[q], 2);
    sh->abort = 0;
    tc::fence_barrier_init();
  }
  if (warp == MMA_WARP) tc::tmem_alloc_pair(&sh->tmem_base, TMEM_COLS);
  tc::fence_before_sync();
  // both CTAs' barriers are initialised before any copy, commit or arrival
  // reaches them
  tc::cluster_sync();
  tc::fence_after_sync();
  const uint32_t tmem = sh->tmem_base;
  volatile int* abort = &sh->abort;

  if (warp == TMA_WARP) {
    // ------------------------------------------------------ TMA ----
    if (lane == 0) {
      tc::prefetch_tmap(&tmQ);
      tc::prefetch_tmap(&tmK);
      tc::prefetch_tmap(&tmV);
      uint32_t g = 0;                                 // key blocks loaded so far
      bool ok = true;
      for (int t = 0; ok; ++t) {
        const int i = item_index(t, cluster, nclusters);
        if (i >= num_items) break;
        const Item it = item_of(i, N, causal);
        const int qb = t & 1;
        if (!(ok = tc::mbar_wait(&sh->q_empty[qb], ((uint32_t)(t >> 1) & 1u) ^ 1u, abort))) break;
        if (rank == 0) tc::mbar_arrive_expect_tx(&sh->q_full[qb], 2 * TILE_BYTES);
        const uint32_t q_full0 = tc::mapa(tc::smem_u32(&sh->q_full[qb]), 0);
        const int qrow = it.key0 + (2 * it.pair + rank) * BM;
        tc::tma_load_2d_pair(sQ + qb * TILE_BYTES, &tmQ, q_full0, 0, qrow);
        tc::tma_load_2d_pair(sQ + qb * TILE_BYTES + HALF_BYTES, &tmQ, q_full0, 64, qrow);
        for (int j = 0; j < it.n; ++j, ++g) {
          const int s = (int)(g & 1u);
          const uint32_t ph = (g >> 1) & 1u;
          if (!(ok = tc::mbar_wait(&sh->k_empty[s], ph ^ 1u, abort))) break;
          if (rank == 0) tc::mbar_arrive_expect_tx(&sh->k_full[s], 2 * TILE_BYTES);
          const uint32_t k_full0 = tc::mapa(tc::smem_u32(&sh->k_full[s]), 0);
          uint8_t* k = sK + s * TILE_BYTES;
          const int krow = it.key0 + j * BN + rank * (BN / 2);
          tc::tma_load_2d_pair(k, &tmK, k_full0, 0, krow);
          tc::tma_load_2d_pair(k + HALF_BYTES, &tmK, k_full0, 64, krow);
          if (!(ok = tc::mbar_wait(&sh->v_empty[s], ph ^ 1u, abort))) break;
          if (rank == 0) tc::mbar_arrive_expect_tx(&sh->v_full[s], 2 * TILE_BYTES);
          const uint32_t v_full0 = tc::mapa(tc::smem_u32(&sh->v_full[s]), 0);
          tc::tma_load_2d_pair(sV + s * TILE_BYTES, &tmV, v_full0, rank * 64, it.key0 + j * BN);
        }
      }
    }
  } else if (warp == MMA_WARP) {
    // ------------------------------------------------------ MMA ----
    if (lane == 0 && rank == 0) {
      constexpr uint32_t idesc_s = tc::idesc_bf16_f32(2 * BM, BN, false);
      constexpr uint32_t idesc_pv = tc::idesc_bf16_f32(2 * BM, HD, true);
      // first K-step descriptors; a K-step adds its byte offset >> 4
      const uint64_t q_desc0 = tc::sdesc_sw128(tc::smem_u32(sQ), 16, 1024);
      const uint64_t q_desc1 = tc::sdesc_sw128(tc::smem_u32(sQ + TILE_BYTES), 16, 1024);
      static_assert(STAGES == 2, "one descriptor per stage, picked by g & 1");
      const uint64_t k_desc0 = tc::sdesc_sw128(tc::smem_u32(sK), 16, 1024);
      const uint64_t k_desc1 = tc::sdesc_sw128(tc::smem_u32(sK + TILE_BYTES), 16, 1024);
      // V halves are MN-major: 128-byte rows of 64 head-dimension columns,
      // 8-key groups 1 KiB apart (one swizzle atom wide, so the leading
      // offset is not used)
      const uint64_t v_desc0 = tc::sdesc_sw128(tc::smem_u32(sV), TILE_BYTES, 1024);
      const uint64_t v_desc1 = tc::sdesc_sw128(tc::smem_u32(sV + TILE_BYTES), TILE_BYTES, 1024);
      // S(g) = Q K^T from Q buffer qb: eight K-steps of 16 head-dimension
      // columns; the second 64 columns sit in the second swizzled box.  The
      // item's last S also releases its Q buffer.
      auto issue_s = [&](uint32_t g, int qb, bool last_of_item) -> bool {
        const int s = (int)(g & 1u);
        if (!tc::mbar_wait(&sh->k_full[s], (g >> 1) & 1u, abort)) return false;
        tc::fence_after_sync();
        const uint64_t kd = s ? k_desc1 : k_desc0;
        const uint64_t qd = qb ? q_desc1 : q_desc0;
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const uint64_t off = (uint64_t)(((kk >> 2) * HALF_BYTES + (kk & 3) * 32) >> 4);
          tc::mma_pair_f16_ss(tmem + S_COL, qd + off, kd + off, idesc_s, kk != 0);
        }
        tc::commit_pair_both(&sh->s_full);
        tc::commit_pair_both(&sh->k_empty[s]);
        if (last_of_item) tc::commit_pair_both(&sh->q_empty[qb]);
        return true;
      };
      // O [+]= P V(g): sixteen K-steps of 16 keys (8 TMEM columns of P, 2 KiB of V)
      auto issue_pv = [&](uint32_t g, bool accumulate) -> bool {
        const int s = (int)(g & 1u);
        if (!tc::mbar_wait(&sh->v_full[s], (g >> 1) & 1u, abort)) return false;
        tc::fence_after_sync();
        const uint64_t vd = s ? v_desc1 : v_desc0;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          tc::mma_pair_f16_ts(tmem + O_COL, tmem + P_COL + (uint32_t)(kk * 8),
                              vd + (uint64_t)((kk * 2048) >> 4), idesc_pv,
                              (accumulate || kk > 0) ? 1u : 0u);
        tc::commit_pair_both(&sh->pv_done);
        tc::commit_pair_both(&sh->v_empty[s]);
        return true;
      };
      // the first item's first S; then per block g: S(g + 1) (of this item or
      // the next) as soon as S(g) has been read, then P V(g) once P(g) is in
      bool ok = item_index(0, cluster, nclusters) < num_items;
      if (ok) {
        const Item first = item_of(item_index(0, cluster, nclusters), N, causal);
        ok = tc::mbar_wait(&sh->q_full[0], 0, abort) && issue_s(0, 0, first.n == 1);
      }
      uint32_t g = 0;
      for (int t = 0; ok; ++t) {
        const int i = item_index(t, cluster, nclusters);
        if (i >= num_items) break;
        const Item it = item_of(i, N, causal);
        const int i_next = item_index(t + 1, cluster, nclusters);
        const bool has_next = i_next < num_items;
        for (int j = 0; ok && j < it.n; ++j, ++g) {
          if (j + 1 < it.n || has_next) {
            // S(g + 1) overwrites S(g): both CTAs' softmax warps have read it
            if (!(ok = tc::mbar_wait(&sh->s_free, g & 1u, abort))) break;
            if (j + 1 < it.n) {
              ok = issue_s(g + 1, t & 1, j + 2 == it.n);
            } else {
              const int n_next = item_of(i_next, N, causal).n;
              const int qb = (t + 1) & 1;
              ok = tc::mbar_wait(&sh->q_full[qb], ((uint32_t)(t + 1) >> 1) & 1u, abort) &&
                   issue_s(g + 1, qb, n_next == 1);
            }
            if (!ok) break;
          }
          if (!(ok = tc::mbar_wait(&sh->p_ready, g & 1u, abort))) break;
          // the item's first P V overwrites O: the last item's O has been read
          if (j == 0 && t > 0 && !(ok = tc::mbar_wait(&sh->o_free, (uint32_t)(t - 1) & 1u, abort)))
            break;
          ok = issue_pv(g, j > 0);
        }
      }
    }
  } else {
    // --------------------------------------------------- softmax ----
    const int quarter = warp & 3;                   // TMEM lanes 32 quarter .. + 31
    const int kh = warp >> 2;                       // keys 128 kh .. + 127 of each block
    const int r = quarter * 32 + lane;              // this thread's row of the tile
    const uint32_t lanes = tmem + ((uint32_t)(quarter * 32) << 16);
    const uint32_t s_free0 = tc::mapa(tc::smem_u32(&sh->s_free), 0);
    const uint32_t p_ready0 = tc::mapa(tc::smem_u32(&sh->p_ready), 0);
    const uint32_t o_free0 = tc::mapa(tc::smem_u32(&sh->o_free), 0);
    const uint64_t sl2 = pack_f32x2(scale_log2, scale_log2);
    const bool out32 = (reinterpret_cast<uintptr_t>(out) & 31u) == 0;
    uint32_t g = 0, x = 0;                          // blocks and red_bar exchanges so far
    bool ok = true;
    const long long heads = (long long)num_items / ((((N + BM - 1) / BM) + 1) / 2);
    (void)heads;                                    // read by the checked build only
    bool pend = false;                              // an item's output is still to be written
    float pend_m = 0.f, pend_l = 0.f;
    int pend_row = 0;
    bool pend_in = false;
    // O columns 64 kh .. + 63 of this thread's row
    auto load_o = [&](uint32_t (&v)[64]) {
      uint32_t (&v0)[32] = *reinterpret_cast<uint32_t(*)[32]>(&v[0]);
      uint32_t (&v1)[32] = *reinterpret_cast<uint32_t(*)[32]>(&v[32]);
      tc::tmem_ld_32x32b_x32(lanes + O_COL + (uint32_t)(kh * 64), v0);
      tc::tmem_ld_32x32b_x32(lanes + O_COL + (uint32_t)(kh * 64 + 32), v1);
      tc::tmem_ld_wait();
    };
    auto finish = [&](const uint32_t (&v)[64]) -> bool {
      sh->part_l[kh][r] = pend_l;
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&sh->red_bar[quarter]);
      if (!tc::mbar_wait(&sh->red_bar[quarter], x & 1u, abort)) return false;
      ++x;
      const float lt = sh->part_l[0][r] + sh->part_l[1][r];
      const float inv = 1.f / lt;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        uint32_t pkd[16];
#pragma unroll
        for (int c = 0; c < 16; ++c)
          pkd[c] = pack_bf16x2(__uint_as_float(v[32 * hh + 2 * c]) * inv,
                               __uint_as_float(v[32 * hh + 2 * c + 1]) * inv);
        const int col = kh * 64 + hh * 32;
        if (pend_in && RF_SPAN_OK((size_t)pend_row * HD + col, 32, heads * N * HD)) {
          __nv_bfloat16* dst = out + (size_t)pend_row * HD + col;
          if (out32) {
            st_global_v8(dst, pkd);
            st_global_v8(dst + 16, pkd + 8);
          } else {
            uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
            for (int c = 0; c < 4; ++c)
              d4[c] = make_uint4(pkd[4 * c], pkd[4 * c + 1], pkd[4 * c + 2], pkd[4 * c + 3]);
          }
        }
      }
      if (lse != nullptr && kh == 0 && pend_in && RF_IDX_OK(pend_row, heads * N))
        lse[pend_row] = (pend_m + log2f(lt)) * kLn2;
      return true;
    };
    for (int t = 0; ok; ++t) {
      const int i = item_index(t, cluster, nclusters);
      if (i >= num_items) break;
      const Item it = item_of(i, N, causal);
      const int m_tile = 2 * it.pair + rank;
      float m_ref = -INFINITY, l = 0.f;
      for (int j = 0; j < it.n; ++j, ++g) {
        if (!(ok = tc::mbar_wait(&sh->s_full, g & 1u, abort))) break;
        tc::fence_after_sync();
        float s[128];                               // s[c] = key 128 kh + c of block j
        {
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint32_t (&v)[32] = *reinterpret_cast<uint32_t(*)[32]>(&s[32 * q4]);
            tc::tmem_ld_32x32b_x32(lanes + S_COL + (uint32_t)(kh * 128 + 32 * q4), v);
          }
          tc::tmem_ld_wait();
        }
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) arrive_cluster_relaxed(s_free0);
        if (causal && j == it.n - 1) {
          const int lim = BM * rank + r - kh * 128;
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (c > lim) s[c] = -INFINITY;
        } else if (!causal && j == NKB - 1 && N % BN != 0) {
          const int kmax = N - j * BN - kh * 128;
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (c >= kmax) s[c] = -INFINITY;
        }
        float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int c = 0; c < 128; c += 2) mx[(c >> 1) & 3] = max3(mx[(c >> 1) & 3], s[c], s[c + 1]);
        float* red = &sh->red[x & 1u][0][0];
        red[kh * BM + r] = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&sh->red_bar[quarter]);
        if (!(ok = tc::mbar_wait(&sh->red_bar[quarter], x & 1u, abort))) break;
        ++x;
        const float pm = fmaxf(red[r], red[BM + r]);
        const float mt = pm * scale_log2;
        const bool move = mt > m_ref + RESCALE_THRESHOLD;
        const float m_new = move ? mt : m_ref;
        const float alpha = ex2(m_ref - m_new);
        l *= alpha;
        m_ref = m_new;
        uint32_t w[64];
        {
          const uint64_t nm2 = pack_f32x2(-m_new, -m_new);
          uint64_t sum2 = 0ull;
#pragma unroll
          for (int c = 0; c < 64; ++c) {
            float a0, a1;
            unpack_f32x2(fma_f32x2(pack_f32x2(s[2 * c], s[2 * c + 1]), sl2, nm2), a0, a1);
            const float p0 = ex2(a0), p1 = ex2(a1);
            sum2 = add_f32x2(sum2, pack_f32x2(p0, p1));
            w[c] = pack_bf16x2(p0, p1);
          }
          float s0, s1;
          unpack_f32x2(sum2, s0, s1);
          l += s0 + s1;
        }
        if (j > 0) {
          if (!(ok = tc::mbar_wait(&sh->pv_done, (g - 1) & 1u, abort))) break;
          tc::fence_after_sync();
          if (__any_sync(0xffffffffu, move)) {
#pragma unroll 1
            for (int hh = 0; hh < 2; ++hh) {
              const uint32_t oc = lanes + O_COL + (uint32_t)(kh * 64 + hh * 32);
              uint32_t v[32];
              tc::tmem_ld_32x32b_x32(oc, v);
              tc::tmem_ld_wait();
#pragma unroll
              for (int c = 0; c < 32; ++c) v[c] = __float_as_uint(__uint_as_float(v[c]) * alpha);
              tc::tmem_st_32x32b_x32(oc, v);
            }
          }
        }
        const bool have_o = j == 0 && pend;
        if (have_o) {
          if (!(ok = tc::mbar_wait(&sh->pv_done, (g - 1) & 1u, abort))) break;
          tc::fence_after_sync();
        }
        {
          uint32_t (&w0)[32] = *reinterpret_cast<uint32_t(*)[32]>(&w[0]);
          uint32_t (&w1)[32] = *reinterpret_cast<uint32_t(*)[32]>(&w[32]);
          tc::tmem_st_32x32b_x32(lanes + P_COL + (uint32_t)(kh * 64), w0);
          tc::tmem_st_32x32b_x32(lanes + P_COL + (uint32_t)(kh * 64 + 32), w1);
        }
        tc::tmem_st_wait();
        if (have_o) {
          uint32_t ov[64];
          load_o(ov);
          tc::fence_before_sync();
          __syncwarp();
          if (lane == 0) {
            arrive_cluster_relaxed(o_free0);
            arrive_cluster_relaxed(p_ready0);
          }
          if (!(ok = finish(ov))) break;
          pend = false;
        } else {
          tc::fence_before_sync();
          __syncwarp();
          if (lane == 0) arrive_cluster_relaxed(p_ready0);
        }
      }
      if (!ok) break;
      pend = true;
      pend_m = m_ref;
      pend_l = l;
      pend_row = it.key0 + m_tile * BM + r;
      pend_in = m_tile * BM + r < N;
    }
    if (ok && pend) {
      if (tc::mbar_wait(&sh->pv_done, (g - 1) & 1u, abort)) {
        tc::fence_after_sync();
        uint32_t ov[64];
        load_o(ov);
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) arrive_cluster_relaxed(o_free0);
        finish(ov);
      }
    }
  }

  tc::fence_before_sync();
  __syncwarp();
  // neither CTA leaves while the other may still copy, commit or arrive into it
  tc::cluster_sync();
  if (warp == MMA_WARP) {
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

// clusters of two of these CTAs that are resident at once on the current
// device (cached per device); 0 when none fits
int resident_pairs() {
  static std::atomic<int> count[64];
  static std::atomic<uint64_t> attr_done{0}, known{0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  const uint64_t bit = 1ull << dev;
  if (known.load(std::memory_order_acquire) & bit) return count[dev].load();
  int n = 0;
  if (smem_attr(prefill_2sm_kernel, SMEM_BYTES, attr_done) == RF_OK) {
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = pair_config(attr, 2u, 0);
    if (cudaOccupancyMaxActiveClusters(&n, prefill_2sm_kernel, &cfg) != cudaSuccess) n = 0;
  }
  cudaGetLastError();
  count[dev].store(n);
  known.fetch_or(bit, std::memory_order_release);
  return n;
}

}  // namespace

// RF_ERR_UNSUPPORTED when a cluster of two of these CTAs cannot be resident
// on the device (or the item count overflows an int).
rf_status launch_prefill(const void* q, const void* k, const void* v, int B, int H, int N, int D,
                         int causal, float scale, void* out, float* lse, cudaStream_t st) {
  (void)D;                                      // 128, checked by the caller
  const int pairs = resident_pairs();
  if (pairs <= 0) return RF_ERR_UNSUPPORTED;
  const uint64_t rows = (uint64_t)B * H * N;
  CUtensorMap tq, tk, tv;
  const uint64_t stride = HD * 2;
  if (!tc::make_tmap_2d(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, q, HD, rows, stride, 64, BM,
                        CU_TENSOR_MAP_SWIZZLE_128B) ||
      !tc::make_tmap_2d(&tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, k, HD, rows, stride, 64, BN / 2,
                        CU_TENSOR_MAP_SWIZZLE_128B) ||
      !tc::make_tmap_2d(&tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, v, HD, rows, stride, 64, BN,
                        CU_TENSOR_MAP_SWIZZLE_128B))
    return RF_ERR_CUDA;
  const int NB = (N + BM - 1) / BM;
  const long long items = (long long)B * H * ((NB + 1) / 2);
  if (items > INT32_MAX) return RF_ERR_UNSUPPORTED;
  const int clusters = (int)(pairs < items ? pairs : items);
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pair_config(attr, 2u * (unsigned)clusters, st);
  if (cudaLaunchKernelEx(&cfg, prefill_2sm_kernel, tq, tk, tv, static_cast<__nv_bfloat16*>(out),
                         lse, N, causal, scale * kLog2e, (int)items) != cudaSuccess) {
    cudaGetLastError();
    return RF_ERR_CUDA;
  }
  return launch_status();
}

RF_TIMEOUT_WORD_OF_THIS_FILE

RF_BOUNDS_WORD_OF_THIS_FILE

}  // namespace rf
