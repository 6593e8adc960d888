// Multi-latent attention (MLA) decode, split over key segments, on tcgen05.
//
// The cascade is the attention one (RedFuser episode transcript, cue 9: row
// max, exp-sum, weighted sum) with every query head of a sequence reading one
// shared latent cache C [L, 576]: scores s_hj = scale <q_h, c_j>, values are
// the leading 512 latent dims (cues 41 and 55: the MLA workload, decode with
// one query row).  The key sequence is split into segments whose (m, l, acc)
// states rf_state_merge combines (cue 39, Multi-Segment).
//
// The contraction is laid out transposed: keys go down the 128 TMEM lanes and
// the query heads across the columns, so both products are M = 128 tcgen05
// MMAs however few heads there are:
//   S^T [128 keys x HG heads]  = C_tile [128 x 576] . Q^T [576 x HG]
//   O^T [512 dv  x HG heads] += C_tile[:, :512]^T [512 x 128] . P^T [128 x HG]
// (O^T as four 128-lane column blocks of HG columns).  HG, the heads a CTA
// handles, is 16 or 32; O^T and S^T then take at most 160 TMEM columns,
// where the untransposed form would need all 512 for O alone.
//
// Shared memory holds the whole 144 KiB latent tile of the current 128 keys
// until its P V product is done: the 512 value dims in "pair" slots of 32 KiB
// (two 64-dim boxes with 128-byte swizzle, 16 KiB apart, which is the layout
// the MN-major V^T operand descriptor expects) and the 64 rotary dims in a
// rope slot.  Five pair slots leave one for the next tile while the current
// one is in use.
//
// Each pair slot is released as soon as the O^T MMAs that read it complete,
// so the next tile's loads start during the current tile's P V product.
//
// Warps: 0 TMA, 1 MMA (and TMEM owner), 2-9 softmax: two warps per TMEM lane
// quarter, each thread one key of the tile (one TMEM lane) and half of the
// heads, so each SM sub-partition interleaves two short softmax chains.  Persistent CTAs take contiguous ranges of
// (sequence, head group, segment) units, so Q is reloaded only when the
// sequence or head group changes.
//
// Per tile: S^T MMAs (rope chunk first, then the eight value chunks); each
// softmax thread loads its key's scores for its HG/2 heads, the tile max per
// head is reduced over the warp (redux on order-preserving integer keys) and
// over the four lane quarters (shared memory + an mbarrier per head half), the reference max moves lazily (only
// when a head's tile max exceeds it by more than 8 in log2 units, rescaling
// that head's column of O^T in TMEM and its partial l), P^T is written to
// shared memory as bf16 in the 128-byte-swizzled K-major layout, and the MMA
// thread issues the O^T MMAs (l sums the same bf16-rounded weights, so the
// merged output is a convex combination of the value rows).  At the end of a
// unit the states are written relative to the true segment max: l and acc
// are multiplied by exp2(m_ref - m_true) <= 1 on the way out.
// Every wait is bounded (see tc_common.cuh).

#include <cuda_bf16.h>

#include "tc_common.cuh"

namespace rf {
namespace {

constexpr int DK = 576;                    // latent width (512 value dims + 64 rotary)
constexpr int DV = 512;
constexpr int BK = 128;                    // keys per tile
constexpr int CHUNK = BK * 128;            // one 64-dim box of a tile: 16 KiB
constexpr int PAIR = 2 * CHUNK;            // 128 value dims: 32 KiB
constexpr int NPAIR = 5;                   // pair slots (4 per tile + 1 ahead)
constexpr int THREADS = 10 * 32;          // TMA, MMA, 8 softmax warps
constexpr int TMA_WARP = 0, MMA_WARP = 1;
constexpr int TMEM_COLS = 256;
constexpr uint32_t S_COL = 0;              // S^T: HG columns
constexpr uint32_t O_COL = 32;             // O^T: 4 blocks of HG columns
constexpr float RESCALE_THRESHOLD = 8.0f;  // log2 units

struct MlaShared {
  uint64_t q_full, q_empty;
  uint64_t rope_full, rope_empty;
  uint64_t pair_full[NPAIR], pair_empty[NPAIR];
  uint64_t s_full, p_full, o_done;
  uint64_t red_ready[2][2], l_ready, drain;     // red_ready[tile parity][head half]
  float red[2][4][32];                     // [tile parity][warp][head] tile maxima
  float lred[4][32];                       // [warp][head] partial l
  uint32_t tmem_base;
  int abort;
};

template <int HG>
struct Layout {
  static constexpr int Q_BYTES = 9 * HG * 128;    // nine 64-dim chunks of HG rows
  static constexpr int P_BYTES = 2 * HG * 128;    // two 64-key chunks of HG rows
  static constexpr int PAIRS = Q_BYTES + P_BYTES;
  static constexpr int ROPE = PAIRS + NPAIR * PAIR;
  static constexpr int SHARED = ROPE + CHUNK;
  static constexpr size_t SMEM = (size_t)SHARED + sizeof(MlaShared) + 1024;
  static_assert(SMEM <= 232448, "exceeds the 227 KiB of shared memory a CTA may use");
  static_assert(Q_BYTES % 1024 == 0 && P_BYTES % 1024 == 0, "swizzled tiles need 1 KiB alignment");
};

struct Unit {
  int b, g, s, a, e, nt;                   // sequence, head group, segment, keys [a, e), tiles
};

__device__ __forceinline__ Unit unit_of(long long u, int G, int S, int L, int seg) {
  Unit x;
  x.s = (int)(u % S);
  const long long r = u / S;
  x.g = (int)(r % G);
  x.b = (int)(r / G);
  x.a = min(L, x.s * seg);
  x.e = min(L, x.a + seg);
  x.nt = (x.e - x.a + BK - 1) / BK;
  return x;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// float -> unsigned key with the same order (for integer redux)
__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float order_key_inv(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

__device__ __forceinline__ uint32_t idesc_bf16(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

template <int HG>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&r)[HG]);
template <>
__device__ __forceinline__ void tmem_ld_cols<8>(uint32_t taddr, uint32_t (&r)[8]) {
  tc::tmem_ld_32x32b_x8(taddr, r);
}
template <>
__device__ __forceinline__ void tmem_ld_cols<16>(uint32_t taddr, uint32_t (&r)[16]) {
  tc::tmem_ld_32x32b_x16(taddr, r);
}
template <>
__device__ __forceinline__ void tmem_ld_cols<32>(uint32_t taddr, uint32_t (&r)[32]) {
  tc::tmem_ld_32x32b_x32(taddr, r);
}
template <int N>
__device__ __forceinline__ void tmem_st_cols(uint32_t taddr, const uint32_t (&r)[N]) {
  if constexpr (N == 8) {
    tc::tmem_st_32x32b_x8(taddr, r);
  } else {
#pragma unroll
    for (int h0 = 0; h0 < N; h0 += 16) {
      uint32_t w[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) w[i] = r[h0 + i];
      tc::tmem_st_32x32b_x16(taddr + (uint32_t)h0, w);
    }
  }
}

template <int HG>
__global__ void __launch_bounds__(THREADS, 1)
mla_decode_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmC,
                  int H, int L, int S, int seg, long long units, float scale_log2,
                  float* __restrict__ seg_m, float* __restrict__ seg_l,
                  float* __restrict__ seg_acc) {
  using Lay = Layout<HG>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;
  uint8_t* sP = smem + Lay::Q_BYTES;
  uint8_t* sPair = smem + Lay::PAIRS;
  uint8_t* sRope = smem + Lay::ROPE;
  MlaShared* sh = reinterpret_cast<MlaShared*>(smem + Lay::SHARED);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = H / HG;
  const long long u0 = units * blockIdx.x / gridDim.x;
  const long long u1 = units * (blockIdx.x + 1) / gridDim.x;

  if (threadIdx.x == 0) {
    tc::mbar_init(&sh->q_full, 1);
    tc::mbar_init(&sh->q_empty, 1);
    tc::mbar_init(&sh->rope_full, 1);
    tc::mbar_init(&sh->rope_empty, 1);
    for (int i = 0; i < NPAIR; ++i) {
      tc::mbar_init(&sh->pair_full[i], 1);
      tc::mbar_init(&sh->pair_empty[i], 1);
    }
    tc::mbar_init(&sh->s_full, 1);
    tc::mbar_init(&sh->p_full, 8);
    tc::mbar_init(&sh->o_done, 1);
    for (int i = 0; i < 2; ++i)
      for (int j = 0; j < 2; ++j) tc::mbar_init(&sh->red_ready[i][j], 4);
    tc::mbar_init(&sh->l_ready, 8);
    tc::mbar_init(&sh->drain, 1);
    sh->abort = 0;
    tc::fence_barrier_init();
  }
  if (warp == MMA_WARP) tc::tmem_alloc(&sh->tmem_base, TMEM_COLS);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = sh->tmem_base;
  volatile int* abort = &sh->abort;

  // does the unit after u (within this CTA's range, skipping empty ones) use
  // another Q block?
  auto q_changes_after = [&](long long u, const Unit& x) -> bool {
    for (long long v = u + 1; v < u1; ++v) {
      const Unit y = unit_of(v, G, S, L, seg);
      if (y.nt == 0) continue;
      return y.b != x.b || y.g != x.g;
    }
    return true;
  };

  if (warp == TMA_WARP) {
    // ------------------------------------------------------------ TMA ----
    if (lane == 0) {
      tc::prefetch_tmap(&tmQ);
      tc::prefetch_tmap(&tmC);
      uint32_t nq = 0, nr = 0, np = 0;
      int qb = -1, qg = -1;
      bool ok = true;
      for (long long u = u0; u < u1 && ok; ++u) {
        const Unit x = unit_of(u, G, S, L, seg);
        if (x.nt == 0) continue;
        if (x.b != qb || x.g != qg) {
          if (!(ok = tc::mbar_wait(&sh->q_empty, (nq & 1u) ^ 1u, abort))) break;
          tc::mbar_arrive_expect_tx(&sh->q_full, Lay::Q_BYTES);
          for (int c = 0; c < 9; ++c)
            tc::tma_load_2d(sQ + c * HG * 128, &tmQ, &sh->q_full, 64 * c, x.b * H + x.g * HG);
          ++nq;
          qb = x.b;
          qg = x.g;
        }
        for (int t = 0; t < x.nt && ok; ++t) {
          const int row = x.b * L + x.a + t * BK;
          if (!(ok = tc::mbar_wait(&sh->rope_empty, (nr & 1u) ^ 1u, abort))) break;
          tc::mbar_arrive_expect_tx(&sh->rope_full, CHUNK);
          tc::tma_load_2d(sRope, &tmC, &sh->rope_full, DV, row);
          ++nr;
          for (int p = 0; p < 4; ++p) {
            const uint32_t slot = np % NPAIR, ph = (np / NPAIR) & 1u;
            if (!(ok = tc::mbar_wait(&sh->pair_empty[slot], ph ^ 1u, abort))) break;
            uint8_t* dst = sPair + slot * PAIR;
            tc::mbar_arrive_expect_tx(&sh->pair_full[slot], PAIR);
            tc::tma_load_2d(dst, &tmC, &sh->pair_full[slot], 128 * p, row);
            tc::tma_load_2d(dst + CHUNK, &tmC, &sh->pair_full[slot], 128 * p + 64, row);
            ++np;
          }
        }
      }
      // let every copy this thread started land before the CTA can exit
      if (nq > 0) tc::mbar_wait(&sh->q_full, (nq - 1) & 1u, abort);
      if (nr > 0) tc::mbar_wait(&sh->rope_full, (nr - 1) & 1u, abort);
      for (uint32_t i = 0; i < NPAIR && i < np; ++i) {
        const uint32_t n = np - 1 - i;              // the last load into slot n % NPAIR
        tc::mbar_wait(&sh->pair_full[n % NPAIR], (n / NPAIR) & 1u, abort);
      }
    }
  } else if (warp == MMA_WARP) {
    // ------------------------------------------------------------ MMA ----
    if (lane == 0) {
      const uint32_t idesc_s = idesc_bf16(BK, HG, false, false);
      const uint32_t idesc_o = idesc_bf16(BK, HG, true, false);
      const uint32_t q_addr = tc::smem_u32(sQ), p_addr = tc::smem_u32(sP);
      const uint32_t pair_addr = tc::smem_u32(sPair), rope_addr = tc::smem_u32(sRope);
      uint32_t nq = 0, nr = 0, np = 0, nt_all = 0;
      int qb = -1, qg = -1;
      bool ok = true;
      for (long long u = u0; u < u1 && ok; ++u) {
        const Unit x = unit_of(u, G, S, L, seg);
        if (x.nt == 0) continue;
        if (x.b != qb || x.g != qg) {
          if (!(ok = tc::mbar_wait(&sh->q_full, nq & 1u, abort))) break;
          ++nq;
          qb = x.b;
          qg = x.g;
        }
        const bool q_last = q_changes_after(u, x);
        for (int t = 0; t < x.nt && ok; ++t, ++nt_all) {
          // S^T = C_tile Q^T, rope chunk first
          if (!(ok = tc::mbar_wait(&sh->rope_full, nr & 1u, abort))) break;
          tc::fence_after_sync();
#pragma unroll
          for (int k = 0; k < 4; ++k)
            tc::mma_f16_ss(tmem + S_COL, tc::sdesc_sw128(rope_addr + 32 * k, 16, 1024),
                           tc::sdesc_sw128(q_addr + 8 * HG * 128 + 32 * k, 16, 1024), idesc_s,
                           k != 0);
          uint32_t slots[4];
          for (int p = 0; p < 4 && ok; ++p) {
            const uint32_t n = np + p, slot = n % NPAIR;
            slots[p] = slot;
            if (!(ok = tc::mbar_wait(&sh->pair_full[slot], (n / NPAIR) & 1u, abort))) break;
            tc::fence_after_sync();
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
              for (int k = 0; k < 4; ++k)
                tc::mma_f16_ss(
                    tmem + S_COL,
                    tc::sdesc_sw128(pair_addr + slot * PAIR + h * CHUNK + 32 * k, 16, 1024),
                    tc::sdesc_sw128(q_addr + (2 * p + h) * HG * 128 + 32 * k, 16, 1024),
                    idesc_s, 1u);
          }
          if (!ok) break;
          tc::mma_commit(&sh->s_full);
          tc::mma_commit(&sh->rope_empty);
          ++nr;
          if (t == x.nt - 1 && q_last) tc::mma_commit(&sh->q_empty);
          // O^T += V^T P^T once the softmax has written P^T
          if (!(ok = tc::mbar_wait(&sh->p_full, nt_all & 1u, abort))) break;
          tc::fence_after_sync();
          for (int c = 0; c < 4; ++c) {
            const uint32_t v_addr = pair_addr + slots[c] * PAIR;
#pragma unroll
            for (int ks = 0; ks < BK / 16; ++ks)
              tc::mma_f16_ss(tmem + O_COL + (uint32_t)(c * HG),
                             tc::sdesc_sw128(v_addr + ks * 2048, CHUNK, 1024),
                             tc::sdesc_sw128(p_addr + (ks >> 2) * HG * 128 + (ks & 3) * 32, 16,
                                             1024),
                             idesc_o, (t > 0 || ks > 0) ? 1u : 0u);
            tc::mma_commit(&sh->pair_empty[slots[c]]);     // this pair is free once read
          }
          tc::mma_commit(&sh->o_done);
          np += 4;
        }
      }
      // every MMA issued above completes before TMEM is released
      tc::mma_commit(&sh->drain);
      tc::mbar_wait(&sh->drain, 0, abort);
    }
  } else {
    // -------------------------------------------------------- softmax ----
    // warps 2..9: two per TMEM lane quarter, each owning HW = HG/2 heads
    constexpr int HW = HG / 2;
    const int quarter = warp & 3;                   // TMEM lane quarter of this warp
    const int hh = (warp - 2) >> 2;                 // which half of the heads
    const int hb = hh * HW;                         // first head of this warp
    const int kt = quarter * 32 + lane;             // key of the tile = TMEM lane
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    uint32_t nt_all = 0, nunits = 0;
    bool ok = true;
    for (long long u = u0; u < u1 && ok; ++u) {
      const Unit x = unit_of(u, G, S, L, seg);
      const size_t st0 = ((size_t)x.b * H + (size_t)x.g * HG) * S + x.s;   // state of head 0
      if (x.nt == 0) {
        // empty segment: the identity state
        // (checked build) states: units * HG = B * H * S of them
        for (int i = threadIdx.x - 64; i < HG * DV; i += THREADS - 64)
          if (RF_IDX_OK((st0 + (size_t)(i / DV) * S) * DV + (i % DV), units * HG * DV))
            seg_acc[(st0 + (size_t)(i / DV) * S) * DV + (i % DV)] = 0.f;
        if (quarter == 0 && lane < HW && RF_IDX_OK(st0 + (size_t)(hb + lane) * S, units * HG)) {
          seg_m[st0 + (size_t)(hb + lane) * S] = -INFINITY;
          seg_l[st0 + (size_t)(hb + lane) * S] = 0.f;
        }
        continue;
      }
      float mref[HW], mtrue[HW], lp[HW];
#pragma unroll
      for (int h = 0; h < HW; ++h) {
        mref[h] = -INFINITY;
        mtrue[h] = -INFINITY;
        lp[h] = 0.f;
      }
      for (int t = 0; t < x.nt; ++t, ++nt_all) {
        if (!(ok = tc::mbar_wait(&sh->s_full, nt_all & 1u, abort))) break;
        tc::fence_after_sync();
        float sv[HW];
        {
          uint32_t r[HW];
          tmem_ld_cols<HW>(lane_base + S_COL + (uint32_t)hb, r);
          tc::tmem_ld_wait();
          const bool valid = x.a + t * BK + kt < x.e;
#pragma unroll
          for (int h = 0; h < HW; ++h) sv[h] = valid ? __uint_as_float(r[h]) * scale_log2 : -INFINITY;
        }
        // tile max per head: over the warp, then over the four lane quarters
        const int par = (int)(nt_all & 1u);
#pragma unroll
        for (int h = 0; h < HW; ++h) {
          const uint32_t k = __reduce_max_sync(0xffffffffu, order_key(sv[h]));
          if (lane == h) sh->red[par][quarter][hb + h] = order_key_inv(k);
        }
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&sh->red_ready[par][hh]);
        if (!(ok = tc::mbar_wait(&sh->red_ready[par][hh], (nt_all >> 1) & 1u, abort))) break;
        float alpha[HW];
        bool any_move = false;
#pragma unroll
        for (int h = 0; h < HW; ++h) {
          const float tm = fmaxf(fmaxf(sh->red[par][0][hb + h], sh->red[par][1][hb + h]),
                                 fmaxf(sh->red[par][2][hb + h], sh->red[par][3][hb + h]));
          mtrue[h] = fmaxf(mtrue[h], tm);
          const bool move = tm > mref[h] + RESCALE_THRESHOLD;
          const float mn = move ? tm : mref[h];
          alpha[h] = move ? ex2(mref[h] - mn) : 1.f;
          any_move |= move;
          mref[h] = mn;
        }
        // the previous tile's O^T MMAs must be done before P^T is overwritten
        // and before O^T is rescaled
        if (t > 0) {
          if (!(ok = tc::mbar_wait(&sh->o_done, (nt_all - 1) & 1u, abort))) break;
          tc::fence_after_sync();
          if (any_move) {
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
              const uint32_t oc = lane_base + O_COL + (uint32_t)(c * HG + hb);
              uint32_t r[HW];
              tmem_ld_cols<HW>(oc, r);
              tc::tmem_ld_wait();
#pragma unroll
              for (int h = 0; h < HW; ++h) r[h] = __float_as_uint(__uint_as_float(r[h]) * alpha[h]);
              tmem_st_cols<HW>(oc, r);
            }
            tc::tmem_st_wait();
          }
        }
        // P^T[h][kt] as bf16 into the K-major swizzled tile: row h, 64-key chunk kt / 64
        {
          uint8_t* chunk = sP + (kt >> 6) * HG * 128;
          const int gran = (kt & 63) >> 3;
#pragma unroll
          for (int j = 0; j < HW; ++j) {
            const int h = hb + j;
            // l sums the same bf16-rounded weights the MMA multiplies V by
            const __nv_bfloat16 pb = __float2bfloat16_rn(ex2(sv[j] - mref[j]));
            lp[j] = fmaf(lp[j], alpha[j], __bfloat162float(pb));
            const uint32_t off = (uint32_t)(h * 128 + ((gran ^ (h & 7)) << 4) + ((kt & 7) << 1));
            *reinterpret_cast<__nv_bfloat16*>(chunk + off) = pb;
          }
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&sh->p_full);
      }
      if (!ok) break;
      // ---- end of the unit: states relative to the true segment max
      if (!(ok = tc::mbar_wait(&sh->o_done, (nt_all - 1) & 1u, abort))) break;
      tc::fence_after_sync();
      float f[HW];
#pragma unroll
      for (int h = 0; h < HW; ++h) {
        f[h] = ex2(mref[h] - mtrue[h]);
        const float w = group_sum<32>(lp[h]);
        if (lane == h) sh->lred[quarter][hb + h] = w;
      }
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&sh->l_ready);
      if (!(ok = tc::mbar_wait(&sh->l_ready, nunits & 1u, abort))) break;
      ++nunits;
      if (quarter == 0 && lane < HW) {
        float fk = 0.f, mk = 0.f;
#pragma unroll
        for (int h = 0; h < HW; ++h)
          if (h == lane) {
            fk = f[h];
            mk = mtrue[h];
          }
        const int hd = hb + lane;
        const float lt = (sh->lred[0][hd] + sh->lred[1][hd]) + (sh->lred[2][hd] + sh->lred[3][hd]);
        if (RF_IDX_OK(st0 + (size_t)hd * S, units * HG)) {
          seg_l[st0 + (size_t)hd * S] = lt * fk;
          seg_m[st0 + (size_t)hd * S] = mk * kLn2;
        }
      }
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t r[HW];
        tmem_ld_cols<HW>(lane_base + O_COL + (uint32_t)(c * HG + hb), r);
        tc::tmem_ld_wait();
        float* dst = seg_acc + (st0 + (size_t)hb * S) * DV + c * BK + kt;
#pragma unroll
        for (int h = 0; h < HW; ++h)
          if (RF_IDX_OK((st0 + (size_t)(hb + h) * S) * DV + c * BK + kt, units * HG * DV))
            dst[(size_t)h * S * DV] = __uint_as_float(r[h]) * f[h];
      }
      tc::fence_before_sync();
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == MMA_WARP) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, TMEM_COLS);
  }
}

template <int HG>
rf_status launch_hg(const void* q, const void* c, int B, int H, int L, int S, float scale,
                    float* seg_m, float* seg_l, float* seg_acc, cudaStream_t st) {
  CUtensorMap tq, tcm;
  const uint64_t stride = DK * 2;
  if (!tc::make_tmap_2d(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, q, DK, (uint64_t)B * H, stride, 64,
                        HG, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !tc::make_tmap_2d(&tcm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, c, DK, (uint64_t)B * L, stride, 64,
                        BK, CU_TENSOR_MAP_SWIZZLE_128B))
    return RF_ERR_CUDA;
  auto kern = mla_decode_kernel<HG>;
  static std::atomic<uint64_t> attr{0};
  if (smem_attr(kern, Layout<HG>::SMEM, attr) != RF_OK) return RF_ERR_CUDA;
  const int seg = (L + S - 1) / S;
  const long long units = (long long)B * (H / HG) * S;
  const long long sms = tc::sm_count();
  const unsigned grid = (unsigned)(units < sms ? units : sms);
  kern<<<grid, THREADS, Layout<HG>::SMEM, st>>>(tq, tcm, H, L, S, seg, units, scale * kLog2e,
                                                seg_m, seg_l, seg_acc);
  return launch_status();
}

}  // namespace

rf_status launch_mla_decode(const void* q, const void* c, int B, int H, int L, int S, float scale,
                            float* seg_m, float* seg_l, float* seg_acc, cudaStream_t st) {
  if (H % 32 == 0) return launch_hg<32>(q, c, B, H, L, S, scale, seg_m, seg_l, seg_acc, st);
  return launch_hg<16>(q, c, B, H, L, S, scale, seg_m, seg_l, seg_acc, st);
}

RF_TIMEOUT_WORD_OF_THIS_FILE

RF_BOUNDS_WORD_OF_THIS_FILE

}  // namespace rf
