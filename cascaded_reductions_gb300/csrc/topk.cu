// MoE routing: softmax over experts, then top-k, from one read of each row.
//
// The cascade (RedFuser episode transcript, cue 11; "Online normalizer
// calculation for softmax", abstract on its citation page): the row max, the
// exp-sum denominator and the k largest entries all come from a single pass
// over the logits held in registers.
//
// Four kernels.  For k <= 2 and E a multiple of 32 up to 128,
// softmax_top2_row_kernel: one thread per token over a row staged in shared
// memory (below).  For E = 256 and k <= 8, softmax_top8_pair_kernel: two
// threads per token over a staged row (below).  For other E <= 128 (with
// k <= G), softmax_topk_merge_kernel:
// each lane keeps its best two logits and the group merges lane heads round by
// round (below).  Otherwise softmax_topk_kernel:
//
// Layout: a group of G lanes (G = 8, 16 or 32) owns TPG tokens, one after the
// other; lane g of the group holds NV logits of each token, loaded W at a
// time (W = 4, 2 or 1 consecutive floats, coalesced across the group).  With
// G < 32 several groups share each warp instruction, so the warp-level work
// per token shrinks with G; the group reductions use redux.sync / ballot /
// shuffles restricted to the group's lanes.  Values that enter a reduction
// are turned into order-preserving 32-bit keys (-0 is first mapped to +0, so
// keys compare exactly like the float values).
//   * plain rounds (small NV): round r of top-k: every lane proposes its
//     largest untaken slot (slots are visited in increasing expert index, so
//     among equal values the lowest index is proposed); the group takes the
//     maximum key with one redux.sync, then the minimum expert index among the
//     lanes proposing that key with a second; the owner marks it taken and
//     lane r keeps it.  Equal logits therefore come out in index order;
//   * threshold rounds (NV >= 8, G = 32): thr = the k-th largest of the 32
//     lane maxima (k rounds of redux.sync + ballot).  The k lanes supplying
//     those maxima hold k distinct elements >= thr, so the top k all lie at
//     or above thr.  The candidates >= thr (about k + 1 on random logits) are
//     compacted through shared memory to one per lane and the plain rounds
//     run on those single values.  If more than 32 survive (many ties), the
//     plain rounds run on every slot instead (same result);
//   * the row max m is round 0's key; with renormalisation the weights are
//     exp(x_i - m) / sum over the k selected, otherwise exp(x_i - m) / l with
//     l = sum over all E of exp(x - m);
//   * lanes r < k of the group store index and weight, one coalesced store
//     each.

#include <math.h>

#include "common.cuh"

namespace rf {
namespace {

constexpr uint32_t FULL = 0xffffffffu;


__device__ __forceinline__ uint32_t order_key(float x) {
  const uint32_t u = __float_as_uint(x + 0.0f);     // -0 -> +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ float key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// sum over the group's lanes (xor offsets below G stay inside the group)
template <int G>
__device__ __forceinline__ float gsum(float v, int upto) {
#pragma unroll
  for (int o = 1; o < G; o <<= 1)
    if (o < upto) v += __shfl_xor_sync(FULL, v, o);
  return v;
}

// G lanes per token, NV logits per lane (E <= G*NV), W consecutive logits per
// load, TPG tokens per group, KT = k when known at compile time (0: runtime),
// THRESH: use the threshold rounds.  Padding slots (expert index >= E) never
// take part.
template <int G, int NV, int W, int TPG, int KT, bool THRESH>
__global__ void __launch_bounds__(256)
softmax_topk_kernel(const float* __restrict__ logits, int T, int E, int k_rt, int renorm,
                    int32_t* __restrict__ idx_out, float* __restrict__ w_out) {
  static_assert(NV % W == 0 && NV <= 32 && 32 % G == 0, "layout");
  static_assert(!THRESH || G == 32, "threshold rounds use whole warps");
  constexpr int GPW = 32 / G;                       // groups per warp
  const int k = KT > 0 ? KT : k_rt;
  const int lane = threadIdx.x & 31;
  const int gl = lane & (G - 1);                    // lane within the group
  const int warp = threadIdx.x >> 5;
  const uint32_t gmask = G == 32 ? FULL : (((1u << G) - 1u) << (lane & ~(G - 1)));
  const int group_global = ((blockIdx.x * blockDim.x + threadIdx.x) >> 5) * GPW + (lane / G);
  const int tok0 = group_global * TPG;
  __shared__ float sm_val[8][32];
  __shared__ int sm_idx[8][32];

  // expert index of slot i of this lane
  auto expert = [&](int i) -> int { return (i / W) * G * W + gl * W + (i % W); };

  float x[TPG][NV];
#pragma unroll
  for (int t = 0; t < TPG; ++t) {
    const int token = tok0 + t;
    const bool live = token < T;
    const float* row = logits + (size_t)(live ? token : 0) * E;
#pragma unroll
    for (int c = 0; c < NV / W; ++c) {
      const int e0 = c * G * W + gl * W;
      const bool in = live && e0 < E && RF_SPAN_OK(e0, W, E) && RF_IDX_OK(token, T);
      if (W == 4) {
        const float4 f = in ? __ldcs(reinterpret_cast<const float4*>(row + e0))
                            : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        x[t][4 * c + 0] = f.x;
        x[t][4 * c + 1] = f.y;
        x[t][4 * c + 2] = f.z;
        x[t][4 * c + 3] = f.w;
      } else if (W == 2) {
        const float2 f = in ? __ldcs(reinterpret_cast<const float2*>(row + e0))
                            : make_float2(-INFINITY, -INFINITY);
        x[t][2 * c + 0] = f.x;
        x[t][2 * c + 1] = f.y;
      } else {
        x[t][c] = in ? __ldcs(row + e0) : -INFINITY;
      }
    }
  }
  // slots that hold a real expert (the same for every token of the group)
  uint32_t valid = 0u;
#pragma unroll
  for (int i = 0; i < NV; ++i) valid |= (expert(i) < E ? 1u : 0u) << i;

  uint32_t mykey[TPG];
  int myidx[TPG];
#pragma unroll
  for (int t = 0; t < TPG; ++t) {
    mykey[t] = 0u;
    myidx[t] = 0;
  }

#pragma unroll
  for (int t = 0; t < TPG; ++t) {
    bool done = false;
    if (THRESH) {
      // threshold thr: the k-th largest of the 32 lane maxima
      float lmf = -INFINITY;
#pragma unroll
      for (int i = 0; i < NV; ++i) lmf = fmaxf(lmf, x[t][i]);
      uint32_t act = valid ? order_key(lmf) : 0u;
      uint32_t thr = 0u;
#pragma unroll
      for (int r = 0; r < (KT > 0 ? KT : 32); ++r) {
        if (KT == 0 && r >= k) break;
        const uint32_t g = __reduce_max_sync(FULL, act);
        const uint32_t holders = __ballot_sync(FULL, act == g);
        if (lane == __ffs(holders) - 1) act = 0u;
        thr = g;
      }
      const float thr_f = key_value(thr);
      uint32_t cmask = 0u;
      if (thr != 0u) {
#pragma unroll
        for (int i = 0; i < NV; ++i) cmask |= (x[t][i] >= thr_f ? 1u : 0u) << i;
      } else {
        cmask = valid;              // fewer than k lanes hold experts: keep all
      }
      cmask &= valid;
      const int n = __popc(cmask);
      // exclusive prefix of the candidate counts across the warp
      int incl = n;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(FULL, incl, o);
        if (lane >= o) incl += y;
      }
      const int total = __shfl_sync(FULL, incl, 31);
      if (total <= 32) {
        done = true;
        // compact the candidates to one per lane through shared memory
        int pos = incl - n;
#pragma unroll
        for (int i = 0; i < NV; ++i) {
          if (((cmask >> i) & 1u) && RF_IDX_OK(pos, 32)) {
            sm_val[warp][pos] = x[t][i];
            sm_idx[warp][pos] = expert(i);
            ++pos;
          }
        }
        __syncwarp();
        uint32_t ck = 0u;
        int ci = 0x7fffffff;
        if (lane < total) {
          ck = order_key(sm_val[warp][lane]);
          ci = sm_idx[warp][lane];
        }
        __syncwarp();
#pragma unroll
        for (int r = 0; r < (KT > 0 ? KT : 32); ++r) {
          if (KT == 0 && r >= k) break;
          const uint32_t g = __reduce_max_sync(FULL, ck);
          const int gi = (int)__reduce_min_sync(FULL, ck == g ? (uint32_t)ci : 0x7fffffffu);
          if (ck == g && ci == gi) ck = 0u;
          if (lane == r) {
            mykey[t] = g;
            myidx[t] = gi;
          }
        }
      }
    }
    if (!done) {
      // plain rounds over every slot
      uint32_t taken = ~valid;
#pragma unroll
      for (int r = 0; r < (KT > 0 ? KT : 32); ++r) {
        if (KT == 0 && r >= k) break;
        float bv = -INFINITY;
        int bs = -1;
#pragma unroll
        for (int i = 0; i < NV; ++i) {
          // strict > keeps the lowest index among equal values; the first
          // untaken slot is accepted even at -inf
          if (!((taken >> i) & 1u) && (bs < 0 || x[t][i] > bv)) {
            bv = x[t][i];
            bs = i;
          }
        }
        int bi = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < NV; ++i)
          if (i == bs) bi = expert(i);
        const uint32_t bk = bs >= 0 ? order_key(bv) : 0u;
        const uint32_t gk = __reduce_max_sync(gmask, bk);
        const int gi = (int)__reduce_min_sync(gmask, bk == gk ? (uint32_t)bi : 0x7fffffffu);
        if (bs >= 0 && bk == gk && bi == gi) taken |= 1u << bs;
        if (gl == r) {
          mykey[t] = gk;
          myidx[t] = gi;
        }
      }
    }
  }

#pragma unroll
  for (int t = 0; t < TPG; ++t) {
    const int token = tok0 + t;
    // round 0 = row max, held by group lane 0
    const float m = key_value(__shfl_sync(FULL, mykey[t], 0, G));
    // weights exp(x - m); the fast exponential and divide stay far inside the
    // fp32 tolerance (a few ulp)
    const float w = gl < k ? __expf(key_value(mykey[t]) - m) : 0.f;
    float denom;
    if (renorm) {
      denom = gsum<G>(w, k);              // lanes >= k hold 0
    } else {
      float l = 0.f;
#pragma unroll
      for (int i = 0; i < NV; ++i)
        if ((valid >> i) & 1u) l += __expf(x[t][i] - m);
      denom = gsum<G>(l, G);
    }
    if (token < T && gl < k && RF_IDX_OK((size_t)token * k + gl, (long long)T * k)) {
      idx_out[(size_t)token * k + gl] = myidx[t];
      w_out[(size_t)token * k + gl] = __fdividef(w, denom);
    }
  }
}

// Per-lane top-2, then a k-way merge over the group's lanes.
//
// Each lane scans its NV slots once (slot order is expert order, and a strict
// comparison keeps the lower expert first among equal values) and keeps its
// best two as (order key, slot).  Round r of the merge: every lane offers its
// head; the group takes the largest key with one redux.sync and the lowest
// expert among the lanes offering it with a second; the winner pops its head,
// which becomes its second best.  A lane that wins a third time has no
// precomputed successor, so it rescans its untaken slots (a branch only that
// lane takes).  Every round therefore sees each lane's true best untaken
// value, and the result is the exact top-k with ties by lower expert index,
// for any k <= G.
// the group's NV logits of one token (-inf for padding slots and past T)
template <int G, int NV, int W>
__device__ __forceinline__ void load_token(const float* __restrict__ logits, int T, int E, int token,
                                           int gl, float (&x)[NV]) {
  const bool live = token < T;
  const float* row = logits + (size_t)(live ? token : 0) * E;
#pragma unroll
  for (int c = 0; c < NV / W; ++c) {
    const int e0 = c * G * W + gl * W;
    const bool in = live && e0 < E && RF_SPAN_OK(e0, W, E) && RF_IDX_OK(token, T);
    if (W == 4) {
      const float4 f = in ? __ldcs(reinterpret_cast<const float4*>(row + e0))
                          : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
      x[4 * c + 0] = f.x;
      x[4 * c + 1] = f.y;
      x[4 * c + 2] = f.z;
      x[4 * c + 3] = f.w;
    } else {
      x[c] = in ? __ldcs(row + e0) : -INFINITY;
    }
  }
}

template <int G, int NV, int W, int KT>
__device__ __forceinline__ void merge_select(const float (&x)[NV], int token, int T, int k,
                                             int renorm, int gl, uint32_t gmask,
                                             int32_t* __restrict__ idx_out,
                                             float* __restrict__ w_out) {
  auto expert = [&](int i) -> int { return (i / W) * G * W + gl * W + (i % W); };
  // Padding slots (expert >= E) hold -inf and come after every real slot of
  // the lane in slot order, and after every real expert in index order, so
  // they are never chosen while k <= E and add 0 to the softmax sum.
  {
    // the lane's best two slots, compared as floats (-0 == +0, as the keys)
    float v1 = x[0], v2 = -INFINITY;
    int s1 = 0, s2 = -1;
    if (NV > 1) {
      const bool sw = x[1] > x[0];
      v1 = sw ? x[1] : x[0];
      s1 = sw ? 1 : 0;
      v2 = sw ? x[0] : x[1];
      s2 = sw ? 0 : 1;
    }
#pragma unroll
    for (int i = 2; i < NV; ++i) {
      const bool c1 = x[i] > v1, c2 = x[i] > v2;
      v2 = c1 ? v1 : (c2 ? x[i] : v2);
      s2 = c1 ? s1 : (c2 ? i : s2);
      v1 = c1 ? x[i] : v1;
      s1 = c1 ? i : s1;
    }
    uint32_t k1 = order_key(v1), k2 = s2 >= 0 ? order_key(v2) : 0u;
    int e1 = expert(s1), e2 = s2 >= 0 ? expert(s2) : 0x7fffffff;
    uint32_t taken = 0u;
    bool have_next = true;
    uint32_t mykey = 0u;
    int myidx = 0;
#pragma unroll
    for (int r = 0; r < (KT > 0 ? KT : 32); ++r) {
      if (KT == 0 && r >= k) break;
      const uint32_t g = __reduce_max_sync(gmask, k1);
      const int gi = (int)__reduce_min_sync(gmask, k1 == g ? (uint32_t)e1 : 0x7fffffffu);
      if (gl == r) {
        mykey = g;
        myidx = gi;
      }
      if (k1 == g && e1 == gi) {
        taken |= 1u << s1;
        if (have_next) {
          k1 = k2;
          e1 = e2;
          s1 = s2;
          have_next = false;
        } else {
          // third pop of this lane: its best untaken slot
          int b = -1;
          float bv = -INFINITY;
#pragma unroll
          for (int i = 0; i < NV; ++i)
            if (!((taken >> i) & 1u) && (b < 0 || x[i] > bv)) {
              b = i;
              bv = x[i];
            }
          k1 = b >= 0 ? order_key(bv) : 0u;
          e1 = b >= 0 ? expert(b) : 0x7fffffff;
          s1 = b;
        }
      }
    }
    const float m = key_value(__shfl_sync(FULL, mykey, 0, G));
    const float w = gl < k ? __expf(key_value(mykey) - m) : 0.f;
    float denom;
    if (renorm) {
      denom = gsum<G>(w, k);
    } else {
      float l = 0.f;
#pragma unroll
      for (int i = 0; i < NV; ++i) l += __expf(x[i] - m);
      denom = gsum<G>(l, G);
    }
    if (token < T && gl < k && RF_IDX_OK((size_t)token * k + gl, (long long)T * k)) {
      idx_out[(size_t)token * k + gl] = myidx;
      w_out[(size_t)token * k + gl] = __fdividef(w, denom);
    }
  }
}

// Grid-stride over tokens: each group loads the logits of its next token into
// a second register buffer before it selects from the current one, so the
// loads of one token are in flight under the selection work of the previous.
// The loop bound is uniform across the warp (groups past T select from -inf
// and store nothing), so full-warp shuffles stay legal.
template <int G, int NV, int W, int KT>
__global__ void __launch_bounds__(256)
softmax_topk_merge_kernel(const float* __restrict__ logits, int T, int E, int k_rt, int renorm,
                          int32_t* __restrict__ idx_out, float* __restrict__ w_out) {
  static_assert(NV % W == 0 && NV <= 32 && 32 % G == 0, "layout");
  constexpr int GPW = 32 / G;
  const int k = KT > 0 ? KT : k_rt;
  const int lane = threadIdx.x & 31;
  const int gl = lane & (G - 1);
  const uint32_t gmask = G == 32 ? FULL : (((1u << G) - 1u) << (lane & ~(G - 1)));
  const int warp_global = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  const int stride = (int)((gridDim.x * blockDim.x) >> 5) * GPW;
  int base = warp_global * GPW;                      // the warp's first token, uniform
  const int grp = lane / G;
  float xa[NV], xb[NV];
  load_token<G, NV, W>(logits, T, E, base + grp, gl, xa);
  while (base < T) {
    load_token<G, NV, W>(logits, T, E, base + stride + grp, gl, xb);
    merge_select<G, NV, W, KT>(xa, base + grp, T, k, renorm, gl, gmask, idx_out, w_out);
    base += stride;
    if (base >= T) break;
    load_token<G, NV, W>(logits, T, E, base + stride + grp, gl, xa);
    merge_select<G, NV, W, KT>(xb, base + grp, T, k, renorm, gl, gmask, idx_out, w_out);
    base += stride;
  }
}

// One thread per token, for k <= 2 and E a multiple of 32 (up to 128).
//
// A block of TPB threads stages its TPB rows in shared memory with 16-byte
// cp.async copies, coalesced across the block, in two commit groups: the
// first half of every row's chunks, then the second half.  Chunk c of row r
// lands at position c ^ (r & 7) of the row, so when the 32 threads of a warp
// each read the same chunk of their own rows, every 8-thread phase of the
// 16-byte loads touches 8 different bank groups.  Each thread scans its row
// in expert order with NCH independent top-2 chains (chunk c belongs to chain
// c % NCH, so the chains' compares overlap), the first half while the second
// half is still landing, and merges the chains under the same order: larger
// value first, equal values by lower expert index.  Per token this is a few
// dozen thread instructions, about one warp instruction per element of 32
// tokens, against a few hundred warp instructions per token in the warp-wide
// selection.  Measured at [65536 x 64]: the staging alone runs at the read
// floor, and the second commit group hides half of the scan behind the
// stream.  The weights need only the best two: with renormalisation
// w1 = 1 / (1 + e), w2 = e / (1 + e), e = exp(x2 - x1); without it a second
// pass over the staged row sums exp(x - x1).
template <int E, int TPB, int NCH>
__global__ void __launch_bounds__(TPB)
softmax_top2_row_kernel(const float* __restrict__ logits, int T, int k, int renorm,
                        int32_t* __restrict__ idx_out, float* __restrict__ w_out) {
  constexpr int CH = E / 4;                       // 16-byte chunks per row
  // the row arrives in NG commit groups of chunks; the scan of each group
  // runs while the later ones land (four groups: 2 -> 4 cut the time by
  // about 7 % at [65536 x 64])
  constexpr int NG = 4;
  constexpr int GS = CH / NG;
  static_assert(E % 32 == 0 && GS % NCH == 0, "rows of whole 8-chunk swizzle groups");
  __shared__ __align__(16) float4 rows[TPB * CH];
  const int t0 = blockIdx.x * TPB;
  const int nrows = min(TPB, T - t0);
  const float4* src = reinterpret_cast<const float4*>(logits) + (size_t)t0 * CH;
#pragma unroll
  for (int h = 0; h < NG; ++h) {
    for (int q = threadIdx.x; q < nrows * GS; q += TPB) {
      const int r = q / GS, c = h * GS + q % GS;
      if (RF_SPAN_OK(((size_t)t0 * CH + (size_t)r * CH + c) * 4, 4, (long long)T * E)) {
        const uint32_t dst = (uint32_t)__cvta_generic_to_shared(&rows[r * CH + (c ^ (r & 7))]);
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src + r * CH + c)
                     : "memory");
      }
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  }
  asm volatile("cp.async.wait_group %0;" ::"n"(NG - 1) : "memory");
  __syncthreads();
  // threads past the last row stay for the second barrier, then leave
  const int r = threadIdx.x < nrows ? threadIdx.x : nrows - 1;
  const float4* row = rows + r * CH;
  const int sw = r & 7;
  float v1[NCH], v2[NCH];
  int s1[NCH], s2[NCH];
  // strict compares keep the lower expert first among equal values, because
  // each chain visits its experts in increasing order
  auto fold = [&](int p, float x, int i) {
    const bool c1 = x > v1[p], c2 = x > v2[p];
    v2[p] = c1 ? v1[p] : (c2 ? x : v2[p]);
    s2[p] = c1 ? s1[p] : (c2 ? i : s2[p]);
    v1[p] = c1 ? x : v1[p];
    s1[p] = c1 ? i : s1[p];
  };
  // chain p starts from chunk p: its first two values in order, then the rest
#pragma unroll
  for (int p = 0; p < NCH; ++p) {
    const float4 f = row[p ^ sw];
    const int b = 4 * p;
    const bool up = f.y > f.x;
    v1[p] = up ? f.y : f.x;
    s1[p] = up ? b + 1 : b;
    v2[p] = up ? f.x : f.y;
    s2[p] = up ? b : b + 1;
    fold(p, f.z, b + 2);
    fold(p, f.w, b + 3);
  }
#pragma unroll
  for (int j = 1; j < CH / NCH; ++j) {
    if (j % (GS / NCH) == 0) {
      // group j / (GS / NCH) has landed once no more than NG - 1 - j / (GS / NCH)
      // groups are pending
      const int pending = NG - 1 - j / (GS / NCH);
      if (pending == 2) asm volatile("cp.async.wait_group 2;" ::: "memory");
      if (pending == 1) asm volatile("cp.async.wait_group 1;" ::: "memory");
      if (pending == 0) asm volatile("cp.async.wait_group 0;" ::: "memory");
      __syncthreads();
    }
#pragma unroll
    for (int p = 0; p < NCH; ++p) {
      const int c = NCH * j + p;
      const float4 f = row[c ^ sw];
      fold(p, f.x, 4 * c);
      fold(p, f.y, 4 * c + 1);
      fold(p, f.z, 4 * c + 2);
      fold(p, f.w, 4 * c + 3);
    }
  }
  if (threadIdx.x >= nrows) return;
  // merge the chains: (a, ia) ranks above (b, ib) if a > b, or a == b and ia < ib
  auto above = [](float a, int ia, float b, int ib) { return a > b || (a == b && ia < ib); };
  float x1 = v1[0], x2 = v2[0];
  int i1 = s1[0], i2 = s2[0];
#pragma unroll
  for (int p = 1; p < NCH; ++p) {
    const bool c = above(v1[p], s1[p], x1, i1);
    const float a = c ? x1 : x2, b = c ? v2[p] : v1[p];
    const int ia = c ? i1 : i2, ib = c ? s2[p] : s1[p];
    const bool d = above(b, ib, a, ia);
    x1 = c ? v1[p] : x1;
    i1 = c ? s1[p] : i1;
    x2 = d ? b : a;
    i2 = d ? ib : ia;
  }
  const float e2 = __expf(x2 - x1);             // weight of the second, relative to the first
  float denom;
  if (renorm) {
    denom = k == 2 ? 1.f + e2 : 1.f;
  } else {
    float l = 0.f;
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      const float4 f = row[c ^ sw];
      l += __expf(f.x - x1) + __expf(f.y - x1) + __expf(f.z - x1) + __expf(f.w - x1);
    }
    denom = l;
  }
  const size_t token = (size_t)(t0 + r);
  if (k == 2) {
    if (RF_SPAN_OK(token * 2, 2, (long long)T * 2)) {
      reinterpret_cast<int2*>(idx_out)[token] = make_int2(i1, i2);
      reinterpret_cast<float2*>(w_out)[token] =
          make_float2(__fdividef(1.f, denom), __fdividef(e2, denom));
    }
  } else if (RF_IDX_OK(token, T)) {
    idx_out[token] = i1;
    w_out[token] = __fdividef(1.f, denom);
  }
}

// Two threads per token, for E = 256 and k <= 8.
//
// A block of 32 threads stages its 16 rows (1 KiB each) with 16-byte cp.async
// copies.  Thread h of a token's pair owns experts [128 h, 128 h + 128), the
// 16-byte chunks [32 h, 32 h + 32) of the row; chunk C of row t lands at
// position C ^ (2 (t & 3) + C / 32), so the 8-thread phases of the 16-byte
// loads (four tokens x two halves reading the same chunk offset) hit 8
// different bank groups.  The copies go out in eight commit groups by
// column, group g holding chunks 32 h + 4 g .. 32 h + 4 g + 3 of every row
// (the thread's value group g, below), and each thread takes the maximum of
// group g as soon as that commit group has landed, while the later ones are
// still in flight ([16384 x 256] top-8: 7.47 -> 7.33 us in a CUDA graph over
// copies larger than L2; 9.95 -> 8.89 us in a loop of plain launches).  Per
// token:
//   * each thread takes the maxima of its 8 groups of 16 values and sorts
//     them; the 8 largest of the pair's 16 are max(mine[i], partner[7-i])
//     (one shuffle each), and thr, the smallest of those, has at least 8
//     distinct values at or above it: the top 8 all lie at or above thr;
//   * each thread marks its values >= thr (about six on random logits) and
//     inserts them, in expert order, into a sorted top-8 of its half
//     (strict compares: an equal value from a later expert goes after);
//   * the two halves' lists merge bitonically: max(a[i], b[7-i]) under
//     (larger value, lower expert), then three compare-exchange stages;
//     both threads hold the result, and thread h stores entries 4h .. 4h + 3.
// The top k <= 8 are the first k entries.  Measured against the one-warp
// selection at [16384 x 256] top-8: 7.05 vs 8.37 us (probe, same inputs).
// A token with thr = -inf (8 or more experts at -inf) takes the insertion
// that also fills empty slots with -inf values.
__device__ __forceinline__ bool ranks_before(float av, int ai, float bv, int bi) {
  return av > bv || (av == bv && ai < bi);
}

template <bool RENORM, int KT>      // KT = k when known at compile time (0: runtime)
__global__ void __launch_bounds__(32)
softmax_top8_pair_kernel(const float* __restrict__ logits, int T, int k_rt,
                         int32_t* __restrict__ idx_out, float* __restrict__ w_out) {
  const int k = KT > 0 ? KT : k_rt;
  constexpr int E = 256, CH = 64, TOK = 16, KK = 8;
  constexpr int EMPTY = 0x7fffffff;
  __shared__ __align__(16) float4 rows[TOK * CH];
  const int t0 = blockIdx.x * TOK;
  const int nrows = min(TOK, T - t0);
  const float4* src = reinterpret_cast<const float4*>(logits) + (size_t)t0 * CH;
#pragma unroll
  for (int kq = 0; kq < 8; ++kq) {     // commit group kq: chunks 4 kq .. 4 kq + 3 of each half
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int q2 = threadIdx.x + 32 * i;
      const int t = q2 >> 3, lc = q2 & 7;
      const int c = ((lc >> 2) << 5) + 4 * kq + (lc & 3);
      if (t < nrows && RF_SPAN_OK(((size_t)t0 * CH + t * CH + c) * 4, 4, (long long)T * E)) {
        const int f = ((t & 3) << 1) | (c >> 5);
        const uint32_t dst = (uint32_t)__cvta_generic_to_shared(&rows[t * CH + (c ^ f)]);
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src + t * CH + c)
                     : "memory");
      }
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  }
  // pairs past the last row work on the last row (the shuffles need every
  // lane) and store nothing
  const int tl = min(threadIdx.x >> 1, nrows - 1), h = threadIdx.x & 1;
  const int f = ((tl & 3) << 1) | h;
  const float4* row = rows + tl * CH;
  const float* rowf = reinterpret_cast<const float*>(row);
  // maxima of the thread's 8 groups of 16 values, sorted descending
  float sm[8];
#pragma unroll
  for (int kq = 0; kq < 8; ++kq) {
    if (kq == 0) asm volatile("cp.async.wait_group 7;" ::: "memory");
    if (kq == 1) asm volatile("cp.async.wait_group 6;" ::: "memory");
    if (kq == 2) asm volatile("cp.async.wait_group 5;" ::: "memory");
    if (kq == 3) asm volatile("cp.async.wait_group 4;" ::: "memory");
    if (kq == 4) asm volatile("cp.async.wait_group 3;" ::: "memory");
    if (kq == 5) asm volatile("cp.async.wait_group 2;" ::: "memory");
    if (kq == 6) asm volatile("cp.async.wait_group 1;" ::: "memory");
    if (kq == 7) asm volatile("cp.async.wait_group 0;" ::: "memory");
    __syncwarp();     // the block is one warp: the other lanes' copies are visible
    float m = -INFINITY;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float4 v = row[(32 * h + 4 * kq + j) ^ f];
      m = max3f(m, max3f(v.x, v.y, v.z), v.w);
    }
    sm[kq] = m;
  }
  auto cs = [](float& a, float& b) {
    const float hi = fmaxf(a, b), lo = fminf(a, b);
    a = hi;
    b = lo;
  };
  cs(sm[0], sm[1]); cs(sm[2], sm[3]); cs(sm[4], sm[5]); cs(sm[6], sm[7]);
  cs(sm[0], sm[2]); cs(sm[1], sm[3]); cs(sm[4], sm[6]); cs(sm[5], sm[7]);
  cs(sm[1], sm[2]); cs(sm[5], sm[6]); cs(sm[0], sm[4]); cs(sm[3], sm[7]);
  cs(sm[1], sm[5]); cs(sm[2], sm[6]);
  cs(sm[1], sm[4]); cs(sm[3], sm[6]);
  cs(sm[2], sm[4]); cs(sm[3], sm[5]);
  cs(sm[3], sm[4]);
  float thr = INFINITY;
#pragma unroll
  for (int i = 0; i < 8; ++i) thr = fminf(thr, fmaxf(sm[i], __shfl_xor_sync(FULL, sm[7 - i], 1)));
  const float rmax = fmaxf(sm[0], __shfl_xor_sync(FULL, sm[0], 1));
  // candidates: values >= thr, one bit per value in expert order
  uint32_t cm[4] = {0u, 0u, 0u, 0u};
#pragma unroll
  for (int c = 0; c < 32; ++c) {
    const float4 v = row[(32 * h + c) ^ f];
    const uint32_t b = (v.x >= thr ? 1u : 0u) | (v.y >= thr ? 2u : 0u) |
                       (v.z >= thr ? 4u : 0u) | (v.w >= thr ? 8u : 0u);
    cm[c >> 3] |= b << (4 * (c & 7));
  }
  float tv[KK];
  int ti[KK];
#pragma unroll
  for (int i = 0; i < KK; ++i) {
    tv[i] = -INFINITY;
    ti[i] = EMPTY;
  }
  auto insert = [&](float x, int e, bool any_empty) {
    bool c[KK];
#pragma unroll
    for (int i = 0; i < KK; ++i) c[i] = x > tv[i] || (any_empty && ti[i] == EMPTY);
#pragma unroll
    for (int i = KK - 1; i > 0; --i) {
      tv[i] = c[i] ? (c[i - 1] ? tv[i - 1] : x) : tv[i];
      ti[i] = c[i] ? (c[i - 1] ? ti[i - 1] : e) : ti[i];
    }
    tv[0] = c[0] ? x : tv[0];
    ti[0] = c[0] ? e : ti[0];
  };
  auto insert_all = [&](bool any_empty) {
#pragma unroll
    for (int wv = 0; wv < 4; ++wv) {
      uint32_t m = cm[wv];
      while (m) {
        const int b = __ffs(m) - 1;
        m &= m - 1;
        const int pos = 32 * wv + b;                     // 0..127 within the half
        insert(rowf[4 * ((32 * h + (pos >> 2)) ^ f) + (pos & 3)], 128 * h + pos, any_empty);
      }
    }
  };
  // with a finite thr every candidate beats the -inf of an empty slot
  if (__all_sync(FULL, thr > -INFINITY))
    insert_all(false);
  else
    insert_all(true);
  // merge the halves: the 8 best of the 16 as a bitonic sequence, then sort
  float mv[KK];
  int mi[KK];
#pragma unroll
  for (int i = 0; i < KK; ++i) {
    const float ov = __shfl_xor_sync(FULL, tv[KK - 1 - i], 1);
    const int oi = __shfl_xor_sync(FULL, ti[KK - 1 - i], 1);
    const bool mine = ranks_before(tv[i], ti[i], ov, oi);
    mv[i] = mine ? tv[i] : ov;
    mi[i] = mine ? ti[i] : oi;
  }
  auto cas = [&](int a, int b) {
    const bool keep = ranks_before(mv[a], mi[a], mv[b], mi[b]);
    const float va = keep ? mv[a] : mv[b], vb = keep ? mv[b] : mv[a];
    const int ia = keep ? mi[a] : mi[b], ib = keep ? mi[b] : mi[a];
    mv[a] = va;
    mv[b] = vb;
    mi[a] = ia;
    mi[b] = ib;
  };
  cas(0, 4); cas(1, 5); cas(2, 6); cas(3, 7);
  cas(0, 2); cas(1, 3); cas(4, 6); cas(5, 7);
  cas(0, 1); cas(2, 3); cas(4, 5); cas(6, 7);
  // weights exp(x - m) over the selected (renormalised) or over the row
  float ex[KK], sel = 0.f;
#pragma unroll
  for (int i = 0; i < KK; ++i) {
    ex[i] = i < k ? __expf(mv[i] - rmax) : 0.f;
    sel += ex[i];
  }
  float denom = sel;
  if (!RENORM) {
    float l = 0.f;
#pragma unroll
    for (int c = 0; c < 32; ++c) {
      const float4 v = row[(32 * h + c) ^ f];
      l += __expf(v.x - rmax) + __expf(v.y - rmax) + __expf(v.z - rmax) + __expf(v.w - rmax);
    }
    denom = l + __shfl_xor_sync(FULL, l, 1);
  }
  const float inv = __fdividef(1.f, denom);
  if ((int)(threadIdx.x >> 1) < nrows) {
    const size_t token = (size_t)(t0 + tl);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int j = 4 * h + i;
      const int id = h ? mi[4 + i] : mi[i];
      const float wj = (h ? ex[4 + i] : ex[i]) * inv;
      if (j < k && RF_IDX_OK(token * k + j, (long long)T * k)) {
        idx_out[token * k + j] = id;
        w_out[token * k + j] = wj;
      }
    }
  }
}

template <int E>
void launch_top2_rows(const float* logits, int T, int k, int renorm, int32_t* idx, float* w,
                      cudaStream_t st) {
  constexpr int TPB = 64;      // measured at E = 64: 64 and 128 alike, 32 slower
  const unsigned grid = (unsigned)((T + TPB - 1) / TPB);
  softmax_top2_row_kernel<E, TPB, 2><<<grid, TPB, 0, st>>>(logits, T, k, renorm, idx, w);
}

constexpr int kMergeBlocksPerSm = 8;     // measured best of 2, 4, 8, 16 at [65536 x 64]

template <int G, int NV, int W>
void launch_merge(const float* logits, int T, int E, int k, int renorm, int32_t* idx, float* w,
                  cudaStream_t st) {
  constexpr int tokens_per_block = 256 / G;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long long need = (T + tokens_per_block - 1) / tokens_per_block;
  const long long cap = (long long)(sms > 0 ? sms : 1) * kMergeBlocksPerSm;
  const unsigned grid = (unsigned)(need < cap ? need : cap);
  if (k == 8)
    softmax_topk_merge_kernel<G, NV, W, 8><<<grid, 256, 0, st>>>(logits, T, E, k, renorm, idx, w);
  else if (k == 2)
    softmax_topk_merge_kernel<G, NV, W, 2><<<grid, 256, 0, st>>>(logits, T, E, k, renorm, idx, w);
  else
    softmax_topk_merge_kernel<G, NV, W, 0><<<grid, 256, 0, st>>>(logits, T, E, k, renorm, idx, w);
}

template <int G, int NV, int W, int TPG, bool THRESH>
void launch_one(const float* logits, int T, int E, int k, int renorm, int32_t* idx, float* w,
                cudaStream_t st) {
  constexpr int tokens_per_block = 256 / G * TPG;
  const unsigned grid = (unsigned)((T + tokens_per_block - 1) / tokens_per_block);
  if (k == 8)
    softmax_topk_kernel<G, NV, W, TPG, 8, THRESH><<<grid, 256, 0, st>>>(logits, T, E, k, renorm, idx, w);
  else if (k == 2)
    softmax_topk_kernel<G, NV, W, TPG, 2, THRESH><<<grid, 256, 0, st>>>(logits, T, E, k, renorm, idx, w);
  else
    softmax_topk_kernel<G, NV, W, TPG, 0, THRESH><<<grid, 256, 0, st>>>(logits, T, E, k, renorm, idx, w);
}

}  // namespace

rf_status launch_softmax_topk(const float* logits, int T, int E, int k, int renormalize,
                              int32_t* idx, float* w, cudaStream_t st) {
  const bool v4 = E % 4 == 0;
  if (k <= 2 && E % 32 == 0 && E <= 128) {
    switch (E) {
      case 32: launch_top2_rows<32>(logits, T, k, renormalize, idx, w, st); break;
      case 64: launch_top2_rows<64>(logits, T, k, renormalize, idx, w, st); break;
      case 96: launch_top2_rows<96>(logits, T, k, renormalize, idx, w, st); break;
      default: launch_top2_rows<128>(logits, T, k, renormalize, idx, w, st); break;
    }
    return launch_status();
  }
  if (E == 256 && k <= 8) {
    const unsigned grid = (unsigned)((T + 15) / 16);
    if (renormalize && k == 8)
      softmax_top8_pair_kernel<true, 8><<<grid, 32, 0, st>>>(logits, T, k, idx, w);
    else if (renormalize)
      softmax_top8_pair_kernel<true, 0><<<grid, 32, 0, st>>>(logits, T, k, idx, w);
    else
      softmax_top8_pair_kernel<false, 0><<<grid, 32, 0, st>>>(logits, T, k, idx, w);
    return launch_status();
  }
  // lanes r < k of a group keep round r's winner, so G >= k
  if (E <= 64 && k <= 4) {
    if (v4) launch_merge<4, 16, 4>(logits, T, E, k, renormalize, idx, w, st);
    else launch_merge<4, 16, 1>(logits, T, E, k, renormalize, idx, w, st);
  } else if (E <= 64 && k <= 8) {
    if (v4) launch_merge<8, 8, 4>(logits, T, E, k, renormalize, idx, w, st);
    else launch_merge<8, 8, 1>(logits, T, E, k, renormalize, idx, w, st);
  } else if (E <= 128 && k <= 16) {
    if (v4) launch_merge<16, 8, 4>(logits, T, E, k, renormalize, idx, w, st);
    else launch_merge<16, 8, 1>(logits, T, E, k, renormalize, idx, w, st);
  } else if (E <= 128) {
    if (v4) launch_one<32, 4, 4, 2, false>(logits, T, E, k, renormalize, idx, w, st);
    else launch_one<32, 4, 1, 2, false>(logits, T, E, k, renormalize, idx, w, st);
  } else if (E <= 256) {
    if (v4) launch_one<32, 8, 4, 1, true>(logits, T, E, k, renormalize, idx, w, st);
    else launch_one<32, 8, 1, 1, true>(logits, T, E, k, renormalize, idx, w, st);
  } else if (E <= 512) {
    if (v4) launch_one<32, 16, 4, 1, true>(logits, T, E, k, renormalize, idx, w, st);
    else launch_one<32, 16, 1, 1, true>(logits, T, E, k, renormalize, idx, w, st);
  } else if (E <= 1024) {
    if (v4) launch_one<32, 32, 4, 1, true>(logits, T, E, k, renormalize, idx, w, st);
    else launch_one<32, 32, 1, 1, true>(logits, T, E, k, renormalize, idx, w, st);
  } else {
    return RF_ERR_UNSUPPORTED;
  }
  return launch_status();
}

RF_BOUNDS_WORD_OF_THIS_FILE

}  // namespace rf
