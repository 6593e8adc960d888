// MoE routing: softmax over experts, then top-k, from one read of each row.
//
// The cascade (RedFuser episode transcript, cue 11; "Online normalizer
// calculation for softmax", abstract on its citation page): the row max, the
// exp-sum denominator and the k largest entries all come from a single pass
// over the logits held in registers.
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
      const bool in = live && e0 < E;
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
          if ((cmask >> i) & 1u) {
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
    if (token < T && gl < k) {
      idx_out[(size_t)token * k + gl] = myidx[t];
      w_out[(size_t)token * k + gl] = __fdividef(w, denom);
    }
  }
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
  // lanes r < k of a group keep round r's winner, so G >= k
  if (E <= 64 && k <= 8) {
    if (v4) launch_one<8, 8, 4, 2, false>(logits, T, E, k, renormalize, idx, w, st);
    else launch_one<8, 8, 1, 2, false>(logits, T, E, k, renormalize, idx, w, st);
  } else if (E <= 128 && k <= 16) {
    if (v4) launch_one<16, 8, 4, 1, false>(logits, T, E, k, renormalize, idx, w, st);
    else launch_one<16, 8, 1, 1, false>(logits, T, E, k, renormalize, idx, w, st);
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

}  // namespace rf
