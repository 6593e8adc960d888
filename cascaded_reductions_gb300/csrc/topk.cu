// MoE routing: softmax over experts, then top-k, from one read of each row.
//
// The cascade (RedFuser episode transcript, cue 11; "Online normalizer
// calculation for softmax", abstract on its citation page): the row max, the
// exp-sum denominator and the k largest entries all come from a single pass
// over the logits held in registers.
//
// Layout: one warp owns TPW tokens; lane j holds NV logits of each token,
// loaded W at a time (W = 4, 2 or 1 consecutive floats, coalesced across the
// warp).  Values that enter a warp reduction are turned into
// order-preserving 32-bit keys (-0 is first mapped to +0, so keys compare
// exactly like the float values).
//   * threshold: T = the k-th largest of the 32 lane maxima (found with k
//     rounds of redux.sync max + ballot).  The k lanes supplying those maxima
//     hold k distinct elements >= T, so the top k all lie at or above T;
//   * the candidates >= T (typically a dozen) are compacted through shared
//     memory to one per lane; round r of top-k then takes the maximum key
//     with one redux.sync and the minimum expert index among the lanes
//     holding it with a second, and lane r keeps the winner.  Equal logits
//     therefore come out in index order.  With fewer than 4 slots per lane,
//     or if more than 32 candidates survive (many ties), the rounds scan every
//     lane's slots instead (same result);
//   * the row max m is round 0's key; with renormalisation the weights are
//     exp(x_i - m) / sum over the k selected, otherwise exp(x_i - m) / l with
//     l = sum over all E of exp(x - m);
//   * lanes r < k store index and weight with one coalesced store each.
// The TPW tokens of a warp are processed side by side so their loads and
// reduction chains overlap.

#include <math.h>

#include "common.cuh"

#ifndef RF_TOPK_TPW256
#define RF_TOPK_TPW256 1
#endif

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

// NV logits per lane (E <= 32*NV), W consecutive logits per load, TPW tokens
// per warp, KT = k when k is known at compile time (0: runtime k).  Logits
// stay floats; integer keys are formed only for the values that enter a
// redux.sync.  Padding slots (expert index >= E) never take part.
template <int NV, int W, int TPW, int KT>
__global__ void __launch_bounds__(256)
softmax_topk_kernel(const float* __restrict__ logits, int T, int E, int k_rt, int renorm,
                    int32_t* __restrict__ idx_out, float* __restrict__ w_out) {
  static_assert(NV % W == 0 && NV <= 32, "layout");
  const int k = KT > 0 ? KT : k_rt;
  const int lane = threadIdx.x & 31;
  const int warp_id = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int warp = threadIdx.x >> 5;
  const int tok0 = warp_id * TPW;
  __shared__ float sm_val[8][32];
  __shared__ int sm_idx[8][32];

  // expert index of slot i of this lane
  auto expert = [&](int i) -> int { return (i / W) * 32 * W + lane * W + (i % W); };

  float x[TPW][NV];
#pragma unroll
  for (int t = 0; t < TPW; ++t) {
    const int token = tok0 + t;
    const bool live = token < T;
    const float* row = logits + (size_t)(live ? token : 0) * E;
#pragma unroll
    for (int c = 0; c < NV / W; ++c) {
      const int e0 = c * 32 * W + lane * W;
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
  // slots that hold a real expert (the same for every token of the warp)
  uint32_t valid = 0u;
#pragma unroll
  for (int i = 0; i < NV; ++i) valid |= (expert(i) < E ? 1u : 0u) << i;

  uint32_t mykey[TPW];
  int myidx[TPW];
#pragma unroll
  for (int t = 0; t < TPW; ++t) {
    mykey[t] = 0u;
    myidx[t] = 0;
  }

#pragma unroll
  for (int t = 0; t < TPW; ++t) {
    bool fast = false;
    if (NV >= 4) {
      // Threshold thr: the k-th largest of the 32 lane maxima.  The k lanes
      // supplying those maxima hold k distinct elements >= thr, so every
      // element of the top k is >= thr; everything below it is discarded.
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
        fast = true;
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
    if (!fast) {
      // few slots per lane, or many equal values: rounds scan every slot
      uint32_t taken = ~valid;
      for (int r = 0; r < k; ++r) {
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
        const uint32_t gk = __reduce_max_sync(FULL, bk);
        const int gi = (int)__reduce_min_sync(FULL, bk == gk ? (uint32_t)bi : 0x7fffffffu);
        if (bs >= 0 && bk == gk && bi == gi) taken |= 1u << bs;
        if (lane == r) {
          mykey[t] = gk;
          myidx[t] = gi;
        }
      }
    }
  }

#pragma unroll
  for (int t = 0; t < TPW; ++t) {
    const int token = tok0 + t;
    const float m = key_value(__shfl_sync(FULL, mykey[t], 0));   // round 0 = row max
    // weights exp(x - m); the fast exponential and divide stay far inside the
    // fp32 tolerance (a few ulp)
    const float w = lane < k ? __expf(key_value(mykey[t]) - m) : 0.f;
    float denom;
    if (renorm) {
      // lanes >= k hold 0: summing over the smallest power-of-two group that
      // covers lanes 0..k-1 is enough
      denom = w;
      if (KT > 0) {
#pragma unroll
        for (int o = 1; o < KT; o <<= 1) denom += __shfl_xor_sync(FULL, denom, o);
      } else {
        denom = group_sum<32>(w);
      }
    } else {
      float l = 0.f;
#pragma unroll
      for (int i = 0; i < NV; ++i)
        if ((valid >> i) & 1u) l += __expf(x[t][i] - m);
      denom = group_sum<32>(l);
    }
    if (token < T && lane < k) {
      idx_out[(size_t)token * k + lane] = myidx[t];
      w_out[(size_t)token * k + lane] = __fdividef(w, denom);
    }
  }
}

template <int NV, int W, int TPW>
void launch_one(const float* logits, int T, int E, int k, int renorm, int32_t* idx, float* w,
                cudaStream_t st) {
  const int warps = (T + TPW - 1) / TPW;
  const unsigned grid = (unsigned)((warps + 7) / 8);
  if (k == 8)
    softmax_topk_kernel<NV, W, TPW, 8><<<grid, 256, 0, st>>>(logits, T, E, k, renorm, idx, w);
  else if (k == 2)
    softmax_topk_kernel<NV, W, TPW, 2><<<grid, 256, 0, st>>>(logits, T, E, k, renorm, idx, w);
  else
    softmax_topk_kernel<NV, W, TPW, 0><<<grid, 256, 0, st>>>(logits, T, E, k, renorm, idx, w);
}

}  // namespace

rf_status launch_softmax_topk(const float* logits, int T, int E, int k, int renormalize,
                              int32_t* idx, float* w, cudaStream_t st) {
  const bool v4 = E % 4 == 0, v2 = E % 2 == 0;
  if (E <= 32) {
    launch_one<1, 1, 4>(logits, T, E, k, renormalize, idx, w, st);
  } else if (E <= 64) {
    if (v2) launch_one<2, 2, 8>(logits, T, E, k, renormalize, idx, w, st);
    else launch_one<2, 1, 8>(logits, T, E, k, renormalize, idx, w, st);
  } else if (E <= 128) {
    if (v4) launch_one<4, 4, 2>(logits, T, E, k, renormalize, idx, w, st);
    else launch_one<4, 1, 2>(logits, T, E, k, renormalize, idx, w, st);
  } else if (E <= 256) {
    if (v4) launch_one<8, 4, RF_TOPK_TPW256>(logits, T, E, k, renormalize, idx, w, st);
    else launch_one<8, 1, 2>(logits, T, E, k, renormalize, idx, w, st);
  } else if (E <= 512) {
    if (v4) launch_one<16, 4, 1>(logits, T, E, k, renormalize, idx, w, st);
    else launch_one<16, 1, 1>(logits, T, E, k, renormalize, idx, w, st);
  } else if (E <= 1024) {
    if (v4) launch_one<32, 4, 1>(logits, T, E, k, renormalize, idx, w, st);
    else launch_one<32, 1, 1>(logits, T, E, k, renormalize, idx, w, st);
  } else {
    return RF_ERR_UNSUPPORTED;
  }
  return launch_status();
}

}  // namespace rf
