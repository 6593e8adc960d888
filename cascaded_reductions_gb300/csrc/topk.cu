// MoE routing: softmax over experts, then top-k, from one read of each row.
//
// The cascade (RedFuser episode transcript, cue 11; "Online normalizer
// calculation for softmax", abstract on its citation page): the row max, the
// exp-sum denominator and the k largest entries all come from a single pass
// over the logits held in registers.
//
// Layout: a group of G lanes (G = 32, or 16 for E <= 64 and k <= 16) owns one
// token; each lane holds NV 16-byte chunks of the row (4*NV logits), loaded
// with coalesced 16-byte loads (or scalar loads when E % 4 != 0).  Padding
// slots hold -inf and never win.
//   1. group max m and sum l = sum exp(x - m) (xor shuffles);
//   2. k rounds of group arg-max on the raw fp32 logits: each lane proposes
//      its best untaken slot (larger value, then lower expert index), the
//      group reduces (value, index) pairs, the owner marks the winner taken,
//      and lane r of the group keeps round r's winner;
//   3. lanes r < k turn their winner into a weight exp(x - m) / l, or
//      exp(x - m) / sum over the selected (renormalised), and store the
//      k indices and weights with one coalesced store each.
// Ordering by the raw logits (not by rounded exponentials, which can tie)
// makes equal probabilities come out in index order exactly when their
// logits are equal.

#include <math.h>

#include "common.cuh"

namespace rf {
namespace {

__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}

template <int G, int NV, bool VEC>
__global__ void __launch_bounds__(256)
softmax_topk_kernel(const float* __restrict__ logits, int T, int E, int k, int renorm,
                    int32_t* __restrict__ idx_out, float* __restrict__ w_out) {
  constexpr int NVAL = 4 * NV;   // values per lane
  static_assert(NVAL <= 32, "taken mask is 32 bits");
  const int lane = threadIdx.x & 31;
  const int j = lane & (G - 1);                 // lane within the group
  const int token = (blockIdx.x * 256 + threadIdx.x) / G;
  // All lanes of a warp take part in the shuffles; groups past the end run
  // with all slots at -inf and store nothing.
  const bool live = token < T;
  const float* row = logits + (size_t)(live ? token : 0) * E;

  float x[NVAL];
#pragma unroll
  for (int v = 0; v < NV; ++v) {
    if (VEC) {
      const int e0 = (v * G + j) * 4;
      if (live && e0 < E) {
        const float4 f = __ldcs(reinterpret_cast<const float4*>(row + e0));
        x[4 * v + 0] = f.x; x[4 * v + 1] = f.y; x[4 * v + 2] = f.z; x[4 * v + 3] = f.w;
      } else {
        x[4 * v + 0] = x[4 * v + 1] = x[4 * v + 2] = x[4 * v + 3] = -INFINITY;
      }
    } else {
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const int e = (4 * v + t) * G + j;
        x[4 * v + t] = (live && e < E) ? __ldcs(row + e) : -INFINITY;
      }
    }
  }
  // expert index of slot i of this lane
  auto slot_index = [&](int i) -> int {
    return VEC ? ((i >> 2) * G + j) * 4 + (i & 3) : i * G + j;
  };

  // reduction 1: max; reduction 2: sum of exp(x - m)
  float m = -INFINITY;
#pragma unroll
  for (int i = 0; i < NVAL; ++i) m = fmaxf(m, x[i]);
  m = group_max<G>(m);
  const float mref = m == -INFINITY ? 0.f : m;
  float l = 0.f;
#pragma unroll
  for (int i = 0; i < NVAL; ++i) l += expf(x[i] - mref);
  l = group_sum<G>(l);

  // top-k rounds
  uint32_t taken = 0;
  float my_val = -INFINITY;
  int my_idx = 0x7fffffff;
  for (int r = 0; r < k; ++r) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    int bslot = -1;
#pragma unroll
    for (int i = 0; i < NVAL; ++i) {
      const int e = slot_index(i);
      if (!((taken >> i) & 1u) && e < E && better(x[i], e, bv, bi)) {
        bv = x[i];
        bi = e;
        bslot = i;
      }
    }
    float gv = bv;
    int gi = bi;
#pragma unroll
    for (int o = G / 2; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, gv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, gi, o);
      if (better(ov, oi, gv, gi)) {
        gv = ov;
        gi = oi;
      }
    }
    if (bslot >= 0 && bi == gi) taken |= 1u << bslot;
    if (j == r) {
      my_val = gv;
      my_idx = gi;
    }
  }

  float w = (j < k) ? expf(my_val - mref) : 0.f;
  float denom = l;
  if (renorm) denom = group_sum<G>(w);
  if (live && j < k) {
    idx_out[(size_t)token * k + j] = my_idx;
    w_out[(size_t)token * k + j] = w / denom;
  }
}

template <int G, int NV>
void launch_one(const float* logits, int T, int E, int k, int renorm, int32_t* idx, float* w,
                cudaStream_t st) {
  const int tokens_per_block = 256 / G;
  const unsigned grid = (unsigned)((T + tokens_per_block - 1) / tokens_per_block);
  if (E % 4 == 0)
    softmax_topk_kernel<G, NV, true><<<grid, 256, 0, st>>>(logits, T, E, k, renorm, idx, w);
  else
    softmax_topk_kernel<G, NV, false><<<grid, 256, 0, st>>>(logits, T, E, k, renorm, idx, w);
}

}  // namespace

rf_status launch_softmax_topk(const float* logits, int T, int E, int k, int renormalize,
                              int32_t* idx, float* w, cudaStream_t st) {
  // lanes r < k hold round r's winner, so a group needs at least k lanes
  if (E <= 64 && k <= 16) {
    launch_one<16, 1>(logits, T, E, k, renormalize, idx, w, st);
  } else if (E <= 128) {
    launch_one<32, 1>(logits, T, E, k, renormalize, idx, w, st);
  } else if (E <= 256) {
    launch_one<32, 2>(logits, T, E, k, renormalize, idx, w, st);
  } else if (E <= 512) {
    launch_one<32, 4>(logits, T, E, k, renormalize, idx, w, st);
  } else if (E <= 1024) {
    launch_one<32, 8>(logits, T, E, k, renormalize, idx, w, st);
  } else {
    return RF_ERR_UNSUPPORTED;
  }
  return launch_status();
}

}  // namespace rf
