// Split-KV decode attention: segment-state producer and state merge.
//
// The cascade (RedFuser episode transcript, cue 9): scores s_j = scale<q,k_j>,
// then max, then sum exp(s_j - m), then sum exp(s_j - m) v_j, then divide.
// The fused form (transcript cues 15-19 and 31) streams K and V once and
// keeps (m, l, acc) per row, rescaling by exp(m_old - m_new) whenever the max
// grows; segments of the key axis are processed by different CTAs and their
// states merged afterwards (cue 21 and cue 39, Multi-Segment).
//
// Kernel layout (both dtypes store a key row in 256 bytes: 64 fp32 or 128
// bf16):
//   * one CTA per (row, segment); its warps take turns over tiles of
//     2*U consecutive keys; a 16-byte load instruction of a warp covers two
//     whole key rows (512 contiguous bytes), lane half h = lane/16 takes key
//     2u+h of the tile and lane c = lane%16 the c-th 16-byte chunk of it;
//   * K and V of a tile are loaded together (2*U 16-byte streaming loads per
//     lane in flight; U = 8, or 4 for short segments on large grids, where
//     more CTAs per SM matter more), the partial dot products are summed across the 16
//     lanes of a half with xor shuffles, so every lane of the half holds all
//     U scores of its keys;
//   * each half-warp keeps its own running state in the log2 domain
//     (scores pre-multiplied by scale*log2(e), exp2 instead of exp); lane c
//     owns acc for its chunk of D;
//   * at the end the two halves, then the CTA's warps (through shared
//     memory) merge their states with the same rescaling, and the CTA writes
//     the segment's (m, l, acc), m converted back to natural-log units.

#include <math.h>

#include <cuda_bf16.h>

#include "common.cuh"

namespace rf {
namespace {

// The fused form of the merge (FUSED): the CTA that finishes a row's last
// segment merges that row's S states and writes out and lse.  Each CTA
// publishes its state, fences, and counts itself in counters[row]; the CTA
// that brings the count to S is the last, reads every state of the row
// (written by the others before their own fence and count), merges them with
// the same rescale as state_merge_kernel, and sets the counter back to 0 for
// the next call.  No CTA waits for another.
struct FusedMerge {
  int* counters;       // [R], zero before the call, zero after it
  void* out;           // [R, D], fp32 or bf16
  float* lse;          // [R] or null
  int out_bf16;
};

template <typename T, int WARPS, int U, bool FUSED>
__global__ void __launch_bounds__(WARPS * 32)
decode_split_kernel(const uint8_t* __restrict__ q, const uint8_t* __restrict__ k,
                    const uint8_t* __restrict__ v, int L, int S, int seg_len, float scale_log2,
                    float* __restrict__ seg_m, float* __restrict__ seg_l,
                    float* __restrict__ seg_acc, FusedMerge fm) {
  constexpr int E = Chunk<T>::N;       // elements per 16-byte chunk
  constexpr int D = 16 * E;            // 16 chunks per 256-byte key row
  constexpr int ROW_BYTES = 256;

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int half = lane >> 4;
  const int c = lane & 15;

  const int row = blockIdx.x / S;
  const int seg = blockIdx.x - row * S;
  const int a = min(L, seg * seg_len);
  const int b = min(L, a + seg_len);

  // this lane's chunk of q, pre-scaled into the log2 domain (R = gridDim.x / S rows)
  float qf[E];
  uint4 qv = make_uint4(0, 0, 0, 0);
  if (RF_SPAN_OK((size_t)row * ROW_BYTES + c * 16, 16, (long long)(gridDim.x / S) * ROW_BYTES))
    qv = *reinterpret_cast<const uint4*>(q + (size_t)row * ROW_BYTES + c * 16);
  Chunk<T>::unpack(qv, qf);
#pragma unroll
  for (int e = 0; e < E; ++e) qf[e] *= scale_log2;

  const uint8_t* kr = k + (size_t)row * L * ROW_BYTES + c * 16;
  const uint8_t* vr = v + (size_t)row * L * ROW_BYTES + c * 16;

  float m = -INFINITY, l = 0.f;
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;

  for (int t0 = a + warp * 2 * U; t0 < b; t0 += WARPS * 2 * U) {
    uint4 kv[U], vv[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int key = t0 + 2 * u + half;
      if (key < b && RF_SPAN_OK(((size_t)row * L + key) * ROW_BYTES + c * 16, 16,
                                (long long)(gridDim.x / S) * L * ROW_BYTES)) {
        kv[u] = ld_stream_v4(kr + (size_t)key * ROW_BYTES);
        vv[u] = ld_stream_v4(vr + (size_t)key * ROW_BYTES);
      } else {
        kv[u] = make_uint4(0, 0, 0, 0);
        vv[u] = make_uint4(0, 0, 0, 0);
      }
    }
    float s[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      float kf[E];
      Chunk<T>::unpack(kv[u], kf);
      float d = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) d = fmaf(qf[e], kf[e], d);
      s[u] = d;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) s[u] = group_sum<16>(s[u]);
    float mt = -INFINITY;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (t0 + 2 * u + half >= b) s[u] = -INFINITY;
      mt = fmaxf(mt, s[u]);
    }
    const float mn = fmaxf(m, mt);
    const float ref = ref_of(mn);
    const float corr = exp2f(m - ref);
    l *= corr;
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] *= corr;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const float p = exp2f(s[u] - ref);
      l += p;
      float vf[E];
      Chunk<T>::unpack(vv[u], vf);
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] = fmaf(p, vf[e], acc[e]);
    }
    m = mn;
  }

  // merge the two half-warp states (lane c and lane c+16 own the same chunk)
  {
    const float mo = __shfl_xor_sync(0xffffffffu, m, 16);
    const float lo = __shfl_xor_sync(0xffffffffu, l, 16);
    const float mn = fmaxf(m, mo);
    const float ref = ref_of(mn);
    const float cs = exp2f(m - ref), co = exp2f(mo - ref);
    l = l * cs + lo * co;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const float ao = __shfl_xor_sync(0xffffffffu, acc[e], 16);
      acc[e] = acc[e] * cs + ao * co;
    }
    m = mn;
  }

  // merge the CTA's warps through shared memory
  __shared__ float sm_m[WARPS], sm_l[WARPS];
  __shared__ float sm_acc[WARPS][D];
  if (lane < 16) {
#pragma unroll
    for (int e = 0; e < E; ++e) sm_acc[warp][c * E + e] = acc[e];
  }
  if (lane == 0) {
    sm_m[warp] = m;
    sm_l[warp] = l;
  }
  __syncthreads();
  const size_t state = (size_t)row * S + seg;
  for (int d = threadIdx.x; d < D; d += WARPS * 32) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < WARPS; ++w) M = fmaxf(M, sm_m[w]);
    const float ref = ref_of(M);
    float A = 0.f, Lsum = 0.f;
#pragma unroll
    for (int w = 0; w < WARPS; ++w) {
      const float f = exp2f(sm_m[w] - ref);
      A = fmaf(f, sm_acc[w][d], A);
      Lsum = fmaf(f, sm_l[w], Lsum);
    }
    if (RF_IDX_OK(state * D + d, (long long)gridDim.x * D)) seg_acc[state * D + d] = A;
    if (d == 0 && RF_IDX_OK(state, gridDim.x)) {
      seg_m[state] = M * kLn2;   // -inf stays -inf
      seg_l[state] = Lsum;
    }
  }
  if constexpr (FUSED) {
    // last arriver of the row merges: publish this segment, then count it
    __shared__ int last;
    __syncthreads();
    if (threadIdx.x == 0) {
      __threadfence();
      const int seen = RF_IDX_OK(row, gridDim.x / S) ? atomicAdd(fm.counters + row, 1) : -1;
      last = seen == S - 1;
    }
    __syncthreads();
    if (!last) return;
    __threadfence();
    const size_t s0 = (size_t)row * S;
    for (int d = threadIdx.x; d < D; d += WARPS * 32) {
      // L2 reads (__ldcg): the states were written by other CTAs of this launch
      float Mx = -INFINITY;
      for (int s = 0; s < S; ++s) Mx = fmaxf(Mx, __ldcg(seg_m + s0 + s));
      const float ref = Mx == -INFINITY ? 0.f : Mx;
      float A = 0.f, Lsum = 0.f;
      for (int s = 0; s < S; ++s) {
        const float f = expf(__ldcg(seg_m + s0 + s) - ref);
        Lsum = fmaf(f, __ldcg(seg_l + s0 + s), Lsum);
        A = fmaf(f, __ldcg(seg_acc + (s0 + s) * D + d), A);
      }
      const float o = A / Lsum;
      if (RF_IDX_OK((size_t)row * D + d, (long long)(gridDim.x / S) * D)) {
        if (fm.out_bf16)
          reinterpret_cast<__nv_bfloat16*>(fm.out)[(size_t)row * D + d] = __float2bfloat16_rn(o);
        else
          reinterpret_cast<float*>(fm.out)[(size_t)row * D + d] = o;
      }
      if (d == 0) {
        if (fm.lse != nullptr) fm.lse[row] = Mx + logf(Lsum);
        fm.counters[row] = 0;               // ready for the next call
      }
    }
  }
}

// One warp per (row, 128-wide block of D) -- D/128 warps per row for D >= 128,
// one for D = 64.  Lane j owns 4 consecutive elements of the block (lanes
// 0..15 for D = 64); every warp of a row recomputes the row's segment weights
// exp(m_s - M) from seg_m (S values, cached), and the first writes lse.
template <int D, bool BF16_OUT>
__global__ void __launch_bounds__(256)
state_merge_kernel(const float* __restrict__ seg_m, const float* __restrict__ seg_l,
                   const float* __restrict__ seg_acc, int R, int S, void* __restrict__ out,
                   float* __restrict__ lse) {
  constexpr int PARTS = D >= 128 ? D / 128 : 1;
  constexpr int V4 = D / 4;                     // float4s per state
  constexpr int LANES = V4 < 32 ? V4 : 32;      // float4s of this warp's block
  const int lane = threadIdx.x & 31;
  const long long wid = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int row = (int)(wid / PARTS);
  const int part = (int)(wid % PARTS);
  if (row >= R) return;
  const float* mr = seg_m + (size_t)row * S;
  const float* lr = seg_l + (size_t)row * S;

  float M = -INFINITY;
  for (int s = lane; s < S; s += 32)
    if (RF_IDX_OK((size_t)row * S + s, (long long)R * S)) M = fmaxf(M, mr[s]);
  M = group_max<32>(M);
  const float ref = M == -INFINITY ? 0.f : M;

  float Lsum = 0.f;
  for (int s = lane; s < S; s += 32)
    if (RF_IDX_OK((size_t)row * S + s, (long long)R * S)) Lsum = fmaf(expf(mr[s] - ref), lr[s], Lsum);
  Lsum = group_sum<32>(Lsum);

  if (lane < LANES) {
    float4 A = make_float4(0.f, 0.f, 0.f, 0.f);
    const float4* ar =
        reinterpret_cast<const float4*>(seg_acc + (size_t)row * S * D) + part * 32 + lane;
    for (int s = 0; s < S; ++s) {
      if (!RF_IDX_OK(((size_t)row * S + s) * V4 + part * 32 + lane, (long long)R * S * V4)) continue;
      const float f = expf(mr[s] - ref);
      const float4 x = ar[(size_t)s * V4];
      A.x = fmaf(f, x.x, A.x);
      A.y = fmaf(f, x.y, A.y);
      A.z = fmaf(f, x.z, A.z);
      A.w = fmaf(f, x.w, A.w);
    }
    const float inv = 1.f / Lsum;
    A.x *= inv; A.y *= inv; A.z *= inv; A.w *= inv;
    const size_t o = (size_t)row * V4 + part * 32 + lane;
    if (!RF_IDX_OK(o, (long long)R * V4)) {
    } else if (BF16_OUT) {
      uint2 p;
      p.x = pack_bf16x2(A.x, A.y);
      p.y = pack_bf16x2(A.z, A.w);
      reinterpret_cast<uint2*>(out)[o] = p;
    } else {
      reinterpret_cast<float4*>(out)[o] = A;
    }
  }
  if (lse != nullptr && lane == 0 && part == 0 && RF_IDX_OK(row, R)) lse[row] = M + logf(Lsum);
}

}  // namespace

template <bool FUSED>
static rf_status launch_split_t(const void* q, const void* k, const void* v, int R, int L, int D, int S,
                         float scale, int dtype, float* seg_m, float* seg_l, float* seg_acc,
                         FusedMerge fm, cudaStream_t st) {
  const int seg_len = (L + S - 1) / S;
  const float sl2 = scale * kLog2e;
  const unsigned grid = (unsigned)R * (unsigned)S;
  constexpr int WARPS = 8;
  const auto* qb = static_cast<const uint8_t*>(q);
  const auto* kb = static_cast<const uint8_t*>(k);
  const auto* vb = static_cast<const uint8_t*>(v);
  // Segments of at most 128 keys: a shallower unroll (4 key pairs in flight
  // per half-warp instead of 8, far fewer registers) lets an SM hold more
  // CTAs, which is what keeps memory busy when every CTA's stream is short
  // (measured on 512-key rows, D = 64: 5 % faster at 128 keys per segment,
  // 28 % at 64; slower from 256 keys up).  With few CTAs in all (a single
  // row) the deeper unroll keeps more in flight and stays faster.
  const bool short_seg = seg_len <= 128 && grid >= 1024;   // many CTAs: occupancy decides
  if (dtype == RF_BF16 && D == 128) {
    if (short_seg)
      decode_split_kernel<Bf16Tag, WARPS, 4, FUSED><<<grid, WARPS * 32, 0, st>>>(
          qb, kb, vb, L, S, seg_len, sl2, seg_m, seg_l, seg_acc, fm);
    else
      decode_split_kernel<Bf16Tag, WARPS, 8, FUSED><<<grid, WARPS * 32, 0, st>>>(
          qb, kb, vb, L, S, seg_len, sl2, seg_m, seg_l, seg_acc, fm);
  } else if (dtype == RF_F32 && D == 64) {
    if (short_seg)
      decode_split_kernel<float, WARPS, 4, FUSED><<<grid, WARPS * 32, 0, st>>>(
          qb, kb, vb, L, S, seg_len, sl2, seg_m, seg_l, seg_acc, fm);
    else
      decode_split_kernel<float, WARPS, 8, FUSED><<<grid, WARPS * 32, 0, st>>>(
          qb, kb, vb, L, S, seg_len, sl2, seg_m, seg_l, seg_acc, fm);
  } else {
    return RF_ERR_UNSUPPORTED;
  }
  return launch_status();
}

rf_status launch_decode_split(const void* q, const void* k, const void* v, int R, int L, int D,
                              int S, float scale, int dtype, float* seg_m, float* seg_l,
                              float* seg_acc, cudaStream_t st) {
  return launch_split_t<false>(q, k, v, R, L, D, S, scale, dtype, seg_m, seg_l, seg_acc,
                               FusedMerge{nullptr, nullptr, nullptr, 0}, st);
}

rf_status launch_decode_fused(const void* q, const void* k, const void* v, int R, int L, int D,
                              int S, float scale, int dtype, float* seg_m, float* seg_l,
                              float* seg_acc, int* counters, void* out, int out_dtype, float* lse,
                              cudaStream_t st) {
  return launch_split_t<true>(q, k, v, R, L, D, S, scale, dtype, seg_m, seg_l, seg_acc,
                              FusedMerge{counters, out, lse, out_dtype == RF_BF16 ? 1 : 0}, st);
}

rf_status launch_state_merge(const float* seg_m, const float* seg_l, const float* seg_acc, int R,
                             int S, int D, void* out, int out_dtype, float* lse, cudaStream_t st) {
  const long long warps = (long long)R * (D >= 128 ? D / 128 : 1);
  const unsigned grid = (unsigned)((warps + 7) / 8);
  const bool bf = out_dtype == RF_BF16;
  if (D == 128) {
    if (bf) state_merge_kernel<128, true><<<grid, 256, 0, st>>>(seg_m, seg_l, seg_acc, R, S, out, lse);
    else state_merge_kernel<128, false><<<grid, 256, 0, st>>>(seg_m, seg_l, seg_acc, R, S, out, lse);
  } else if (D == 64) {
    if (bf) state_merge_kernel<64, true><<<grid, 256, 0, st>>>(seg_m, seg_l, seg_acc, R, S, out, lse);
    else state_merge_kernel<64, false><<<grid, 256, 0, st>>>(seg_m, seg_l, seg_acc, R, S, out, lse);
  } else if (D == 512) {
    if (bf) state_merge_kernel<512, true><<<grid, 256, 0, st>>>(seg_m, seg_l, seg_acc, R, S, out, lse);
    else state_merge_kernel<512, false><<<grid, 256, 0, st>>>(seg_m, seg_l, seg_acc, R, S, out, lse);
  } else {
    return RF_ERR_UNSUPPORTED;
  }
  return launch_status();
}

RF_BOUNDS_WORD_OF_THIS_FILE

}  // namespace rf
