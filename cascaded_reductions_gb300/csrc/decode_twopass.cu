// Non-incremental split-KV decode: the ablation of the incremental form.
//
// RedFuser episode transcript, cue 45: the non-incremental version only fits
// when each block handles short sequences, and at matched parallelism it can
// be faster; longer per-block sequences need the incremental form.  This
// kernel is that non-incremental counterpart of decode_split_kernel, with the
// same inputs and the same segment states out:
//   phase 1  stream the segment's K rows, keep every score of the segment in
//            shared memory, and reduce the segment max M (reduction 1);
//   phase 2  stream the segment's V rows and accumulate l = sum exp(s - M),
//            acc = sum exp(s - M) v with the final max: no rescaling at all.
// The scores must fit in shared memory, so segments are limited to
// kTwopassMaxSeg keys.  Bytes read are the same as the incremental kernel's
// (K once, V once); what changes is on-chip storage, which grows with the
// segment length, and a block-wide barrier between the two phases.
//
// Layout per CTA and warp as in decode_split_kernel: a 16-byte load
// instruction of a warp covers two key rows (256 bytes each), lane half h
// takes key 2u+h of a tile and lane c the c-th 16-byte chunk of it.

#include <math.h>

#include "common.cuh"

namespace rf {

constexpr int kTwopassMaxSeg = 16384;

namespace {

template <typename T, int WARPS, int U>
__global__ void __launch_bounds__(WARPS * 32)
decode_twopass_kernel(const uint8_t* __restrict__ q, const uint8_t* __restrict__ k,
                      const uint8_t* __restrict__ v, int L, int S, int seg_len, float scale_log2,
                      float* __restrict__ seg_m, float* __restrict__ seg_l,
                      float* __restrict__ seg_acc) {
  constexpr int E = Chunk<T>::N;
  constexpr int D = 16 * E;
  constexpr int ROW_BYTES = 256;
  extern __shared__ float sc[];                 // the segment's scores, log2 domain
  __shared__ float sm_red[WARPS];
  __shared__ float sm_l[WARPS];
  __shared__ float sm_acc[WARPS][D];

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int half = lane >> 4;
  const int c = lane & 15;
  const int row = blockIdx.x / S;
  const int seg = blockIdx.x - row * S;
  const int a = min(L, seg * seg_len);
  const int b = min(L, a + seg_len);

  float qf[E];
  uint4 qv = make_uint4(0, 0, 0, 0);
  if (RF_SPAN_OK((size_t)row * ROW_BYTES + c * 16, 16, (long long)(gridDim.x / S) * ROW_BYTES))
    qv = *reinterpret_cast<const uint4*>(q + (size_t)row * ROW_BYTES + c * 16);
  Chunk<T>::unpack(qv, qf);
#pragma unroll
  for (int e = 0; e < E; ++e) qf[e] *= scale_log2;
  const uint8_t* kr = k + (size_t)row * L * ROW_BYTES + c * 16;
  const uint8_t* vr = v + (size_t)row * L * ROW_BYTES + c * 16;

  // phase 1: scores and their max
  float mloc = -INFINITY;
  for (int t0 = a + warp * 2 * U; t0 < b; t0 += WARPS * 2 * U) {
    uint4 kv[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int key = t0 + 2 * u + half;
      kv[u] = key < b && RF_SPAN_OK(((size_t)row * L + key) * ROW_BYTES + c * 16, 16,
                                    (long long)(gridDim.x / S) * L * ROW_BYTES)
                  ? ld_stream_v4(kr + (size_t)key * ROW_BYTES)
                  : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      float kf[E];
      Chunk<T>::unpack(kv[u], kf);
      float d = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) d = fmaf(qf[e], kf[e], d);
      d = group_sum<16>(d);
      const int key = t0 + 2 * u + half;
      if (key < b) {
        if (c == 0 && RF_IDX_OK(key - a, seg_len)) sc[key - a] = d;   // seg_len floats of smem
        mloc = fmaxf(mloc, d);
      }
    }
  }
  mloc = group_max<32>(mloc);
  if (lane == 0) sm_red[warp] = mloc;
  __syncthreads();                               // scores and per-warp maxima visible
  float M = -INFINITY;
#pragma unroll
  for (int w = 0; w < WARPS; ++w) M = fmaxf(M, sm_red[w]);
  const float ref = ref_of(M);

  // phase 2: weighted sum with the final max
  float l = 0.f;
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  for (int t0 = a + warp * 2 * U; t0 < b; t0 += WARPS * 2 * U) {
    uint4 vv[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int key = t0 + 2 * u + half;
      vv[u] = key < b && RF_SPAN_OK(((size_t)row * L + key) * ROW_BYTES + c * 16, 16,
                                    (long long)(gridDim.x / S) * L * ROW_BYTES)
                  ? ld_stream_v4(vr + (size_t)key * ROW_BYTES)
                  : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int key = t0 + 2 * u + half;
      const float p = key < b && RF_IDX_OK(key - a, seg_len) ? exp2f(sc[key - a] - ref) : 0.f;
      l += p;
      float vf[E];
      Chunk<T>::unpack(vv[u], vf);
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] = fmaf(p, vf[e], acc[e]);
    }
  }
  // every lane of a half saw the same keys: combine the halves, then the warps
  l += __shfl_xor_sync(0xffffffffu, l, 16);
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], 16);
  if (lane < 16) {
#pragma unroll
    for (int e = 0; e < E; ++e) sm_acc[warp][c * E + e] = acc[e];
  }
  if (lane == 0) sm_l[warp] = l;
  __syncthreads();
  const size_t state = (size_t)row * S + seg;
  for (int d = threadIdx.x; d < D; d += WARPS * 32) {
    float A = 0.f;
#pragma unroll
    for (int w = 0; w < WARPS; ++w) A += sm_acc[w][d];
    if (RF_IDX_OK(state * D + d, (long long)gridDim.x * D)) seg_acc[state * D + d] = A;
    if (d == 0 && RF_IDX_OK(state, gridDim.x)) {
      float Ls = 0.f;
#pragma unroll
      for (int w = 0; w < WARPS; ++w) Ls += sm_l[w];
      seg_m[state] = M * kLn2;                  // -inf stays -inf for an empty segment
      seg_l[state] = Ls;
    }
  }
}

template <typename T>
rf_status launch_twopass_t(const void* q, const void* k, const void* v, int R, int L, int S,
                           int seg_len, float sl2, float* seg_m, float* seg_l, float* seg_acc,
                           cudaStream_t st) {
  constexpr int WARPS = 8, U = 8;
  const size_t smem = (size_t)(seg_len > 0 ? seg_len : 1) * sizeof(float);
  auto kern = decode_twopass_kernel<T, WARPS, U>;
  static std::atomic<uint64_t> attr{0};
  if (smem_attr(kern, kTwopassMaxSeg * sizeof(float), attr) != RF_OK) return RF_ERR_CUDA;
  const unsigned grid = (unsigned)R * (unsigned)S;
  kern<<<grid, WARPS * 32, smem, st>>>(static_cast<const uint8_t*>(q),
                                       static_cast<const uint8_t*>(k),
                                       static_cast<const uint8_t*>(v), L, S, seg_len, sl2, seg_m,
                                       seg_l, seg_acc);
  return launch_status();
}

}  // namespace

rf_status launch_decode_twopass(const void* q, const void* k, const void* v, int R, int L, int D,
                                int S, float scale, int dtype, float* seg_m, float* seg_l,
                                float* seg_acc, cudaStream_t st) {
  const int seg_len = (L + S - 1) / S;
  if (seg_len > kTwopassMaxSeg) return RF_ERR_UNSUPPORTED;
  const float sl2 = scale * kLog2e;
  if (dtype == RF_BF16 && D == 128)
    return launch_twopass_t<Bf16Tag>(q, k, v, R, L, S, seg_len, sl2, seg_m, seg_l, seg_acc, st);
  if (dtype == RF_F32 && D == 64)
    return launch_twopass_t<float>(q, k, v, R, L, S, seg_len, sl2, seg_m, seg_l, seg_acc, st);
  return RF_ERR_UNSUPPORTED;
}

RF_BOUNDS_WORD_OF_THIS_FILE

}  // namespace rf
