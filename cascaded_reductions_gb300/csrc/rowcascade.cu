// Single-row cascades at several fusion levels: safe softmax of a row,
// variance, moment of inertia (RedFuser episode transcript, cue 47: safe
// softmax over 1K-8K elements at thread, warp and block fusion levels, and
// variance and moment of inertia as further cascades), and layer
// normalisation (the bookshelf explainer's "Problem" section names
// normalisation layers among the cascaded reductions).
//
// Every cascade here has two dependent reductions; the fused forms carry a
// mergeable state through one read of the row (cue 31: rescale the state for
// the changed earlier result, then add the new term):
//   softmax   (m, l):          merge  M = max, l = l_a e^{m_a-M} + l_b e^{m_b-M}
//   variance  (n, mean, M2):   merge  d = mean_b - mean_a,
//                              mean = mean_a + d n_b/n, M2 = M2_a + M2_b + d^2 n_a n_b / n
//   inertia   (M, c, I):       merge  d = c_b - c_a, c = c_a + d M_b/M,
//                              I = I_a + I_b + |d|^2 M_a M_b / M  (parallel-axis theorem)
// The fusion level is the level of the reduction tree at which each new
// element (or tile) is folded into the state (cue 47's study):
//   RF_FUSE_THREAD   each thread folds its elements one at a time, then the
//                    thread states are merged across the warp and the block;
//   RF_FUSE_WARP     each warp reduces a 128-element tile with shuffles and
//                    folds the tile into a warp state; warps merge at the end;
//   RF_FUSE_BLOCK    the block reduces a 1024-element tile (shuffles + shared
//                    memory) and folds it into one block state;
//   RF_FUSE_NONE     the unfused cascade: one kernel per reduction, each
//                    re-reading the row from global memory.
// One CTA of 256 threads per row; 16-byte loads issued several at a time
// before they are folded, rows of n % 4 == 0 floats.
// Softmax keeps the row in registers between the reduction and the write
// (n <= 8192 for the fused levels).

#include <math.h>

#include "common.cuh"

namespace rf {
namespace {

constexpr int TH = 256;
constexpr int NW = TH / 32;
constexpr int U = 4;                     // 16-byte loads in flight per thread (variance)

// ------------------------------------------------------------- softmax ----
struct SmState {
  float m, l;
};

__device__ __forceinline__ SmState sm_merge(SmState a, SmState b) {
  const float M = fmaxf(a.m, b.m);
  const float ref = M == -INFINITY ? 0.f : M;
  return {M, a.l * __expf(a.m - ref) + b.l * __expf(b.m - ref)};
}

__device__ __forceinline__ SmState sm_block_merge(SmState s, SmState* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    SmState t{__shfl_xor_sync(0xffffffffu, s.m, o), __shfl_xor_sync(0xffffffffu, s.l, o)};
    s = sm_merge(s, t);
  }
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = s;
  __syncthreads();
  SmState r = red[0];
#pragma unroll
  for (int w = 1; w < NW; ++w) r = sm_merge(r, red[w]);
  return r;
}

__device__ __forceinline__ float bmax(float v, float* red) {
  v = group_max<32>(v);
  __syncthreads();                       // red may still be read from a previous use
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float r = red[0];
#pragma unroll
  for (int w = 1; w < NW; ++w) r = fmaxf(r, red[w]);
  return r;
}

__device__ __forceinline__ float bsum(float v, float* red) {
  v = group_sum<32>(v);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float r = red[0];
#pragma unroll
  for (int w = 1; w < NW; ++w) r += red[w];
  return r;
}

// Bounds checks of the row accesses (no-ops unless built with RF_CHECK_BOUNDS):
// float4 chunk c of this block's row in a buffer of gridDim.x rows of `width`
// floats, and chunk c of a vector of n floats.  Outputs of one value per row
// are indexed by blockIdx.x alone and need none.
__device__ __forceinline__ bool row_ok(long long c, long long width) {
  return RF_SPAN_OK((long long)blockIdx.x * width + 4 * c, 4, (long long)gridDim.x * width);
}
__device__ __forceinline__ bool vec_ok(long long c, long long n) { return RF_SPAN_OK(4 * c, 4, n); }

__device__ __forceinline__ float get(const float4& v, int e) {
  return e == 0 ? v.x : (e == 1 ? v.y : (e == 2 ? v.z : v.w));
}

template <int LEVEL, int VPT>
__global__ void __launch_bounds__(TH)
softmax_fused_kernel(const float* __restrict__ x, int n, float* __restrict__ y) {
  __shared__ SmState red_s[NW];
  __shared__ float red_f[NW];
  const int n4 = n >> 2;
  const float4* xr = reinterpret_cast<const float4*>(x + (size_t)blockIdx.x * n);
  float4* yr = reinterpret_cast<float4*>(y + (size_t)blockIdx.x * n);
  const float NI = -INFINITY;
  float4 v[VPT];
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int c = i * TH + threadIdx.x;
    v[i] = c < n4 && row_ok(c, n) ? __ldcs(xr + c) : make_float4(NI, NI, NI, NI);
  }
  SmState st{-INFINITY, 0.f};
  if (LEVEL == RF_FUSE_THREAD) {
    // one element at a time: m' = max(m, x), l = l e^{m - m'} + e^{x - m'}
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      if (i * TH + (int)threadIdx.x >= n4) break;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float xe = get(v[i], e);
        const float mn = fmaxf(st.m, xe);
        st.l = st.l * __expf(st.m - mn) + __expf(xe - mn);
        st.m = mn;
      }
    }
    st = sm_block_merge(st, red_s);
  } else if (LEVEL == RF_FUSE_WARP) {
    // one 128-element tile per warp at a time, state uniform across the warp
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      float tm = fmaxf(fmaxf(v[i].x, v[i].y), fmaxf(v[i].z, v[i].w));
      tm = group_max<32>(tm);
      if (tm == -INFINITY) continue;        // the whole tile is past the row's end
      const float mn = fmaxf(st.m, tm);
      float ps = __expf(v[i].x - mn) + __expf(v[i].y - mn) + __expf(v[i].z - mn) + __expf(v[i].w - mn);
      ps = group_sum<32>(ps);
      st.l = st.l * __expf(st.m - mn) + ps;
      st.m = mn;
    }
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red_s[threadIdx.x >> 5] = st;
    __syncthreads();
    SmState r = red_s[0];
#pragma unroll
    for (int w = 1; w < NW; ++w) r = sm_merge(r, red_s[w]);
    st = r;
  } else {
    // one 1024-element tile per block at a time, one block-wide state
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const float tm = bmax(fmaxf(fmaxf(v[i].x, v[i].y), fmaxf(v[i].z, v[i].w)), red_f);
      if (tm == -INFINITY) break;           // past the row's end for the whole block
      const float mn = fmaxf(st.m, tm);
      const float ps = bsum(__expf(v[i].x - mn) + __expf(v[i].y - mn) + __expf(v[i].z - mn) +
                                __expf(v[i].w - mn),
                            red_f);
      st.l = st.l * __expf(st.m - mn) + ps;
      st.m = mn;
    }
  }
  const float inv = 1.f / st.l;
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int c = i * TH + threadIdx.x;
    if (c < n4 && row_ok(c, n))
      __stcs(yr + c, make_float4(__expf(v[i].x - st.m) * inv, __expf(v[i].y - st.m) * inv,
                                 __expf(v[i].z - st.m) * inv, __expf(v[i].w - st.m) * inv));
  }
}

// unfused softmax: three kernels, each reading the row from global memory
__global__ void __launch_bounds__(TH)
softmax_max_kernel(const float* __restrict__ x, int n, float* __restrict__ work) {
  __shared__ float red[NW];
  const float4* xr = reinterpret_cast<const float4*>(x + (size_t)blockIdx.x * n);
  float m = -INFINITY;
  for (int c = threadIdx.x; c < (n >> 2); c += TH) {
    if (!row_ok(c, n)) continue;
    const float4 v = __ldcs(xr + c);
    m = fmaxf(m, fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w)));
  }
  m = bmax(m, red);
  if (threadIdx.x == 0) work[blockIdx.x] = m;
}

__global__ void __launch_bounds__(TH)
softmax_sum_kernel(const float* __restrict__ x, int n, int R, float* __restrict__ work) {
  __shared__ float red[NW];
  const float4* xr = reinterpret_cast<const float4*>(x + (size_t)blockIdx.x * n);
  const float m = work[blockIdx.x];
  float s = 0.f;
  for (int c = threadIdx.x; c < (n >> 2); c += TH) {
    if (!row_ok(c, n)) continue;
    const float4 v = __ldcs(xr + c);
    s += __expf(v.x - m) + __expf(v.y - m) + __expf(v.z - m) + __expf(v.w - m);
  }
  s = bsum(s, red);
  if (threadIdx.x == 0 && RF_IDX_OK(R + blockIdx.x, 2LL * gridDim.x)) work[R + blockIdx.x] = s;
}

__global__ void __launch_bounds__(TH)
softmax_norm_kernel(const float* __restrict__ x, int n, int R, const float* __restrict__ work,
                    float* __restrict__ y) {
  const float4* xr = reinterpret_cast<const float4*>(x + (size_t)blockIdx.x * n);
  float4* yr = reinterpret_cast<float4*>(y + (size_t)blockIdx.x * n);
  const float m = work[blockIdx.x], inv = 1.f / work[R + blockIdx.x];
  for (int c = threadIdx.x; c < (n >> 2); c += TH) {
    if (!row_ok(c, n)) continue;
    const float4 v = __ldcs(xr + c);
    __stcs(yr + c, make_float4(__expf(v.x - m) * inv, __expf(v.y - m) * inv,
                               __expf(v.z - m) * inv, __expf(v.w - m) * inv));
  }
}

// ------------------------------------------------------------ variance ----
struct VarState {
  float n, mean, m2;
};

__device__ __forceinline__ VarState var_merge(VarState a, VarState b) {
  const float n = a.n + b.n;
  if (n == 0.f) return a;
  const float d = b.mean - a.mean;
  const float fb = b.n / n;
  return {n, a.mean + d * fb, a.m2 + b.m2 + d * d * a.n * fb};
}

__device__ __forceinline__ VarState var_warp_merge(VarState s) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    VarState t{__shfl_xor_sync(0xffffffffu, s.n, o), __shfl_xor_sync(0xffffffffu, s.mean, o),
               __shfl_xor_sync(0xffffffffu, s.m2, o)};
    s = var_merge(s, t);
  }
  return s;
}

// mean and M2 of a tile of `cnt` values held as per-thread partial sums, all
// threads of the warp (or block) taking part; returns the tile state
template <int LEVEL>
__global__ void __launch_bounds__(TH)
variance_fused_kernel(const float* __restrict__ x, int n, float* __restrict__ mean_out,
                      float* __restrict__ var_out) {
  __shared__ VarState red_v[NW];
  __shared__ float red_f[NW];
  const int n4 = n >> 2;
  const float4* xr = reinterpret_cast<const float4*>(x + (size_t)blockIdx.x * n);
  VarState st{0.f, 0.f, 0.f};
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (LEVEL == RF_FUSE_THREAD) {
    // Welford, one element at a time (U loads in flight per thread)
    for (int base = 0; base < n4; base += TH * U) {
      float4 v[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int c = base + u * TH + (int)threadIdx.x;
        v[u] = c < n4 && row_ok(c, n) ? __ldcs(xr + c) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (base + u * TH + (int)threadIdx.x >= n4) break;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float xe = get(v[u], e);
          st.n += 1.f;
          const float d = xe - st.mean;
          st.mean += __fdividef(d, st.n);
          st.m2 += d * (xe - st.mean);
        }
      }
    }
    st = var_warp_merge(st);
    if (lane == 0) red_v[warp] = st;
    __syncthreads();
    st = red_v[0];
    for (int w = 1; w < NW; ++w) st = var_merge(st, red_v[w]);
  } else if (LEVEL == RF_FUSE_WARP) {
    // one 128-element tile per warp: tile mean, tile M2, fold into the warp state
    for (int base0 = warp * 32; base0 < n4; base0 += TH * U) {
      float4 v[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int c = base0 + u * TH + lane;
        v[u] = c < n4 && row_ok(c, n) ? __ldcs(xr + c) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int base = base0 + u * TH;
        if (base >= n4) break;                  // uniform across the warp
        const bool ok = base + lane < n4;
        const float cnt = (float)(4 * min(32, n4 - base));
        const float tmean = group_sum<32>(v[u].x + v[u].y + v[u].z + v[u].w) / cnt;
        const float dx = v[u].x - tmean, dy = v[u].y - tmean, dz = v[u].z - tmean,
                    dw = v[u].w - tmean;
        const float tm2 = group_sum<32>(ok ? dx * dx + dy * dy + dz * dz + dw * dw : 0.f);
        st = var_merge(st, VarState{cnt, tmean, tm2});
      }
    }
    if (lane == 0) red_v[warp] = st;
    __syncthreads();
    st = red_v[0];
    for (int w = 1; w < NW; ++w) st = var_merge(st, red_v[w]);
  } else {
    // one 1024-element tile per block: block mean, block M2, fold into the block state
    for (int base0 = 0; base0 < n4; base0 += TH * U) {
      float4 v[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int c = base0 + u * TH + (int)threadIdx.x;
        v[u] = c < n4 && row_ok(c, n) ? __ldcs(xr + c) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int base = base0 + u * TH;
        if (base >= n4) break;                  // uniform across the block
        const bool ok = base + (int)threadIdx.x < n4;
        const float cnt = (float)(4 * min(TH, n4 - base));
        const float tmean = bsum(v[u].x + v[u].y + v[u].z + v[u].w, red_f) / cnt;
        const float dx = v[u].x - tmean, dy = v[u].y - tmean, dz = v[u].z - tmean,
                    dw = v[u].w - tmean;
        const float tm2 = bsum(ok ? dx * dx + dy * dy + dz * dz + dw * dw : 0.f, red_f);
        st = var_merge(st, VarState{cnt, tmean, tm2});
      }
    }
  }
  if (threadIdx.x == 0) {
    mean_out[blockIdx.x] = st.mean;
    var_out[blockIdx.x] = st.m2 / (float)n;
  }
}

__global__ void __launch_bounds__(TH)
mean_kernel(const float* __restrict__ x, int n, float* __restrict__ mean_out) {
  __shared__ float red[NW];
  const float4* xr = reinterpret_cast<const float4*>(x + (size_t)blockIdx.x * n);
  float s = 0.f;
  for (int c = threadIdx.x; c < (n >> 2); c += TH) {
    if (!row_ok(c, n)) continue;
    const float4 v = __ldcs(xr + c);
    s += (v.x + v.y) + (v.z + v.w);
  }
  s = bsum(s, red);
  if (threadIdx.x == 0) mean_out[blockIdx.x] = s / (float)n;
}

__global__ void __launch_bounds__(TH)
var_from_mean_kernel(const float* __restrict__ x, int n, const float* __restrict__ mean_in,
                     float* __restrict__ var_out) {
  __shared__ float red[NW];
  const float4* xr = reinterpret_cast<const float4*>(x + (size_t)blockIdx.x * n);
  const float mu = mean_in[blockIdx.x];
  float s = 0.f;
  for (int c = threadIdx.x; c < (n >> 2); c += TH) {
    if (!row_ok(c, n)) continue;
    const float4 v = __ldcs(xr + c);
    const float dx = v.x - mu, dy = v.y - mu, dz = v.z - mu, dw = v.w - mu;
    s += (dx * dx + dy * dy) + (dz * dz + dw * dw);
  }
  s = bsum(s, red);
  if (threadIdx.x == 0) var_out[blockIdx.x] = s / (float)n;
}

// ---------------------------------------------------- moment of inertia ----
struct InState {
  float M, cx, cy, cz, I;
};

__device__ __forceinline__ InState in_merge(InState a, InState b) {
  const float M = a.M + b.M;
  if (M == 0.f) return a;
  const float fb = b.M / M;
  const float dx = b.cx - a.cx, dy = b.cy - a.cy, dz = b.cz - a.cz;
  return {M, a.cx + dx * fb, a.cy + dy * fb, a.cz + dz * fb,
          a.I + b.I + (dx * dx + dy * dy + dz * dz) * a.M * fb};
}

__device__ __forceinline__ InState in_shfl_merge(InState s, int o) {
  InState t{__shfl_xor_sync(0xffffffffu, s.M, o), __shfl_xor_sync(0xffffffffu, s.cx, o),
            __shfl_xor_sync(0xffffffffu, s.cy, o), __shfl_xor_sync(0xffffffffu, s.cz, o),
            __shfl_xor_sync(0xffffffffu, s.I, o)};
  return in_merge(s, t);
}

// tile state of up to 4 points per thread reduced over a warp (or block):
// M = sum m, c = sum m p / M, I = sum m |p - c|^2
template <bool BLOCK>
__device__ __forceinline__ InState in_tile(const float4& m, const float4& px, const float4& py,
                                           const float4& pz, float* red) {
  auto red_sum = [&](float v) { return BLOCK ? bsum(v, red) : group_sum<32>(v); };
  const float Mt = red_sum((m.x + m.y) + (m.z + m.w));
  if (Mt == 0.f) return InState{0.f, 0.f, 0.f, 0.f, 0.f};
  const float cx = red_sum(m.x * px.x + m.y * px.y + m.z * px.z + m.w * px.w) / Mt;
  const float cy = red_sum(m.x * py.x + m.y * py.y + m.z * py.z + m.w * py.w) / Mt;
  const float cz = red_sum(m.x * pz.x + m.y * pz.y + m.z * pz.z + m.w * pz.w) / Mt;
  float I = 0.f;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float dx = get(px, e) - cx, dy = get(py, e) - cy, dz = get(pz, e) - cz;
    I += get(m, e) * (dx * dx + dy * dy + dz * dz);
  }
  return InState{Mt, cx, cy, cz, red_sum(I)};
}

template <int LEVEL>
__global__ void __launch_bounds__(TH)
inertia_fused_kernel(const float* __restrict__ mass, const float* __restrict__ pos, int n,
                     float* __restrict__ center, float* __restrict__ inertia) {
  __shared__ InState red_s[NW];
  __shared__ float red_f[NW];
  const int n4 = n >> 2;
  const float4* mr = reinterpret_cast<const float4*>(mass + (size_t)blockIdx.x * n);
  const float4* xr = reinterpret_cast<const float4*>(pos + (size_t)blockIdx.x * 3 * n);
  const float4* yr = xr + n4;
  const float4* zr = yr + n4;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
  InState st{0.f, 0.f, 0.f, 0.f, 0.f};
  if (LEVEL == RF_FUSE_THREAD) {
    // weighted Welford, one point at a time: c += (m/M') d, I += m (1 - m/M') |d|^2
    for (int base = 0; base < n4; base += TH * 2) {
      float4 mv[2], xv[2], yv[2], zv[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int c = base + u * TH + (int)threadIdx.x;
        const bool ok = c < n4;
        mv[u] = ok && row_ok(c, n) ? __ldcs(mr + c) : zero;
        xv[u] = ok && row_ok(c, 3LL * n) ? __ldcs(xr + c) : zero;
        yv[u] = ok && row_ok(n4 + c, 3LL * n) ? __ldcs(yr + c) : zero;
        zv[u] = ok && row_ok(2 * n4 + c, 3LL * n) ? __ldcs(zr + c) : zero;
      }
#pragma unroll
      for (int u = 0; u < 2; ++u) {
      const float4 m = mv[u], px = xv[u], py = yv[u], pz = zv[u];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float me = get(m, e);
        const float Mn = st.M + me;
        if (Mn == 0.f) continue;
        const float f = __fdividef(me, Mn);
        const float dx = get(px, e) - st.cx, dy = get(py, e) - st.cy, dz = get(pz, e) - st.cz;
        st.cx += f * dx;
        st.cy += f * dy;
        st.cz += f * dz;
        st.I += me * (1.f - f) * (dx * dx + dy * dy + dz * dz);
        st.M = Mn;
      }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) st = in_shfl_merge(st, o);
    if (lane == 0) red_s[warp] = st;
    __syncthreads();
    st = red_s[0];
    for (int w = 1; w < NW; ++w) st = in_merge(st, red_s[w]);
  } else if (LEVEL == RF_FUSE_WARP) {
    for (int base0 = warp * 32; base0 < n4; base0 += TH * 2) {
      float4 mv[2], xv[2], yv[2], zv[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int c = base0 + u * TH + lane;
        const bool ok = c < n4;
        mv[u] = ok && row_ok(c, n) ? __ldcs(mr + c) : zero;
        xv[u] = ok && row_ok(c, 3LL * n) ? __ldcs(xr + c) : zero;
        yv[u] = ok && row_ok(n4 + c, 3LL * n) ? __ldcs(yr + c) : zero;
        zv[u] = ok && row_ok(2 * n4 + c, 3LL * n) ? __ldcs(zr + c) : zero;
      }
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        if (base0 + u * TH >= n4) break;        // uniform across the warp
        st = in_merge(st, in_tile<false>(mv[u], xv[u], yv[u], zv[u], red_f));
      }
    }
    if (lane == 0) red_s[warp] = st;
    __syncthreads();
    st = red_s[0];
    for (int w = 1; w < NW; ++w) st = in_merge(st, red_s[w]);
  } else {
    for (int base0 = 0; base0 < n4; base0 += TH * 2) {
      float4 mv[2], xv[2], yv[2], zv[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int c = base0 + u * TH + (int)threadIdx.x;
        const bool ok = c < n4;
        mv[u] = ok && row_ok(c, n) ? __ldcs(mr + c) : zero;
        xv[u] = ok && row_ok(c, 3LL * n) ? __ldcs(xr + c) : zero;
        yv[u] = ok && row_ok(n4 + c, 3LL * n) ? __ldcs(yr + c) : zero;
        zv[u] = ok && row_ok(2 * n4 + c, 3LL * n) ? __ldcs(zr + c) : zero;
      }
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        if (base0 + u * TH >= n4) break;        // uniform across the block
        st = in_merge(st, in_tile<true>(mv[u], xv[u], yv[u], zv[u], red_f));
      }
    }
  }
  if (threadIdx.x == 0) {
    center[blockIdx.x * 3 + 0] = st.cx;
    center[blockIdx.x * 3 + 1] = st.cy;
    center[blockIdx.x * 3 + 2] = st.cz;
    inertia[blockIdx.x] = st.I;
  }
}

// unfused: kernel 1 writes the centre of mass, kernel 2 re-reads the row
__global__ void __launch_bounds__(TH)
center_kernel(const float* __restrict__ mass, const float* __restrict__ pos, int n,
              float* __restrict__ center) {
  __shared__ float red[NW];
  const int n4 = n >> 2;
  const float4* mr = reinterpret_cast<const float4*>(mass + (size_t)blockIdx.x * n);
  const float4* xr = reinterpret_cast<const float4*>(pos + (size_t)blockIdx.x * 3 * n);
  float M = 0.f, sx = 0.f, sy = 0.f, sz = 0.f;
  for (int c = threadIdx.x; c < n4; c += TH) {
    if (!row_ok(c, n) || !row_ok(2 * n4 + c, 3LL * n)) continue;
    const float4 m = __ldcs(mr + c), px = __ldcs(xr + c), py = __ldcs(xr + n4 + c),
                 pz = __ldcs(xr + 2 * n4 + c);
    M += (m.x + m.y) + (m.z + m.w);
    sx += m.x * px.x + m.y * px.y + m.z * px.z + m.w * px.w;
    sy += m.x * py.x + m.y * py.y + m.z * py.z + m.w * py.w;
    sz += m.x * pz.x + m.y * pz.y + m.z * pz.z + m.w * pz.w;
  }
  M = bsum(M, red);
  sx = bsum(sx, red);
  sy = bsum(sy, red);
  sz = bsum(sz, red);
  if (threadIdx.x == 0) {
    center[blockIdx.x * 3 + 0] = sx / M;
    center[blockIdx.x * 3 + 1] = sy / M;
    center[blockIdx.x * 3 + 2] = sz / M;
  }
}

__global__ void __launch_bounds__(TH)
inertia_from_center_kernel(const float* __restrict__ mass, const float* __restrict__ pos, int n,
                           const float* __restrict__ center, float* __restrict__ inertia) {
  __shared__ float red[NW];
  const int n4 = n >> 2;
  const float4* mr = reinterpret_cast<const float4*>(mass + (size_t)blockIdx.x * n);
  const float4* xr = reinterpret_cast<const float4*>(pos + (size_t)blockIdx.x * 3 * n);
  const float cx = center[blockIdx.x * 3 + 0], cy = center[blockIdx.x * 3 + 1],
              cz = center[blockIdx.x * 3 + 2];
  float I = 0.f;
  for (int c = threadIdx.x; c < n4; c += TH) {
    if (!row_ok(c, n) || !row_ok(2 * n4 + c, 3LL * n)) continue;
    const float4 m = __ldcs(mr + c), px = __ldcs(xr + c), py = __ldcs(xr + n4 + c),
                 pz = __ldcs(xr + 2 * n4 + c);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float dx = get(px, e) - cx, dy = get(py, e) - cy, dz = get(pz, e) - cz;
      I += get(m, e) * (dx * dx + dy * dy + dz * dz);
    }
  }
  I = bsum(I, red);
  if (threadIdx.x == 0) inertia[blockIdx.x] = I;
}

// --------------------------------------------------- layer normalisation ----
// Fused: the row stays in registers; each thread reduces its values to
// (count, mean, M2) in two passes over registers, the states merge across the
// block, and the same registers are normalised and written.
template <int VPT>
__global__ void __launch_bounds__(TH)
layernorm_fused_kernel(const float* __restrict__ x, const float* __restrict__ gamma,
                       const float* __restrict__ beta, int n, float eps, float* __restrict__ y) {
  __shared__ VarState red_v[NW];
  const int n4 = n >> 2;
  const float4* xr = reinterpret_cast<const float4*>(x + (size_t)blockIdx.x * n);
  float4* yr = reinterpret_cast<float4*>(y + (size_t)blockIdx.x * n);
  float4 v[VPT];
  float cnt = 0.f, sum = 0.f;
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int c = i * TH + threadIdx.x;
    v[i] = c < n4 && row_ok(c, n) ? __ldcs(xr + c) : make_float4(0.f, 0.f, 0.f, 0.f);
    if (c < n4) {
      cnt += 4.f;
      sum += (v[i].x + v[i].y) + (v[i].z + v[i].w);
    }
  }
  VarState st{cnt, cnt > 0.f ? sum / cnt : 0.f, 0.f};
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    if (i * TH + (int)threadIdx.x < n4) {
      const float dx = v[i].x - st.mean, dy = v[i].y - st.mean, dz = v[i].z - st.mean,
                  dw = v[i].w - st.mean;
      st.m2 += (dx * dx + dy * dy) + (dz * dz + dw * dw);
    }
  }
  st = var_warp_merge(st);
  if ((threadIdx.x & 31) == 0) red_v[threadIdx.x >> 5] = st;
  __syncthreads();
  VarState r = red_v[0];
#pragma unroll
  for (int w = 1; w < NW; ++w) r = var_merge(r, red_v[w]);
  const float mu = r.mean, rstd = rsqrtf(r.m2 / (float)n + eps);
  const float4* g4 = reinterpret_cast<const float4*>(gamma);
  const float4* b4 = reinterpret_cast<const float4*>(beta);
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int c = i * TH + threadIdx.x;
    if (c < n4 && row_ok(c, n) && vec_ok(c, n)) {
      const float4 g = __ldg(g4 + c), b = __ldg(b4 + c);
      __stcs(yr + c, make_float4((v[i].x - mu) * rstd * g.x + b.x, (v[i].y - mu) * rstd * g.y + b.y,
                                 (v[i].z - mu) * rstd * g.z + b.z, (v[i].w - mu) * rstd * g.w + b.w));
    }
  }
}

// unfused: mean kernel, variance kernel (both re-read the row), then normalise
__global__ void __launch_bounds__(TH)
layernorm_apply_kernel(const float* __restrict__ x, const float* __restrict__ gamma,
                       const float* __restrict__ beta, int n, float eps, int R,
                       const float* __restrict__ work, float* __restrict__ y) {
  const float4* xr = reinterpret_cast<const float4*>(x + (size_t)blockIdx.x * n);
  float4* yr = reinterpret_cast<float4*>(y + (size_t)blockIdx.x * n);
  const float mu = work[blockIdx.x], rstd = rsqrtf(work[R + blockIdx.x] + eps);
  const float4* g4 = reinterpret_cast<const float4*>(gamma);
  const float4* b4 = reinterpret_cast<const float4*>(beta);
  for (int c = threadIdx.x; c < (n >> 2); c += TH) {
    if (!row_ok(c, n) || !vec_ok(c, n)) continue;
    const float4 v = __ldcs(xr + c), g = __ldg(g4 + c), b = __ldg(b4 + c);
    __stcs(yr + c, make_float4((v.x - mu) * rstd * g.x + b.x, (v.y - mu) * rstd * g.y + b.y,
                               (v.z - mu) * rstd * g.z + b.z, (v.w - mu) * rstd * g.w + b.w));
  }
}

// ---------------------------------------------------------- RMS norm ----
// fused: the row stays in registers (VPT float4 per thread); the sum of
// squares is reduced across the block, then the same registers are scaled
// by rsqrt(ms + eps) * gamma and written
template <int VPT>
__global__ void __launch_bounds__(TH)
rmsnorm_fused_kernel(const float* __restrict__ x, const float* __restrict__ gamma, int n, float eps,
                     float* __restrict__ y) {
  __shared__ float red[NW];
  const int n4 = n >> 2;
  const float4* xr = reinterpret_cast<const float4*>(x + (size_t)blockIdx.x * n);
  float4* yr = reinterpret_cast<float4*>(y + (size_t)blockIdx.x * n);
  float4 v[VPT];
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int c = i * TH + threadIdx.x;
    v[i] = c < n4 && row_ok(c, n) ? __ldcs(xr + c) : make_float4(0.f, 0.f, 0.f, 0.f);
    ss += (v[i].x * v[i].x + v[i].y * v[i].y) + (v[i].z * v[i].z + v[i].w * v[i].w);
  }
  const float rs = rsqrtf(bsum(ss, red) / (float)n + eps);
  const float4* g4 = reinterpret_cast<const float4*>(gamma);
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int c = i * TH + threadIdx.x;
    if (c < n4 && row_ok(c, n) && vec_ok(c, n)) {
      const float4 g = __ldg(g4 + c);
      __stcs(yr + c, make_float4(v[i].x * rs * g.x, v[i].y * rs * g.y, v[i].z * rs * g.z,
                                 v[i].w * rs * g.w));
    }
  }
}

// unfused: one kernel for the mean of squares, one that re-reads the row
__global__ void __launch_bounds__(TH)
meansq_kernel(const float* __restrict__ x, int n, float* __restrict__ ms_out) {
  __shared__ float red[NW];
  const float4* xr = reinterpret_cast<const float4*>(x + (size_t)blockIdx.x * n);
  float s = 0.f;
  for (int c = threadIdx.x; c < (n >> 2); c += TH) {
    if (!row_ok(c, n)) continue;
    const float4 v = __ldcs(xr + c);
    s += (v.x * v.x + v.y * v.y) + (v.z * v.z + v.w * v.w);
  }
  s = bsum(s, red);
  if (threadIdx.x == 0) ms_out[blockIdx.x] = s / (float)n;
}

__global__ void __launch_bounds__(TH)
rmsnorm_apply_kernel(const float* __restrict__ x, const float* __restrict__ gamma, int n, float eps,
                     const float* __restrict__ ms, float* __restrict__ y) {
  const float4* xr = reinterpret_cast<const float4*>(x + (size_t)blockIdx.x * n);
  float4* yr = reinterpret_cast<float4*>(y + (size_t)blockIdx.x * n);
  const float rs = rsqrtf(ms[blockIdx.x] + eps);
  const float4* g4 = reinterpret_cast<const float4*>(gamma);
  for (int c = threadIdx.x; c < (n >> 2); c += TH) {
    if (!row_ok(c, n) || !vec_ok(c, n)) continue;
    const float4 v = __ldcs(xr + c), g = __ldg(g4 + c);
    __stcs(yr + c, make_float4(v.x * rs * g.x, v.y * rs * g.y, v.z * rs * g.z, v.w * rs * g.w));
  }
}

template <int LEVEL>
void launch_softmax_level(const float* x, int R, int n, float* y, cudaStream_t st) {
  const int vpt = (n / 4 + TH - 1) / TH;
  if (vpt <= 1) softmax_fused_kernel<LEVEL, 1><<<R, TH, 0, st>>>(x, n, y);
  else if (vpt <= 2) softmax_fused_kernel<LEVEL, 2><<<R, TH, 0, st>>>(x, n, y);
  else if (vpt <= 4) softmax_fused_kernel<LEVEL, 4><<<R, TH, 0, st>>>(x, n, y);
  else softmax_fused_kernel<LEVEL, 8><<<R, TH, 0, st>>>(x, n, y);
}

}  // namespace

rf_status launch_row_softmax(const float* x, int R, int n, float* y, int level, float* work,
                             cudaStream_t st) {
  switch (level) {
    case RF_FUSE_NONE:
      softmax_max_kernel<<<R, TH, 0, st>>>(x, n, work);
      softmax_sum_kernel<<<R, TH, 0, st>>>(x, n, R, work);
      softmax_norm_kernel<<<R, TH, 0, st>>>(x, n, R, work, y);
      break;
    case RF_FUSE_THREAD: launch_softmax_level<RF_FUSE_THREAD>(x, R, n, y, st); break;
    case RF_FUSE_WARP: launch_softmax_level<RF_FUSE_WARP>(x, R, n, y, st); break;
    default: launch_softmax_level<RF_FUSE_BLOCK>(x, R, n, y, st); break;
  }
  return launch_status();
}

rf_status launch_layer_norm(const float* x, const float* gamma, const float* beta, int R, int n,
                            float eps, float* y, int level, float* work, cudaStream_t st) {
  if (level == RF_FUSE_NONE) {
    mean_kernel<<<R, TH, 0, st>>>(x, n, work);
    var_from_mean_kernel<<<R, TH, 0, st>>>(x, n, work, work + R);
    layernorm_apply_kernel<<<R, TH, 0, st>>>(x, gamma, beta, n, eps, R, work, y);
  } else {
    const int vpt = (n / 4 + TH - 1) / TH;
    if (vpt <= 1) layernorm_fused_kernel<1><<<R, TH, 0, st>>>(x, gamma, beta, n, eps, y);
    else if (vpt <= 2) layernorm_fused_kernel<2><<<R, TH, 0, st>>>(x, gamma, beta, n, eps, y);
    else if (vpt <= 4) layernorm_fused_kernel<4><<<R, TH, 0, st>>>(x, gamma, beta, n, eps, y);
    else layernorm_fused_kernel<8><<<R, TH, 0, st>>>(x, gamma, beta, n, eps, y);
  }
  return launch_status();
}

rf_status launch_rms_norm(const float* x, const float* gamma, int R, int n, float eps, float* y,
                          int level, float* work, cudaStream_t st) {
  if (level == RF_FUSE_NONE) {
    meansq_kernel<<<R, TH, 0, st>>>(x, n, work);
    rmsnorm_apply_kernel<<<R, TH, 0, st>>>(x, gamma, n, eps, work, y);
  } else {
    const int vpt = (n / 4 + TH - 1) / TH;
    if (vpt <= 1) rmsnorm_fused_kernel<1><<<R, TH, 0, st>>>(x, gamma, n, eps, y);
    else if (vpt <= 2) rmsnorm_fused_kernel<2><<<R, TH, 0, st>>>(x, gamma, n, eps, y);
    else if (vpt <= 4) rmsnorm_fused_kernel<4><<<R, TH, 0, st>>>(x, gamma, n, eps, y);
    else rmsnorm_fused_kernel<8><<<R, TH, 0, st>>>(x, gamma, n, eps, y);
  }
  return launch_status();
}

rf_status launch_row_variance(const float* x, int R, int n, float* mean, float* var, int level,
                              cudaStream_t st) {
  switch (level) {
    case RF_FUSE_NONE:
      mean_kernel<<<R, TH, 0, st>>>(x, n, mean);
      var_from_mean_kernel<<<R, TH, 0, st>>>(x, n, mean, var);
      break;
    case RF_FUSE_THREAD: variance_fused_kernel<RF_FUSE_THREAD><<<R, TH, 0, st>>>(x, n, mean, var); break;
    case RF_FUSE_WARP: variance_fused_kernel<RF_FUSE_WARP><<<R, TH, 0, st>>>(x, n, mean, var); break;
    default: variance_fused_kernel<RF_FUSE_BLOCK><<<R, TH, 0, st>>>(x, n, mean, var); break;
  }
  return launch_status();
}

rf_status launch_moment_of_inertia(const float* mass, const float* pos, int R, int n,
                                   float* center, float* inertia, int level, cudaStream_t st) {
  switch (level) {
    case RF_FUSE_NONE:
      center_kernel<<<R, TH, 0, st>>>(mass, pos, n, center);
      inertia_from_center_kernel<<<R, TH, 0, st>>>(mass, pos, n, center, inertia);
      break;
    case RF_FUSE_THREAD:
      inertia_fused_kernel<RF_FUSE_THREAD><<<R, TH, 0, st>>>(mass, pos, n, center, inertia);
      break;
    case RF_FUSE_WARP:
      inertia_fused_kernel<RF_FUSE_WARP><<<R, TH, 0, st>>>(mass, pos, n, center, inertia);
      break;
    default:
      inertia_fused_kernel<RF_FUSE_BLOCK><<<R, TH, 0, st>>>(mass, pos, n, center, inertia);
      break;
  }
  return launch_status();
}

RF_BOUNDS_WORD_OF_THIS_FILE

}  // namespace rf
