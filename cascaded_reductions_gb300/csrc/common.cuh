// Shared device helpers and internal launcher declarations for librf.so.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "rf.h"

namespace rf {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// ---------------------------------------------------------------- loads ----
// 16-byte streaming load through the non-coherent path; not kept in L1 (every
// byte is read once), with a 256-byte L2 prefetch hint for the sequential
// stream that follows.
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// bf16 pair packed in a 32-bit word -> two floats (exact widening).
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two floats -> bf16 pair, round to nearest even (hardware cvt).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

template <int WIDTH>
__device__ __forceinline__ float group_max(float x) {
#pragma unroll
  for (int o = WIDTH / 2; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

template <int WIDTH>
__device__ __forceinline__ float group_sum(float x) {
#pragma unroll
  for (int o = WIDTH / 2; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// A 16-byte chunk of a key/value row as floats: 4 fp32 or 8 bf16 values.
template <typename T>
struct Chunk;

template <>
struct Chunk<float> {
  static constexpr int N = 4;
  __device__ __forceinline__ static void unpack(const uint4& u, float* f) {
    f[0] = __uint_as_float(u.x);
    f[1] = __uint_as_float(u.y);
    f[2] = __uint_as_float(u.z);
    f[3] = __uint_as_float(u.w);
  }
};

struct Bf16Tag {};
template <>
struct Chunk<Bf16Tag> {
  static constexpr int N = 8;
  __device__ __forceinline__ static void unpack(const uint4& u, float* f) {
    f[0] = bf16_lo(u.x); f[1] = bf16_hi(u.x);
    f[2] = bf16_lo(u.y); f[3] = bf16_hi(u.y);
    f[4] = bf16_lo(u.z); f[5] = bf16_hi(u.z);
    f[6] = bf16_lo(u.w); f[7] = bf16_hi(u.w);
  }
};

// Rescale reference for a running max that may still be -inf (no key seen):
// exp2(x - ref) is then 0 for x = -inf and the state stays the identity.
__device__ __forceinline__ float ref_of(float m) { return m == -INFINITY ? 0.f : m; }

// -------------------------------------------------------- status words ----
// A translation unit that owns a device status word (the bounded-wait word of
// the tensor-core files, the index-check word of the bounds-checked build)
// registers a reader of it when the library loads; read_device_error calls
// every registered reader, each of which reads and clears its word.
using status_take_fn = rf_status (*)(int*);
bool register_status_word(status_take_fn take);
#define RF_STATUS_WORD_READER(fn, word)                                                     \
  namespace {                                                                               \
  rf_status fn(int* status) {                                                               \
    int v = 0, zero = 0;                                                                    \
    if (cudaMemcpyFromSymbol(&v, word, sizeof(int)) != cudaSuccess) return RF_ERR_CUDA;     \
    if (cudaMemcpyToSymbol(word, &zero, sizeof(int)) != cudaSuccess) return RF_ERR_CUDA;    \
    *status = v;                                                                            \
    return RF_OK;                                                                           \
  }                                                                                         \
  const bool fn##_registered = register_status_word(&fn);                                   \
  }

// ------------------------------------------------------- bounds checks ----
// Built with -DRF_CHECK_BOUNDS, every kernel checks each global load and
// store against the extent of its buffer, computed in the kernel from the
// call's size arguments (never from the pointer it is checking).  A refused
// index skips its access (a load yields zeros) and records RF_ERR_BOUNDS in
// this translation unit's device word, which the file registers with
// RF_BOUNDS_WORD_OF_THIS_FILE.  Without the flag RF_SPAN_OK is the constant
// true and the checks compile to nothing.
#ifdef RF_CHECK_BOUNDS
static __device__ int g_bounds_status;
// elements [i, i + w) of a buffer of n elements
__device__ __forceinline__ bool span_ok(long long i, long long w, long long n) {
  if (i >= 0 && i + w <= n) return true;
  atomicExch(&g_bounds_status, (int)RF_ERR_BOUNDS);
  return false;
}
#define RF_SPAN_OK(i, w, n) ::rf::span_ok((long long)(i), (long long)(w), (long long)(n))
#define RF_BOUNDS_WORD_OF_THIS_FILE RF_STATUS_WORD_READER(take_bounds_word, g_bounds_status)
#else
#define RF_SPAN_OK(i, w, n) true
#define RF_BOUNDS_WORD_OF_THIS_FILE
#endif
#define RF_IDX_OK(i, n) RF_SPAN_OK(i, 1, n)

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Opt a kernel into `bytes` of dynamic shared memory on the current device,
// once per device: the attribute belongs to the device's context, so each
// kernel keeps one flag bit per device (up to 64), set atomically.
template <typename Kernel>
inline rf_status smem_attr(Kernel kern, size_t bytes, std::atomic<uint64_t>& done) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return RF_ERR_CUDA;
  const uint64_t bit = dev < 64 ? (1ull << dev) : 0ull;
  if (bit != 0 && (done.load(std::memory_order_acquire) & bit)) return RF_OK;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) !=
      cudaSuccess)
    return RF_ERR_CUDA;
  done.fetch_or(bit, std::memory_order_release);
  return RF_OK;
}

inline rf_status launch_status() {
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? RF_OK : RF_ERR_CUDA;
}

// ------------------------------------------------------------ launchers ----
// Each returns RF_OK or RF_ERR_CUDA; arguments were validated by the C ABI.
rf_status launch_decode_split(const void* q, const void* k, const void* v, int R, int L, int D,
                              int S, float scale, int dtype, float* seg_m, float* seg_l,
                              float* seg_acc, cudaStream_t st);
rf_status launch_decode_fused(const void* q, const void* k, const void* v, int R, int L, int D,
                              int S, float scale, int dtype, float* seg_m, float* seg_l,
                              float* seg_acc, int* counters, void* out, int out_dtype, float* lse,
                              cudaStream_t st);
rf_status launch_decode_twopass(const void* q, const void* k, const void* v, int R, int L, int D,
                                int S, float scale, int dtype, float* seg_m, float* seg_l,
                                float* seg_acc, cudaStream_t st);
rf_status launch_state_merge(const float* seg_m, const float* seg_l, const float* seg_acc, int R,
                             int S, int D, void* out, int out_dtype, float* lse, cudaStream_t st);
rf_status launch_softmax_topk(const float* logits, int T, int E, int k, int renormalize,
                              int32_t* idx, float* w, cudaStream_t st);
rf_status launch_absmax_quant(const void* x, int M, int K, uint8_t* xq, float* sx,
                              cudaStream_t st);
rf_status launch_fp8_gemm_2sm(const uint8_t* xq, const float* sx, const uint8_t* wq,
                              const float* sw, int M, int N, int K, void* y, cudaStream_t st);
rf_status launch_fp8_gemm(const uint8_t* xq, const float* sx, const uint8_t* wq, const float* sw,
                          int M, int N, int K, void* y, cudaStream_t st);
rf_status launch_prefill(const void* q, const void* k, const void* v, int B, int H, int N, int D,
                         int causal, float scale, void* out, float* lse, cudaStream_t st);
rf_status launch_row_softmax(const float* x, int R, int n, float* y, int level, float* work,
                             cudaStream_t st);
rf_status launch_row_variance(const float* x, int R, int n, float* mean, float* var, int level,
                              cudaStream_t st);
rf_status launch_moment_of_inertia(const float* mass, const float* pos, int R, int n,
                                   float* center, float* inertia, int level, cudaStream_t st);
rf_status launch_layer_norm(const float* x, const float* gamma, const float* beta, int R, int n,
                            float eps, float* y, int level, float* work, cudaStream_t st);
rf_status launch_fp8_incremental(const void* x, const uint8_t* wq, const float* sw, int M, int N,
                                 int K, void* y, float* sx_final, cudaStream_t st);
rf_status launch_fp8_incremental_cluster(const void* x, const uint8_t* wq, const float* sw, int M,
                                         int N, int K, void* y, float* sx_final, cudaStream_t st);
rf_status launch_rms_norm(const float* x, const float* gamma, int R, int n, float eps, float* y,
                          int level, float* work, cudaStream_t st);
rf_status launch_mla_decode(const void* q, const void* c, int B, int H, int L, int S, float scale,
                            float* seg_m, float* seg_l, float* seg_acc, cudaStream_t st);
rf_status launch_stream_read(const void* x, size_t nbytes, uint32_t* out_xor, cudaStream_t st);
rf_status launch_selftest_wait_timeout(int* waited_ms, cudaStream_t st);
rf_status launch_selftest_bounds(cudaStream_t st);
rf_status read_device_error(int* status, cudaStream_t st);

}  // namespace rf
