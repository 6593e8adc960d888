// rf_attn_decode_noalloc: split-KV decode attention for callers that cannot
// allocate device memory.
//
// The regular path needs a scratch buffer for the per-segment states that
// rf_attn_decode_split writes and rf_state_merge reads, and expects the caller
// to provide it.  Some callers cannot: a plugin running inside a host engine
// that owns every device allocation and exposes no allocator to it, a
// latency-critical serving loop where cudaMalloc's implicit device-wide
// synchronisation is not acceptable, or a process whose device memory budget
// was fixed at start-up.  This entry point keeps the segment states in a
// fixed array that is part of the library image instead, so the call itself
// allocates nothing.  Every accepted call is one launch: the split kernel with
// the merge done by each row's last CTA (as rf_attn_decode_fused), counting in
// a second fixed array of per-row counters that every completed call leaves
// at zero.  The size of the state array caps the rows at kNoallocMaxRows (a
// static_assert below), so no accepted call needs more counters than that.
//
// Costs and rules of the shared array:
//   * it is kRfNoallocScratchBytes (16 MiB) on every GPU that loads the
//     library, held until the process exits;
//   * every call on a device uses the same array, so calls that may overlap
//     on the GPU (different streams, or host threads without ordering) race
//     and corrupt each other's result; order them on one stream;
//   * the decode kernel writes every segment state it later merges (empty
//     segments included), so nothing left by an earlier call is read and
//     nothing needs clearing.
// The device address of the array is looked up once per device, on the first
// call made while that device is current (cudaGetSymbolAddress); make that
// first call before any stream capture that includes this entry point.

#include <math.h>

#include <mutex>

#include "common.cuh"

namespace rf {
namespace {

constexpr size_t kRfNoallocScratchBytes = 16u << 20;
constexpr int kNoallocMaxRows = 65536;
constexpr int kMaxDevices = 64;

// The smallest request for R rows (S = 1, D = 64) needs 4*R*64 bytes of
// accumulator states, so R rows above kNoallocMaxRows never fit: the size
// check alone keeps every accepted call within the counters array.
static_assert((size_t)(kNoallocMaxRows + 1) * 64 * sizeof(float) > kRfNoallocScratchBytes,
              "the state array must cap the rows at kNoallocMaxRows");

static __device__ __align__(256) unsigned char g_noalloc_scratch[kRfNoallocScratchBytes];
// per-row counters of the one-launch merge: zero when the library loads, and
// every completed call leaves them zero
static __device__ __align__(256) int g_noalloc_counters[kNoallocMaxRows];

std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices] = {nullptr};
int* g_counters_addr[kMaxDevices] = {nullptr};

// Device addresses of the two arrays on the current device (set-up on first use).
rf_status scratch_address(void** out, int** counters) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return RF_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    void* c = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr ||
        cudaGetSymbolAddress(&c, g_noalloc_counters) != cudaSuccess || c == nullptr)
      return RF_ERR_CUDA;
    g_scratch_addr[dev] = p;
    g_counters_addr[dev] = static_cast<int*>(c);
  }
  *out = g_scratch_addr[dev];
  *counters = g_counters_addr[dev];
  return RF_OK;
}

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace
}  // namespace rf

extern "C" rf_status rf_attn_decode_noalloc(const void* q, const void* k, const void* v, int R,
                                            int L, int D, int S, float scale, int dtype,
                                            void* out, int out_dtype, float* lse, void* stream) {
  if (!q || !k || !v || !out) return RF_ERR_INVALID_ARG;
  if (R <= 0 || L <= 0 || D <= 0 || S < 1 || !isfinite(scale)) return RF_ERR_INVALID_ARG;
  if (dtype != RF_F32 && dtype != RF_BF16) return RF_ERR_INVALID_ARG;
  if (out_dtype != RF_F32 && out_dtype != RF_BF16) return RF_ERR_INVALID_ARG;
  if (!((dtype == RF_F32 && D == 64) || (dtype == RF_BF16 && D == 128))) return RF_ERR_UNSUPPORTED;
  // scratch layout: seg_m [R*S] | seg_l [R*S] | seg_acc [R*S*D], seg_acc 256-byte aligned
  const size_t states = (size_t)R * (size_t)S;
  const size_t acc_off = rf::align_up(2 * states * sizeof(float), 256);
  const size_t need = acc_off + states * (size_t)D * sizeof(float);
  if (states > 0x7fffffffu || need > rf::kRfNoallocScratchBytes) return RF_ERR_UNSUPPORTED;
  if (!rf::aligned16(q) || !rf::aligned16(k) || !rf::aligned16(v) || !rf::aligned16(out))
    return RF_ERR_MISALIGNED;
  void* base = nullptr;
  int* counters = nullptr;
  rf_status s = rf::scratch_address(&base, &counters);
  if (s != RF_OK) return s;
  float* seg_m = static_cast<float*>(base);
  float* seg_l = seg_m + states;
  float* seg_acc = reinterpret_cast<float*>(static_cast<unsigned char*>(base) + acc_off);
  // R <= kNoallocMaxRows here: the size check above implies it (static_assert)
  return rf::launch_decode_fused(q, k, v, R, L, D, S, scale, dtype, seg_m, seg_l, seg_acc,
                                 counters, out, out_dtype, lse, static_cast<cudaStream_t>(stream));
}
