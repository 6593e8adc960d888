// Host helpers of the tensor-core kernels: TMA descriptor encoding, SM count,
// and the read-back of the bounded-wait status words.
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

#include "tc_common.cuh"

namespace rf {
namespace tc {

namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
}  // namespace

bool make_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t inner,
                  uint64_t outer, uint64_t row_stride_bytes, uint32_t box_inner,
                  uint32_t box_outer, CUtensorMapSwizzle swizzle) {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (g_encode == nullptr) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_stride_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t elem_strides[2] = {1, 1};
  return g_encode(map, dtype, 2, const_cast<void*>(base), dims, strides, box, elem_strides,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

}  // namespace tc

#ifdef RF_CHECK_BOUNDS
namespace {
// Filled during static initialisation of the library (one entry per kernel
// file); zero-initialised storage, so registration order does not matter.
constexpr int kMaxBoundsWords = 32;
bounds_take_fn g_bounds_words[kMaxBoundsWords];
std::atomic<int> g_n_bounds_words{0};
}  // namespace

bool register_bounds_word(bounds_take_fn take) {
  const int i = g_n_bounds_words.fetch_add(1);
  if (i < kMaxBoundsWords) g_bounds_words[i] = take;
  return i < kMaxBoundsWords;
}
#endif

rf_status take_bounds_words(int* status) {
  *status = RF_OK;
#ifdef RF_CHECK_BOUNDS
  const int n = g_n_bounds_words.load() < kMaxBoundsWords ? g_n_bounds_words.load() : kMaxBoundsWords;
  for (int i = 0; i < n; ++i) {
    int w = RF_OK;
    if (g_bounds_words[i](&w) != RF_OK) return RF_ERR_CUDA;
    if (w != RF_OK && *status == RF_OK) *status = w;
  }
#endif
  return RF_OK;
}

rf_status read_device_error(int* status, cudaStream_t st) {
  if (cudaStreamSynchronize(st) != cudaSuccess) return RF_ERR_CUDA;
  int st_words[6] = {0, 0, 0, 0, 0, 0};
  if (gemm_take_status(&st_words[0]) != RF_OK || prefill_take_status(&st_words[1]) != RF_OK ||
      fp8_incremental_take_status(&st_words[2]) != RF_OK || mla_take_status(&st_words[3]) != RF_OK ||
      selftest_take_status(&st_words[4]) != RF_OK || take_bounds_words(&st_words[5]) != RF_OK)
    return RF_ERR_CUDA;
  *status = RF_OK;
  for (int w : st_words)
    if (w != RF_OK) {
      *status = w;
      break;
    }
  return RF_OK;
}

}  // namespace rf
