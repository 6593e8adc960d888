// Host helpers: TMA descriptor encoding and SM count for the tensor-core
// kernels, and the registry and read-back of every device status word.
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

namespace {
// Filled during static initialisation of the library (one entry per status
// word); zero-initialised storage, so registration order does not matter.
constexpr int kMaxStatusWords = 32;
status_take_fn g_status_words[kMaxStatusWords];
std::atomic<int> g_n_status_words{0};
}  // namespace

bool register_status_word(status_take_fn take) {
  const int i = g_n_status_words.fetch_add(1);
  if (i < kMaxStatusWords) g_status_words[i] = take;
  return i < kMaxStatusWords;
}

rf_status read_device_error(int* status, cudaStream_t st) {
  if (cudaStreamSynchronize(st) != cudaSuccess) return RF_ERR_CUDA;
  *status = RF_OK;
  const int n = g_n_status_words.load() < kMaxStatusWords ? g_n_status_words.load() : kMaxStatusWords;
  for (int i = 0; i < n; ++i) {
    int w = RF_OK;
    if (g_status_words[i](&w) != RF_OK) return RF_ERR_CUDA;
    if (w != RF_OK && *status == RF_OK) *status = w;      // every word is read and cleared
  }
  return RF_OK;
}

}  // namespace rf
