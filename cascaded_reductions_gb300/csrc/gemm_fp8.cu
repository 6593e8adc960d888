// FP8 GEMM with per-row x per-column scale epilogue (phase 2 of the abs-max ->
// quantise -> GEMM cascade).  Placeholder until the tcgen05 kernel lands.
#include "common.cuh"

namespace rf {

rf_status launch_fp8_gemm(const uint8_t*, const float*, const uint8_t*, const float*, int, int,
                          int, void*, cudaStream_t) {
  return RF_ERR_UNSUPPORTED;
}

}  // namespace rf
