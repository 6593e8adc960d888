// Causal prefill attention.  Placeholder until the tcgen05 kernel lands.
#include "common.cuh"

namespace rf {

rf_status launch_prefill(const void*, const void*, const void*, int, int, int, int, int, float,
                         void*, float*, cudaStream_t) {
  return RF_ERR_UNSUPPORTED;
}

rf_status prefill_take_status(int* status) {
  *status = RF_OK;
  return RF_OK;
}

}  // namespace rf
