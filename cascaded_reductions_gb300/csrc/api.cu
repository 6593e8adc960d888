// C ABI of librf.so: argument validation, then one launch per kernel.
// Every check happens on the host before anything is enqueued.

#include <math.h>

#include "common.cuh"

namespace {

inline cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

}  // namespace

extern "C" {

const char* rf_status_string(int status) {
  switch (status) {
    case RF_OK: return "RF_OK";
    case RF_ERR_INVALID_ARG: return "RF_ERR_INVALID_ARG";
    case RF_ERR_UNSUPPORTED: return "RF_ERR_UNSUPPORTED";
    case RF_ERR_MISALIGNED: return "RF_ERR_MISALIGNED";
    case RF_ERR_CUDA: return "RF_ERR_CUDA";
    case RF_ERR_TIMEOUT: return "RF_ERR_TIMEOUT";
    case RF_ERR_BOUNDS: return "RF_ERR_BOUNDS";
    default: return "RF_ERR_UNKNOWN";
  }
}

int rf_version(void) { return 10000; }

rf_status rf_attn_decode_split(const void* q, const void* k, const void* v, int R, int L, int D,
                               int S, float scale, int dtype, float* seg_m, float* seg_l,
                               float* seg_acc, void* stream) {
  if (!q || !k || !v || !seg_m || !seg_l || !seg_acc) return RF_ERR_INVALID_ARG;
  if (R <= 0 || L <= 0 || D <= 0 || S < 1 || !isfinite(scale)) return RF_ERR_INVALID_ARG;
  if (dtype != RF_F32 && dtype != RF_BF16) return RF_ERR_INVALID_ARG;
  if (!((dtype == RF_F32 && D == 64) || (dtype == RF_BF16 && D == 128))) return RF_ERR_UNSUPPORTED;
  if ((long long)R * S > 0x7fffffffLL) return RF_ERR_UNSUPPORTED;
  if (!rf::aligned16(q) || !rf::aligned16(k) || !rf::aligned16(v) || !rf::aligned16(seg_acc))
    return RF_ERR_MISALIGNED;
  return rf::launch_decode_split(q, k, v, R, L, D, S, scale, dtype, seg_m, seg_l, seg_acc,
                                 as_stream(stream));
}

rf_status rf_attn_decode_fused(const void* q, const void* k, const void* v, int R, int L, int D,
                               int S, float scale, int dtype, float* seg_m, float* seg_l,
                               float* seg_acc, int* counters, void* out, int out_dtype,
                               float* lse, void* stream) {
  if (!q || !k || !v || !seg_m || !seg_l || !seg_acc || !counters || !out)
    return RF_ERR_INVALID_ARG;
  if (R <= 0 || L <= 0 || D <= 0 || S < 1 || !isfinite(scale)) return RF_ERR_INVALID_ARG;
  if (dtype != RF_F32 && dtype != RF_BF16) return RF_ERR_INVALID_ARG;
  if (out_dtype != RF_F32 && out_dtype != RF_BF16) return RF_ERR_INVALID_ARG;
  if (!((dtype == RF_F32 && D == 64) || (dtype == RF_BF16 && D == 128))) return RF_ERR_UNSUPPORTED;
  if ((long long)R * S > 0x7fffffffLL) return RF_ERR_UNSUPPORTED;
  if (!rf::aligned16(q) || !rf::aligned16(k) || !rf::aligned16(v) || !rf::aligned16(seg_acc) ||
      !rf::aligned16(out) || !rf::aligned16(counters))
    return RF_ERR_MISALIGNED;
  return rf::launch_decode_fused(q, k, v, R, L, D, S, scale, dtype, seg_m, seg_l, seg_acc,
                                 counters, out, out_dtype, lse, as_stream(stream));
}

rf_status rf_attn_decode_split_twopass(const void* q, const void* k, const void* v, int R, int L,
                                       int D, int S, float scale, int dtype, float* seg_m,
                                       float* seg_l, float* seg_acc, void* stream) {
  if (!q || !k || !v || !seg_m || !seg_l || !seg_acc) return RF_ERR_INVALID_ARG;
  if (R <= 0 || L <= 0 || D <= 0 || S < 1 || !isfinite(scale)) return RF_ERR_INVALID_ARG;
  if (dtype != RF_F32 && dtype != RF_BF16) return RF_ERR_INVALID_ARG;
  if (!((dtype == RF_F32 && D == 64) || (dtype == RF_BF16 && D == 128))) return RF_ERR_UNSUPPORTED;
  if ((long long)R * S > 0x7fffffffLL) return RF_ERR_UNSUPPORTED;
  if (!rf::aligned16(q) || !rf::aligned16(k) || !rf::aligned16(v) || !rf::aligned16(seg_acc))
    return RF_ERR_MISALIGNED;
  return rf::launch_decode_twopass(q, k, v, R, L, D, S, scale, dtype, seg_m, seg_l, seg_acc,
                                   as_stream(stream));
}

rf_status rf_state_merge(const float* seg_m, const float* seg_l, const float* seg_acc, int R,
                         int S, int D, void* out, int out_dtype, float* lse, void* stream) {
  if (!seg_m || !seg_l || !seg_acc || !out) return RF_ERR_INVALID_ARG;
  if (R <= 0 || S <= 0 || D <= 0) return RF_ERR_INVALID_ARG;
  if (out_dtype != RF_F32 && out_dtype != RF_BF16) return RF_ERR_INVALID_ARG;
  if (D != 64 && D != 128 && D != 512) return RF_ERR_UNSUPPORTED;
  if (!rf::aligned16(seg_acc) || !rf::aligned16(out)) return RF_ERR_MISALIGNED;
  return rf::launch_state_merge(seg_m, seg_l, seg_acc, R, S, D, out, out_dtype, lse,
                                as_stream(stream));
}

rf_status rf_mla_decode_split(const void* q, const void* c, int B, int H, int L, int Dk,
                              int Dv, int S, float scale, float* seg_m, float* seg_l,
                              float* seg_acc, void* stream) {
  if (!q || !c || !seg_m || !seg_l || !seg_acc) return RF_ERR_INVALID_ARG;
  if (B <= 0 || H <= 0 || L <= 0 || S < 1 || !isfinite(scale)) return RF_ERR_INVALID_ARG;
  if (Dk != 576 || Dv != 512 || H % 16 != 0) return RF_ERR_UNSUPPORTED;
  if ((long long)B * L >= (1ll << 31) || (long long)B * H >= (1ll << 31)) return RF_ERR_UNSUPPORTED;
  if (!rf::aligned16(q) || !rf::aligned16(c) || !rf::aligned16(seg_acc)) return RF_ERR_MISALIGNED;
  return rf::launch_mla_decode(q, c, B, H, L, S, scale, seg_m, seg_l, seg_acc, as_stream(stream));
}

rf_status rf_attn_prefill(const void* q, const void* k, const void* v, int B, int H, int N, int D,
                          int causal, float scale, void* out, float* lse, void* stream) {
  if (!q || !k || !v || !out) return RF_ERR_INVALID_ARG;
  if (B <= 0 || H <= 0 || N <= 0 || D <= 0 || !isfinite(scale)) return RF_ERR_INVALID_ARG;
  if (D != 128) return RF_ERR_UNSUPPORTED;
  if ((long long)B * H * N >= (1ll << 31)) return RF_ERR_UNSUPPORTED;
  if (!rf::aligned16(q) || !rf::aligned16(k) || !rf::aligned16(v) || !rf::aligned16(out))
    return RF_ERR_MISALIGNED;
  return rf::launch_prefill(q, k, v, B, H, N, D, causal ? 1 : 0, scale, out, lse,
                            as_stream(stream));
}

rf_status rf_softmax_topk(const float* logits, int T, int E, int k, int renormalize, int32_t* idx,
                          float* w, void* stream) {
  if (!logits || !idx || !w) return RF_ERR_INVALID_ARG;
  if (T <= 0 || E <= 0 || k < 1 || k > E) return RF_ERR_INVALID_ARG;
  if (E > 1024 || k > 32) return RF_ERR_UNSUPPORTED;
  if (!rf::aligned16(logits) || !rf::aligned16(idx) || !rf::aligned16(w)) return RF_ERR_MISALIGNED;
  return rf::launch_softmax_topk(logits, T, E, k, renormalize ? 1 : 0, idx, w, as_stream(stream));
}

rf_status rf_absmax_quant_e4m3(const void* x, int M, int K, uint8_t* xq, float* sx,
                               void* stream) {
  if (!x || !xq || !sx) return RF_ERR_INVALID_ARG;
  if (M <= 0 || K <= 0) return RF_ERR_INVALID_ARG;
  if (K % 8 != 0) return RF_ERR_UNSUPPORTED;
  if (!rf::aligned16(x) || !rf::aligned16(xq)) return RF_ERR_MISALIGNED;
  return rf::launch_absmax_quant(x, M, K, xq, sx, as_stream(stream));
}

static rf_status check_gemm_shape(int M, int N, int K) {
  if (M <= 0 || N <= 0 || K <= 0) return RF_ERR_INVALID_ARG;
  if (K % 16 != 0 || K > 65536) return RF_ERR_UNSUPPORTED;
  return RF_OK;
}

rf_status rf_fp8_gemm_scaled(const uint8_t* xq, const float* sx, const uint8_t* wq,
                             const float* sw, int M, int N, int K, void* y, void* stream) {
  if (!xq || !sx || !wq || !sw || !y) return RF_ERR_INVALID_ARG;
  rf_status s = check_gemm_shape(M, N, K);
  if (s != RF_OK) return s;
  if (!rf::aligned16(xq) || !rf::aligned16(wq) || !rf::aligned16(y) || !rf::aligned16(sw))
    return RF_ERR_MISALIGNED;
  return rf::launch_fp8_gemm(xq, sx, wq, sw, M, N, K, y, as_stream(stream));
}

rf_status rf_absmax_quant_fp8_gemm(const void* x, int M, int K, const uint8_t* wq, const float* sw,
                                   int N, uint8_t* xq, float* sx, void* y, void* stream) {
  if (!x || !wq || !sw || !xq || !sx || !y) return RF_ERR_INVALID_ARG;
  rf_status s = check_gemm_shape(M, N, K);
  if (s != RF_OK) return s;
  if (!rf::aligned16(x) || !rf::aligned16(wq) || !rf::aligned16(xq) || !rf::aligned16(y) ||
      !rf::aligned16(sw))
    return RF_ERR_MISALIGNED;
  s = rf::launch_absmax_quant(x, M, K, xq, sx, as_stream(stream));
  if (s != RF_OK) return s;
  return rf::launch_fp8_gemm(xq, sx, wq, sw, M, N, K, y, as_stream(stream));
}

static rf_status check_row_args(int R, int n, int level) {
  if (R <= 0 || n <= 0) return RF_ERR_INVALID_ARG;
  if (level < RF_FUSE_NONE || level > RF_FUSE_BLOCK) return RF_ERR_INVALID_ARG;
  if (n % 4 != 0) return RF_ERR_UNSUPPORTED;
  return RF_OK;
}

rf_status rf_row_softmax(const float* x, int R, int n, float* y, int level, float* work,
                         void* stream) {
  if (!x || !y) return RF_ERR_INVALID_ARG;
  rf_status s = check_row_args(R, n, level);
  if (s != RF_OK) return s;
  if (level == RF_FUSE_NONE && !work) return RF_ERR_INVALID_ARG;
  if (level != RF_FUSE_NONE && n > 8192) return RF_ERR_UNSUPPORTED;
  if (!rf::aligned16(x) || !rf::aligned16(y)) return RF_ERR_MISALIGNED;
  return rf::launch_row_softmax(x, R, n, y, level, work, as_stream(stream));
}

rf_status rf_row_variance(const float* x, int R, int n, float* mean, float* var, int level,
                          void* stream) {
  if (!x || !mean || !var) return RF_ERR_INVALID_ARG;
  rf_status s = check_row_args(R, n, level);
  if (s != RF_OK) return s;
  if (!rf::aligned16(x)) return RF_ERR_MISALIGNED;
  return rf::launch_row_variance(x, R, n, mean, var, level, as_stream(stream));
}

rf_status rf_moment_of_inertia(const float* mass, const float* pos, int R, int n, float* center,
                               float* inertia, int level, void* stream) {
  if (!mass || !pos || !center || !inertia) return RF_ERR_INVALID_ARG;
  rf_status s = check_row_args(R, n, level);
  if (s != RF_OK) return s;
  if (!rf::aligned16(mass) || !rf::aligned16(pos)) return RF_ERR_MISALIGNED;
  return rf::launch_moment_of_inertia(mass, pos, R, n, center, inertia, level, as_stream(stream));
}

rf_status rf_layer_norm(const float* x, const float* gamma, const float* beta, int R, int n,
                        float eps, float* y, int level, float* work, void* stream) {
  if (!x || !gamma || !beta || !y) return RF_ERR_INVALID_ARG;
  rf_status s = check_row_args(R, n, level);
  if (s != RF_OK) return s;
  if (!(eps >= 0.f) || !isfinite(eps)) return RF_ERR_INVALID_ARG;
  if (level == RF_FUSE_NONE && !work) return RF_ERR_INVALID_ARG;
  if (level != RF_FUSE_NONE && n > 8192) return RF_ERR_UNSUPPORTED;
  if (!rf::aligned16(x) || !rf::aligned16(y) || !rf::aligned16(gamma) || !rf::aligned16(beta))
    return RF_ERR_MISALIGNED;
  return rf::launch_layer_norm(x, gamma, beta, R, n, eps, y, level, work, as_stream(stream));
}

rf_status rf_rms_norm(const float* x, const float* gamma, int R, int n, float eps, float* y,
                      int level, float* work, void* stream) {
  if (!x || !gamma || !y) return RF_ERR_INVALID_ARG;
  rf_status s = check_row_args(R, n, level);
  if (s != RF_OK) return s;
  if (!(eps >= 0.f) || !isfinite(eps)) return RF_ERR_INVALID_ARG;
  if (level == RF_FUSE_NONE && !work) return RF_ERR_INVALID_ARG;
  if (level != RF_FUSE_NONE && n > 8192) return RF_ERR_UNSUPPORTED;
  if (!rf::aligned16(x) || !rf::aligned16(y) || !rf::aligned16(gamma)) return RF_ERR_MISALIGNED;
  return rf::launch_rms_norm(x, gamma, R, n, eps, y, level, work, as_stream(stream));
}

rf_status rf_incremental_quant_fp8_gemm(const void* x, int M, int K, const uint8_t* wq,
                                        const float* sw, int N, void* y, float* sx_final,
                                        void* stream) {
  if (!x || !wq || !sw || !y) return RF_ERR_INVALID_ARG;
  if (M <= 0 || N <= 0 || K <= 0) return RF_ERR_INVALID_ARG;
  if (M % 128 != 0 || N % 512 != 0 || K % 128 != 0) return RF_ERR_UNSUPPORTED;
  if (!rf::aligned16(x) || !rf::aligned16(wq) || !rf::aligned16(y) || !rf::aligned16(sw))
    return RF_ERR_MISALIGNED;
  // clusters of 8 (or 4) CTAs share the quantisation where N allows it
  const rf_status s =
      rf::launch_fp8_incremental_cluster(x, wq, sw, M, N, K, y, sx_final, as_stream(stream));
  if (s != RF_ERR_UNSUPPORTED) return s;
  return rf::launch_fp8_incremental(x, wq, sw, M, N, K, y, sx_final, as_stream(stream));
}

rf_status rf_device_error(int* status, void* stream) {
  if (!status) return RF_ERR_INVALID_ARG;
  return rf::read_device_error(status, as_stream(stream));
}

}  // extern "C"

rf_status rf_selftest_wait_timeout(int* waited_ms, void* stream) {
  if (!waited_ms) return RF_ERR_INVALID_ARG;
  return rf::launch_selftest_wait_timeout(waited_ms, as_stream(stream));
}

int rf_bounds_checked(void) {
#ifdef RF_CHECK_BOUNDS
  return 1;
#else
  return 0;
#endif
}

rf_status rf_selftest_bounds(void* stream) {
#ifdef RF_CHECK_BOUNDS
  return rf::launch_selftest_bounds(as_stream(stream));
#else
  (void)stream;
  return RF_ERR_UNSUPPORTED;
#endif
}
