/*
 * rf.h -- C ABI of librf.so: single-pass fused cascaded reductions on GB300.
 *
 * A cascaded reduction is a chain of reductions in which each stage needs
 * the finished result of the one before (RedFuser episode transcript, cue 9:
 * safe softmax's row max, then the exp-sum denominator, then the divide;
 * cue 11: softmax then top-k for MoE routing, abs-max then FP8 quantisation
 * then GEMM).  Every call below computes such a chain in one pass over its
 * input by carrying a running state and rescaling stale partials when an
 * earlier stage's result changes (transcript cues 15-21 and 31; the episode
 * viz page's widgets "Online softmax, step by step" and "Merging partial
 * states across blocks (FlashDecoding-style)").
 *
 * Conventions shared by every call
 * --------------------------------
 * - Pointers named as tensors are DEVICE pointers (CUDA global memory) unless
 *   stated otherwise.  The caller owns every buffer; the library allocates
 *   nothing and frees nothing.
 * - All tensors are dense, row-major and contiguous in the shapes given.
 * - `stream` is a cudaStream_t passed as an opaque pointer (NULL = the legacy
 *   default stream).  Calls only enqueue work: they are asynchronous and
 *   stream-ordered, and never synchronise.
 * - Arguments are checked on the host before anything is launched.  A bad
 *   argument returns its status code with nothing enqueued and no output
 *   touched.  A failed launch returns RF_ERR_CUDA.  Nothing aborts, prints or
 *   throws across this boundary.
 * - Device pointers must be 16-byte aligned (RF_ERR_MISALIGNED otherwise).
 * - Calls are thread-safe and keep no per-call state of their own, with two
 *   exceptions: rf_attn_decode_noalloc's fixed arrays (shared by every call
 *   on a device, see there), and the on-device status words that
 *   rf_device_error reads.  Those words are one set per device for the whole
 *   process: every call of every thread records into the same words, and a
 *   read by any thread clears them for all, so one thread's rf_device_error
 *   can consume a timeout that another thread's call recorded.
 */
#ifndef RF_H
#define RF_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  RF_OK = 0,
  RF_ERR_INVALID_ARG = 1,   /* null pointer, size <= 0, k > E, S < 1, ...     */
  RF_ERR_UNSUPPORTED = 2,   /* a valid request outside the supported set      */
  RF_ERR_MISALIGNED = 3,    /* a pointer is not 16-byte aligned               */
  RF_ERR_CUDA = 4,          /* a CUDA runtime call or kernel launch failed    */
  RF_ERR_TIMEOUT = 5,       /* a bounded on-device wait gave up (see below)   */
  RF_ERR_BOUNDS = 6         /* bounds-checked build only: an index was out of
                               range and its access was skipped (see below)   */
} rf_status;

typedef enum { RF_F32 = 0, RF_BF16 = 1 } rf_dtype;

/* Human-readable name of a status code (static string, never NULL). */
const char* rf_status_string(int status);

/* Library version: major * 10000 + minor * 100 + patch. */
int rf_version(void);

/*
 * rf_attn_decode_split -- split-KV decode attention, producer of segment
 * states (the Multi-Segment strategy: transcript cue 39; viz page widget
 * "Single-Segment vs Multi-Segment").
 *
 * For each row r (r = b*H + h) and each segment s of its L keys, the kernel
 * streams the segment's K and V rows once and keeps the running state of
 * transcript cues 15-19 and 31:
 *   m' = max(m, max_j s_j),   c = exp(m - m'),
 *   l' = c*l + sum_j exp(s_j - m'),   acc' = c*acc + sum_j exp(s_j - m') v_j,
 * with scores s_j = scale * <q_r, k_j>.  It writes the unnormalised state.
 *
 *   q        [R, D]      dtype          query rows
 *   k, v     [R, L, D]   dtype          keys / values of each row
 *   R, L, D  rows, keys per row, head dim
 *   S        number of segments, >= 1.  Segment s holds the keys
 *            [s*c, min(L, (s+1)*c)), c = ceil(L/S).  S > L is allowed: a
 *            segment with no keys gets the identity state (-inf, 0, 0)
 *            (transcript cues 27 and 29: the monoid's identity element).
 *   scale    score scale (1/sqrt(D) for attention)
 *   dtype    RF_F32 with D = 64, or RF_BF16 with D = 128
 *   seg_m    [R, S]      fp32 out       segment max of the scores, natural-log units
 *   seg_l    [R, S]      fp32 out       sum_j exp(s_j - seg_m)
 *   seg_acc  [R, S, D]   fp32 out       sum_j exp(s_j - seg_m) * v_j
 * Errors: RF_ERR_INVALID_ARG for null pointers, R, L, D <= 0, S < 1 or a
 * non-finite scale; RF_ERR_UNSUPPORTED for any other (dtype, D) pair.
 */
rf_status rf_attn_decode_split(const void* q, const void* k, const void* v,
                               int R, int L, int D, int S, float scale, int dtype,
                               float* seg_m, float* seg_l, float* seg_acc,
                               void* stream);

/*
 * rf_attn_decode_split_twopass -- the non-incremental counterpart of
 * rf_attn_decode_split, for the incremental vs non-incremental comparison of
 * transcript cue 45 (the non-incremental form fits only short per-block
 * sequences).  Same arguments and the same segment states out; each CTA
 * first computes and keeps every score of its segment in shared memory and
 * reduces their max, then accumulates l and acc against that final max with
 * no rescaling.  Segments (ceil(L/S) keys) must not exceed 16384 keys:
 * RF_ERR_UNSUPPORTED otherwise.
 */
rf_status rf_attn_decode_split_twopass(const void* q, const void* k, const void* v,
                                       int R, int L, int D, int S, float scale, int dtype,
                                       float* seg_m, float* seg_l, float* seg_acc,
                                       void* stream);

/*
 * rf_state_merge -- combine the S segment states of each row and normalise
 * (transcript cue 21: two partial states, each with its own max, combine with
 * the same rescaling; viz page widget "Merging partial states across blocks").
 *   M = max_s m_s;  w_s = exp(m_s - M) (0 for an identity state);
 *   l = sum_s w_s l_s;  acc = sum_s w_s acc_s;  out = acc / l;  lse = M + ln l.
 *
 *   seg_m, seg_l, seg_acc   as written by rf_attn_decode_split
 *                           or rf_mla_decode_split
 *   R, S, D                 rows, segments, value width (D = 64, 128 or 512)
 *   out        [R, D]       out_dtype out (RF_F32 or RF_BF16, round to nearest even)
 *   lse        [R]          fp32 out, may be NULL
 * Errors: RF_ERR_INVALID_ARG for null inputs/out, R, S, D <= 0;
 * RF_ERR_UNSUPPORTED for D not in {64, 128, 512}.
 * A row whose S states are all identity states gives NaN (it had no keys).
 */
rf_status rf_state_merge(const float* seg_m, const float* seg_l, const float* seg_acc,
                         int R, int S, int D, void* out, int out_dtype, float* lse,
                         void* stream);

/*
 * rf_mla_decode_split -- multi-latent attention (MLA) decode, producer of
 * segment states (transcript cue 41: the MLA workload, compared with
 * DeepSeek's FlashMLA; cue 55: decode shapes, one query row; cue 39: the
 * Multi-Segment split).  Every query head of a sequence reads the same latent
 * cache row c_j [Dk]; the value is its leading Dv dims:
 *   s_hj = scale * <q_h, c_j>,  state (m, l, acc) per (sequence, head,
 *   segment) exactly as rf_attn_decode_split writes it, with v_j = c_j[:Dv].
 * The products run on the tensor cores (S^T = C Q^T and O^T += C[:, :Dv]^T P^T,
 * keys along the 128 TMEM lanes, heads along the columns).
 *
 *   q        [B, H, Dk]   bf16     query heads (already in the latent space)
 *   c        [B, L, Dk]   bf16     latent cache, one row per key, shared by
 *                                  the H heads of a sequence
 *   B, H, L  sequences, query heads (a multiple of 16), keys per sequence
 *   Dk, Dv   latent and value widths: 576 and 512 (512 latent + 64 rotary)
 *   S        number of segments, >= 1, split as in rf_attn_decode_split
 *            (ceil(L/S) keys each; segments past the end get the identity)
 *   scale    score scale
 *   seg_m    [B, H, S]      fp32 out   segment max, natural-log units
 *   seg_l    [B, H, S]      fp32 out   sum_j exp(s_hj - seg_m)
 *   seg_acc  [B, H, S, Dv]  fp32 out   sum_j exp(s_hj - seg_m) * c_j[:Dv]
 * Combine with rf_state_merge(seg_m, seg_l, seg_acc, B*H, S, Dv, ...).
 * Errors: RF_ERR_INVALID_ARG for null pointers, B, H, L <= 0, S < 1 or a
 * non-finite scale; RF_ERR_UNSUPPORTED for (Dk, Dv) other than (576, 512),
 * H not a multiple of 16 or B*L >= 2^31; RF_ERR_MISALIGNED unless q, c and
 * seg_acc are 16-byte aligned; RF_ERR_TIMEOUT (through rf_device_error) if a
 * pipeline wait inside the kernel gave up.
 */
rf_status rf_mla_decode_split(const void* q, const void* c, int B, int H, int L, int Dk,
                              int Dv, int S, float scale, float* seg_m, float* seg_l,
                              float* seg_acc, void* stream);

/*
 * rf_attn_prefill -- causal prefill attention, GEMM -> online softmax -> GEMM
 * (transcript cue 9: attention stacks a GEMM, then softmax, then another GEMM;
 * cue 31: the incremental form sits at the block level of the reduction tree).
 * Each 128-row query tile streams its K/V blocks once: S = Q K^T * scale on
 * the tensor cores, running (m, l) per row, O = c*O + P V, out = O / l.  The
 * kernel runs on clusters of two CTAs (two adjacent query tiles of a head
 * share every K/V block).
 *
 *   q, k, v   [B, H, N, D]  bf16        D = 128
 *   causal    1: query i sees keys 0..i (top-left aligned); 0: all keys
 *   scale     score scale (1/sqrt(D))
 *   out       [B, H, N, D]  bf16 out
 *   lse       [B, H, N]     fp32 out (m + ln l, natural log), may be NULL
 * Any N >= 1: the last query and key tiles of a head are partial (keys past
 * N are left out, rows past N are not stored).
 * Errors: RF_ERR_INVALID_ARG for null pointers or sizes <= 0;
 * RF_ERR_UNSUPPORTED unless D = 128 and B*H*N < 2^31, or when a cluster of
 * two CTAs with about 200 KiB of shared memory each cannot be launched on
 * the device.
 */
rf_status rf_attn_prefill(const void* q, const void* k, const void* v,
                          int B, int H, int N, int D, int causal, float scale,
                          void* out, float* lse, void* stream);

/*
 * rf_softmax_topk -- MoE routing: softmax over experts, then top-k, from one
 * read of each token's logits (transcript cue 11; "Online normalizer
 * calculation for softmax", abstract: softmax and top-k fused).
 *
 *   logits  [T, E]  fp32
 *   k       experts per token, 1 <= k <= min(E, 32)
 *   renormalize  1: w_i = p_i / sum_{j in top-k} p_j;  0: w_i = p_i
 *   idx     [T, k]  int32 out  expert indices, ordered by logit descending,
 *                              equal logits by lower index first
 *   w       [T, k]  fp32 out   routing weights in the same order
 * Errors: RF_ERR_INVALID_ARG for null pointers, T, E <= 0, k < 1 or k > E;
 * RF_ERR_UNSUPPORTED for E > 1024 or k > 32; RF_ERR_MISALIGNED unless
 * logits, idx and w are 16-byte aligned.
 */
rf_status rf_softmax_topk(const float* logits, int T, int E, int k, int renormalize,
                          int32_t* idx, float* w, void* stream);

/*
 * rf_absmax_quant_fp8_gemm -- FP8 per-token quantisation then GEMM
 * (transcript cue 33: the token's abs-max, then the GEMM over values scaled
 * by FP8max / absmax).  Two kernels, enqueued back to back:
 *   1. one pass over each row of X: amax = max |x|, sx = fp32(amax / 448),
 *      xq = e4m3(fp32(x / sx)) rounded to nearest even, saturating at +-448;
 *      a row with amax = 0 gets sx = 0 and zero codes;
 *   2. Y = (Xq . Wq^T) * sx[m] * sw[n], fp32 accumulation on the FP8 tensor
 *      cores, rounded to bf16.
 *
 *   x    [M, K]  bf16           activations
 *   wq   [N, K]  e4m3 codes     weights (K-contiguous storage of W [K, N])
 *   sw   [N]     fp32           per-output-column weight scales
 *   xq   [M, K]  e4m3 codes out
 *   sx   [M]     fp32 out       per-token scales
 *   y    [M, N]  bf16 out
 * Any M, N >= 1; K a multiple of 16 (16-byte code rows) up to 65536.  The
 * GEMM works on 256 x 256 output tiles, each computed by a cluster of two
 * CTAs (128 x 256 tiles on single CTAs when M <= 128 or when such a cluster
 * cannot be launched on the device); partial tiles at the
 * M, N and K edges read zeros past the edge and store only inside Y.
 * Errors: RF_ERR_INVALID_ARG for null pointers or sizes <= 0;
 * RF_ERR_UNSUPPORTED unless K % 16 == 0 and K <= 65536; RF_ERR_MISALIGNED
 * unless x, wq, sw, xq and y are 16-byte aligned.
 */
rf_status rf_absmax_quant_fp8_gemm(const void* x, int M, int K,
                                   const uint8_t* wq, const float* sw, int N,
                                   uint8_t* xq, float* sx, void* y, void* stream);

/*
 * rf_attn_decode_fused -- rf_attn_decode_split and rf_state_merge in one
 * launch, for latency-bound calls (few rows, where the second launch costs
 * as much as the work).  Every CTA writes its segment state as
 * rf_attn_decode_split does, then counts itself in counters[row]; the CTA
 * that completes a row's count merges that row's S states (the merge of
 * rf_state_merge, transcript cue 21) into out and lse and sets the counter
 * back to 0.  No CTA ever waits for another.
 *   q, k, v, R, L, D, S, scale, dtype, seg_m, seg_l, seg_acc
 *            as rf_attn_decode_split (the states are written as there)
 *   counters [R] int32, device memory: all 0 before the call; a call that
 *            completes leaves them 0 again, so one zeroed buffer serves every
 *            later call.  Calls that may overlap on the GPU need separate
 *            counters and states.
 *   out, out_dtype, lse  as rf_state_merge
 * Errors: as rf_attn_decode_split, plus RF_ERR_INVALID_ARG for a null
 * counters or out or a bad out_dtype, and RF_ERR_MISALIGNED unless out and
 * counters are 16-byte aligned.
 */
rf_status rf_attn_decode_fused(const void* q, const void* k, const void* v, int R, int L, int D,
                               int S, float scale, int dtype, float* seg_m, float* seg_l,
                               float* seg_acc, int* counters, void* out, int out_dtype,
                               float* lse, void* stream);

/*
 * rf_attn_decode_noalloc -- split-KV decode with the state merge in the same
 * launch (as rf_attn_decode_fused), for callers that cannot allocate device
 * memory: for example a plugin inside
 * a host engine that owns every device allocation, a latency-critical loop
 * that cannot afford cudaMalloc's implicit device synchronisation, or a
 * process whose memory budget was fixed at start-up.  The pages have no
 * counterpart to this call; it is a deployment convenience.
 *
 * Same q, k, v, R, L, D, S, scale, dtype as rf_attn_decode_split and same
 * out, out_dtype, lse as rf_state_merge.  The segment states live in a fixed
 * 16 MiB array inside the library (allocated once per GPU when the library
 * is loaded, kept until the process exits) instead of caller buffers, so the
 * call itself allocates nothing.  Every accepted call is one launch, as
 * rf_attn_decode_fused, with its per-row counters in a second fixed array
 * of 65536 entries.
 * - It needs 8*R*S bytes rounded up to 256, plus 4*R*S*D bytes, to fit in
 *   16 MiB; larger requests return RF_ERR_UNSUPPORTED with nothing launched.
 *   That limit also caps R at 65536 (even at S = 1, D = 64).
 * - Every call on a GPU shares that array: calls that may overlap on the GPU
 *   (different streams, unordered host threads) race; order them on one
 *   stream.  Each call rewrites every state it reads, so nothing needs
 *   clearing between calls.
 * - The first call on each device (with that device current) looks up the
 *   array's device address; make it before any stream capture.
 * Errors: as rf_attn_decode_split and rf_state_merge; RF_ERR_CUDA if the
 * address look-up fails.
 */
rf_status rf_attn_decode_noalloc(const void* q, const void* k, const void* v,
                                 int R, int L, int D, int S, float scale, int dtype,
                                 void* out, int out_dtype, float* lse, void* stream);

/*
 * rf_incremental_quant_fp8_gemm -- the incremental form of the FP8 cascade in
 * one kernel (transcript cue 33: when the running abs-max grows, multiply the
 * running accumulator by the old abs-max over the new one).  Per row and
 * K-tile of 128 columns, in order: a' = max(a, tile max |x|), s' = fp32(a' /
 * 448); if the scale grew, acc *= s / s'; the tile is quantised with s' (the
 * same rounding as rf_absmax_quant_e4m3) and accumulated on the FP8 tensor
 * cores; Y = bf16(acc * s_final * sw).  The codes of early tiles use the
 * running scale, so Y differs from rf_absmax_quant_fp8_gemm's (it is a
 * different quantisation of X, at least as fine); no Xq is written.  When
 * N / 512 is a multiple of 4 (8), the CTAs that share a 128-row block run as
 * one thread-block cluster and each quantises a band of the rows for all of
 * them; otherwise each CTA quantises its whole block.  Same results either way.
 *   x [M, K] bf16;  wq [N, K] e4m3;  sw [N] fp32;  y [M, N] bf16 out
 *   sx_final [M] fp32 out (the final per-row scale), may be NULL
 * Errors: RF_ERR_INVALID_ARG for null pointers or sizes <= 0;
 * RF_ERR_UNSUPPORTED unless M % 128 == 0, N % 512 == 0 and K % 128 == 0.
 */
rf_status rf_incremental_quant_fp8_gemm(const void* x, int M, int K, const uint8_t* wq,
                                        const float* sw, int N, void* y, float* sx_final,
                                        void* stream);

/* Phase 1 of rf_absmax_quant_fp8_gemm alone (same arguments and rules;
 * any K % 8 == 0 is supported). */
rf_status rf_absmax_quant_e4m3(const void* x, int M, int K, uint8_t* xq, float* sx,
                               void* stream);

/* Phase 2 of rf_absmax_quant_fp8_gemm alone (same arguments and rules). */
rf_status rf_fp8_gemm_scaled(const uint8_t* xq, const float* sx, const uint8_t* wq,
                             const float* sw, int M, int N, int K, void* y, void* stream);

/*
 * Single-row cascades (transcript cue 47: safe softmax of 1K-8K-element rows
 * at several fusion levels; variance; moment of inertia).  One row per CTA.
 * `level` selects where in the reduction tree the incremental state is kept:
 *   RF_FUSE_NONE    unfused: one kernel per reduction, each re-reading the row
 *   RF_FUSE_THREAD  each thread folds its elements one by one into a state,
 *                   thread states are merged at the end
 *   RF_FUSE_WARP    each warp folds 128-element tiles into a warp state
 *   RF_FUSE_BLOCK   the block folds 1024-element tiles into one block state
 * All levels compute the same result (up to fp32 rounding order).
 * Rows hold n fp32 values, n % 4 == 0 (RF_ERR_UNSUPPORTED otherwise).
 */
typedef enum { RF_FUSE_NONE = 0, RF_FUSE_THREAD = 1, RF_FUSE_WARP = 2, RF_FUSE_BLOCK = 3 } rf_fusion_level;

/* rf_row_softmax -- y = softmax(x) per row: max, then sum of exp(x - max),
 * then the divide (transcript cue 9).
 *   x, y  [R, n] fp32 (y may not alias x)
 *   work  [2R] fp32 scratch for RF_FUSE_NONE (row max and sum), else may be NULL
 * Fused levels hold the row in registers: n <= 8192 (RF_ERR_UNSUPPORTED above). */
rf_status rf_row_softmax(const float* x, int R, int n, float* y, int level, float* work,
                         void* stream);

/* rf_row_variance -- population variance per row: mean = sum x / n, then
 * var = sum (x - mean)^2 / n; fused levels merge (count, mean, M2) states.
 *   x [R, n] fp32;  mean [R], var [R] fp32 out */
rf_status rf_row_variance(const float* x, int R, int n, float* mean, float* var, int level,
                          void* stream);

/* rf_moment_of_inertia -- per row of n point masses: centre of mass
 * c = sum m p / sum m, then I = sum m |p - c|^2 (about the centre of mass);
 * fused levels merge (M, c, I) states by the parallel-axis theorem.
 *   mass [R, n] fp32 (positive);  pos [R, 3, n] fp32 (x, y, z coordinates of
 *   each row stored one after the other);  center [R, 3], inertia [R] fp32 out */
rf_status rf_moment_of_inertia(const float* mass, const float* pos, int R, int n, float* center,
                               float* inertia, int level, void* stream);

/* rf_layer_norm -- y = (x - mean) / sqrt(var + eps) * gamma + beta per row:
 * mean, then variance (needs the mean), then the normalisation (needs both)
 * (the bookshelf explainer's "Problem" section lists normalisation layers
 * among the cascaded reductions).  RF_FUSE_NONE runs one kernel per stage,
 * each re-reading the row; any other level runs the fused single-read kernel
 * (the row stays in registers, n <= 8192).
 *   x, y [R, n] fp32;  gamma, beta [n] fp32;  eps >= 0
 *   work [2R] fp32 scratch for RF_FUSE_NONE (row mean and variance), else may be NULL */
rf_status rf_layer_norm(const float* x, const float* gamma, const float* beta, int R, int n,
                        float eps, float* y, int level, float* work, void* stream);

/* rf_rms_norm -- y = x / sqrt(mean(x^2) + eps) * gamma per row: the mean of
 * squares, then the normalisation that needs it (the bookshelf explainer's
 * "Problem" section lists normalisation layers among the cascaded
 * reductions).  RF_FUSE_NONE runs one kernel per stage, each reading the
 * row; any other level runs the fused single-read kernel (the row stays in
 * registers, n <= 8192).
 *   x, y [R, n] fp32 (n % 4 == 0);  gamma [n] fp32;  eps >= 0
 *   work [R] fp32 scratch for RF_FUSE_NONE (row mean of squares), else may be NULL
 * Errors: RF_ERR_INVALID_ARG for null pointers, R, n <= 0, a level outside
 * 0..3, a negative or non-finite eps, or RF_FUSE_NONE without work;
 * RF_ERR_UNSUPPORTED for n % 4 != 0 or a fused call with n > 8192;
 * RF_ERR_MISALIGNED unless x, y and gamma are 16-byte aligned. */
rf_status rf_rms_norm(const float* x, const float* gamma, int R, int n, float eps, float* y,
                      int level, float* work, void* stream);

/*
 * rf_selftest_wait_timeout -- a self-test of the bounded waits (the pages
 * have no counterpart: this checks this library's failure detection).  One
 * thread of a one-CTA kernel waits on a shared-memory barrier that nothing
 * arrives on, through the same bounded wait every tensor-core pipeline wait
 * uses; after the limit (about 1 s) the wait gives up, the kernel records
 * RF_ERR_TIMEOUT for rf_device_error and returns normally (no fault, no
 * hang; the context stays usable).
 *   waited_ms  [1] int32, device memory, out: how long the wait lasted in
 *              milliseconds, or -1 if it completed (it never should)
 * Errors: RF_ERR_INVALID_ARG for a null pointer.  The timeout itself is
 * reported by the next rf_device_error call, not by this call.
 */
rf_status rf_selftest_wait_timeout(int* waited_ms, void* stream);

/*
 * rf_stream_read -- the read-bandwidth probe.  The pages have no counterpart:
 * it is the measuring stick for the HBM-bound calls above.  It reads
 * nbytes of x once, with the 16-byte non-coherent streaming loads the
 * decode and routing kernels use, and XORs every 32-bit word of x into
 * *out_xor (so *out_xor ^= w_0 ^ w_1 ^ ...; zero it first for the plain
 * checksum).  Timed over a cascade's own input it gives that cascade's
 * floor; timed over gigabytes it gives the HBM read ceiling.
 *   x        device memory, nbytes long, 16-byte aligned
 *   out_xor  [1] uint32, device memory, in/out
 * Errors: RF_ERR_INVALID_ARG for null pointers or nbytes == 0;
 * RF_ERR_UNSUPPORTED unless nbytes % 16 == 0; RF_ERR_MISALIGNED unless x is
 * 16-byte and out_xor 4-byte aligned.
 */
rf_status rf_stream_read(const void* x, size_t nbytes, uint32_t* out_xor, void* stream);

/*
 * rf_device_error -- status of the on-device checks.  The tensor-core
 * kernels wait on shared-memory barriers with an iteration limit; a wait
 * that runs out records RF_ERR_TIMEOUT in a device word and the kernel
 * returns early instead of hanging.  In the bounds-checked build (compiled
 * with -DRF_CHECK_BOUNDS, see rf_bounds_checked) every kernel also checks
 * each global-memory index against the extent of its buffer, derived from
 * the call's sizes; an index out of range skips its load or store and
 * records RF_ERR_BOUNDS.  This call synchronises `stream`, reads every such
 * word into *status (RF_OK if nothing was recorded), clears them, and
 * returns RF_OK, or RF_ERR_CUDA if the read failed.
 * The words are process-global (one set per device, not per stream, thread
 * or call): a status recorded by any caller's kernel is reported to whichever
 * thread calls this first, and that read clears it for every other caller.
 * Callers on several threads that need to attribute a status should
 * serialise their calls and this read with a lock of their own.
 */
rf_status rf_device_error(int* status, void* stream);

/*
 * rf_bounds_checked -- 1 if this library was built with -DRF_CHECK_BOUNDS
 * (the debug variant whose kernels check every global index and report
 * RF_ERR_BOUNDS through rf_device_error), else 0.
 */
int rf_bounds_checked(void);

/*
 * rf_selftest_bounds -- a self-test of the bounds checks.  A one-thread
 * kernel presents one index equal to its buffer's extent (one past the end)
 * to the same check every kernel uses; the check refuses it, so the guarded
 * store, which would have gone to element 0 of an internal one-word buffer
 * anyway, is skipped and RF_ERR_BOUNDS is recorded for rf_device_error.
 * Errors: RF_ERR_UNSUPPORTED unless rf_bounds_checked() is 1.
 */
rf_status rf_selftest_bounds(void* stream);

#ifdef __cplusplus
}
#endif

#endif /* RF_H */
