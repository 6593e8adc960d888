// rf_stream_read: the read-bandwidth probe that the HBM-bound cascades are
// measured against.  It streams a buffer once with 16-byte non-coherent loads
// (the same load the decode and routing kernels use) and folds every 32-bit
// word into one XOR checksum, so no load can be dropped and nothing but the
// read itself costs time.  Timed over the routing logits it is that cascade's
// floor (a single read of the same bytes, launched the same way); timed over
// gigabytes it is the HBM read ceiling, which a read+write copy does not give.

#include "common.cuh"

namespace rf {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;           // 16-byte loads in flight per thread per step

__global__ void __launch_bounds__(kThreads)
stream_read_kernel(const uint4* __restrict__ x, size_t n16, uint32_t* __restrict__ out_xor) {
  const size_t stride = (size_t)gridDim.x * kThreads * kUnroll;
  uint32_t acc = 0u;
  for (size_t base = (size_t)blockIdx.x * kThreads * kUnroll + threadIdx.x; base < n16;
       base += stride) {
    uint4 v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const size_t i = base + (size_t)u * kThreads;
      v[u] = (i < n16 && RF_IDX_OK(i, n16)) ? ld_stream_v4(x + i) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) acc ^= v[u].x ^ v[u].y ^ v[u].z ^ v[u].w;
  }
  // fold the block's words into one, then one atomic per block: thousands of
  // warps updating one word would serialise at its L2 slice
  __shared__ uint32_t warp_xor[kThreads / 32];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc ^= __shfl_xor_sync(0xffffffffu, acc, o);
  if ((threadIdx.x & 31) == 0) warp_xor[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t b = 0u;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) b ^= warp_xor[w];
    if (b != 0u) atomicXor(out_xor, b);
  }
}

}  // namespace

rf_status launch_stream_read(const void* x, size_t nbytes, uint32_t* out_xor, cudaStream_t st) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return RF_ERR_CUDA;
  const size_t n16 = nbytes / 16;
  // enough blocks for every element of a small buffer to be loaded in the
  // first step; at most 8 resident blocks per SM, grid-stride beyond that
  const size_t per_block = (size_t)kThreads * kUnroll;
  const size_t need = (n16 + per_block - 1) / per_block;
  const size_t cap = (size_t)(sms > 0 ? sms : 1) * 8;
  const unsigned grid = (unsigned)(need < cap ? need : cap);
  stream_read_kernel<<<grid, kThreads, 0, st>>>(static_cast<const uint4*>(x), n16, out_xor);
  return launch_status();
}

RF_BOUNDS_WORD_OF_THIS_FILE

}  // namespace rf

extern "C" rf_status rf_stream_read(const void* x, size_t nbytes, uint32_t* out_xor,
                                    void* stream) {
  if (!x || !out_xor || nbytes == 0) return RF_ERR_INVALID_ARG;
  if (nbytes % 16 != 0) return RF_ERR_UNSUPPORTED;
  if (!rf::aligned16(x) || (reinterpret_cast<uintptr_t>(out_xor) & 3u) != 0) return RF_ERR_MISALIGNED;
  return rf::launch_stream_read(x, nbytes, out_xor, static_cast<cudaStream_t>(stream));
}
