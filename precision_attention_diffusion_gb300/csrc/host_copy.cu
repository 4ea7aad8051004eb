// host_copy.cu -- gather a chunk of heads from a page-locked host view into a dense device buffer.
//
// The host-buffer entry point copies each chunk of heads of the caller's [T, H, 128] BF16 views
// (any token and head strides) into dense [T, n, 128] device slots. A 2D DMA copy of such a chunk
// moves one row of n x 256 bytes per token and costs a fixed time per row on top of the bytes (on
// GB300 about 6 ns: a 7-head chunk of a 30272-token segment crosses the link at ~118 GB/s instead
// of ~211 GB/s). This kernel reads the page-locked source through its device mapping instead:
// every thread moves 16-byte units with several loads in flight, whatever the row width.
#include <cstdint>

#include "fa_lp_internal.h"

namespace falp {
namespace {

constexpr int kGatherThreads = 256;
constexpr int kGatherUnroll = 8;  // 16-byte loads in flight per thread

__global__ void __launch_bounds__(kGatherThreads) gather_heads_kernel(
    uint4* __restrict__ dst, const uint8_t* __restrict__ src, int64_t src_st_bytes,
    int64_t src_sh_bytes, int64_t T, int n) {
  const int64_t units_per_tok = int64_t(n) * 16;  // 16-byte units of one token's chunk row
  const int64_t total = T * units_per_tok;
  const int64_t stride = int64_t(gridDim.x) * kGatherThreads;
  for (int64_t base = int64_t(blockIdx.x) * kGatherThreads + threadIdx.x; base < total;
       base += stride * kGatherUnroll) {
    uint4 v[kGatherUnroll];
#pragma unroll
    for (int j = 0; j < kGatherUnroll; ++j) {
      const int64_t u = base + int64_t(j) * stride;
      if (u < total) {
        const int64_t t = u / units_per_tok, r = u - t * units_per_tok;
        const int64_t h = r >> 4, part = r & 15;
        v[j] = *reinterpret_cast<const uint4*>(src + t * src_st_bytes + h * src_sh_bytes +
                                               part * 16);
      }
    }
#pragma unroll
    for (int j = 0; j < kGatherUnroll; ++j) {
      const int64_t u = base + int64_t(j) * stride;
      if (u < total) dst[u] = v[j];
    }
  }
}

}  // namespace

int launch_gather_heads(void* dst, const void* src_dev, int64_t src_st, int64_t src_sh,
                        int64_t T, int n, cudaStream_t stream) {
  if (T <= 0 || n <= 0) return FA_LP_OK;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) {
    cudaGetLastError();
    sms = 152;
  }
  gather_heads_kernel<<<unsigned(4 * sms), kGatherThreads, 0, stream>>>(
      static_cast<uint4*>(dst), static_cast<const uint8_t*>(src_dev), src_st * 2, src_sh * 2, T,
      n);
  return cuda_status(cudaGetLastError());
}

}  // namespace falp
