// upload.cu -- the plan-metadata upload as a copy kernel that reads page-locked host memory
// directly.  A host-to-device DMA on the copy engine queues behind whatever copies the caller
// has in flight on other streams (a prefill overlapping the next batch's inputs waits for that
// whole transfer); loads issued by the SMs do not.
#include "ptx.cuh"
#include "sps_internal.h"

namespace sps {
namespace {

__global__ void __launch_bounds__(256)
staged_copy_kernel(const int4* __restrict__ src, int4* __restrict__ dst, int64_t n16,
                   const uint8_t* __restrict__ src_tail, uint8_t* __restrict__ dst_tail,
                   int tail) {
  pdl_trigger();  // the indexer that follows may start its prologue
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += stride)
    dst[i] = src[i];
  if (blockIdx.x == 0 && threadIdx.x < tail) dst_tail[threadIdx.x] = src_tail[threadIdx.x];
}

}  // namespace

cudaError_t launch_staged_copy(const void* src, void* dst, size_t n, cudaStream_t st) {
  const int64_t n16 = (int64_t)(n / 16);
  const int tail = (int)(n % 16);
  if (n == 0) return cudaSuccess;
  const int64_t want = (n16 + 255) / 256;
  const unsigned blocks = (unsigned)(want < 1 ? 1 : (want > 1024 ? 1024 : want));
  staged_copy_kernel<<<blocks, 256, 0, st>>>(
      static_cast<const int4*>(src), static_cast<int4*>(dst), n16,
      static_cast<const uint8_t*>(src) + n16 * 16, static_cast<uint8_t*>(dst) + n16 * 16, tail);
  return cudaGetLastError();
}

}  // namespace sps
