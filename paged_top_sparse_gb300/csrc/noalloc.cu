// noalloc.cu -- sparse_prefill_fwd_noalloc: the sparse forward with its scratch memory in a
// fixed device array that the library itself provides, for callers that cannot allocate
// device memory (see the declaration in sparse_prefill.h for who they are and the rules).
//
// The array is a file-scope __device__ variable, so every GPU that loads the library holds it
// until the process exits.  Host code never uses the symbol directly as an address: it asks
// the runtime for the device address once per device (cudaGetSymbolAddress, with that device
// current) and passes that pointer to the kernels.
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>

#include "sps_internal.h"

namespace sps {
namespace {

constexpr size_t kNoAllocBytes = 48ull << 20;  // 48 MiB of scratch per device
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once per device).
cudaError_t scratch_for_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace sps

// Defined in host.cpp: argument checks, metadata upload and launches on a given scratch area.
sps_status sps_internal_fwd_noalloc(const sps_plan* plan, const void* q, float q_scale,
                                    const void* k_cache, const void* v_cache, const void* k_scales,
                                    const void* v_scales, const int32_t* page_table,
                                    const int32_t* idx, float* partial, int64_t split_stride,
                                    float* lse, int64_t lse_split_stride, void* scratch,
                                    size_t scratch_bytes, int32_t* dev_status,
                                    sps_stream_t stream);
sps_status sps_internal_cuda_fail(cudaError_t e, const char* what);

extern "C" sps_status sparse_prefill_fwd_noalloc(
    const sps_plan* plan, const void* q, float q_scale, const void* k_cache, const void* v_cache,
    const void* k_scales, const void* v_scales, const int32_t* page_table, const int32_t* idx,
    float* partial, int64_t split_stride, float* lse, int64_t lse_split_stride,
    int32_t* dev_status, sps_stream_t stream) {
  void* ws = nullptr;
  cudaError_t e = sps::scratch_for_current_device(&ws);
  if (e != cudaSuccess) return sps_internal_cuda_fail(e, "cudaGetSymbolAddress(scratch)");
  return sps_internal_fwd_noalloc(plan, q, q_scale, k_cache, v_cache, k_scales, v_scales,
                                  page_table, idx, partial, split_stride, lse, lse_split_stride,
                                  ws, sps::kNoAllocBytes, dev_status, stream);
}
