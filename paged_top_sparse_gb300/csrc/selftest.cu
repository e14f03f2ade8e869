// selftest.cu -- sps_check_wait_timeout / sps_check_barrier_timeout: exercise the library's
// bounded mbarrier wait, and the bounded grid barrier of its cooperative launches, on a
// barrier that nothing ever completes.  The wait must give up after the limit, record
// SPS_DEV_TIMEOUT in the status word and return, leaving the context usable; this is how every
// kernel here turns a lost arrive into an error status instead of a hung GPU.
#include "ptx.cuh"
#include "sps_internal.h"

namespace sps {
namespace {

__global__ void wait_timeout_kernel(int32_t* status, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);  // expects one arrive that never comes
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(smem_u32(&bar), 0, &abort_flag, status, limit_ns);
}

// Two blocks of a cooperative launch: block 1 leaves without arriving, so block 0's grid
// barrier never completes and must give up.
__global__ void barrier_timeout_kernel(unsigned int* bar, int32_t* status, uint64_t limit_ns) {
  __shared__ int flag;
  if (blockIdx.x == 1) return;
  grid_barrier(bar, status, &flag, limit_ns);
}

}  // namespace

cudaError_t launch_barrier_timeout(unsigned int* bar, int32_t* status, int64_t limit_ns,
                                   cudaStream_t st) {
  uint64_t lim = (uint64_t)limit_ns;
  void* args[] = {&bar, &status, &lim};
  return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(barrier_timeout_kernel),
                                     dim3(2), dim3(32), args, 0, st);
}

cudaError_t launch_wait_timeout(int32_t* status, int64_t limit_ns, cudaStream_t st) {
  wait_timeout_kernel<<<1, 32, 0, st>>>(status, (uint64_t)limit_ns);
  return cudaGetLastError();
}

}  // namespace sps
