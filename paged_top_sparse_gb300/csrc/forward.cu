// forward.cu -- the sparse forward with FP32 partials (the contract's storage) and the pages'
// FP8 route; the kernel itself is in forward.cuh.
#include "forward.cuh"

namespace sps {

cudaError_t launch_forward(const DevPlan& p, sps_dtype qt, sps_dtype kvt, const void* q,
                           float q_scale, const void* kc, const void* vc, const void* ks,
                           const void* vs, const int32_t* page_table, float* partial,
                           int64_t split_stride, float* lse, int64_t lse_split_stride,
                           cudaStream_t st) {
  return fwd::launch_forward_pt<fwd::kPF32>(p, qt, kvt, q, q_scale, kc, vc, ks, vs, page_table,
                                            partial, split_stride, lse, lse_split_stride, false,
                                            st);
}

cudaError_t launch_forward_fp8qk(const DevPlan& p, sps_dtype qt, sps_dtype kvt, const void* q,
                                 float q_scale, const void* kc, const void* vc, const void* ks,
                                 const void* vs, const int32_t* page_table, float* partial,
                                 int64_t split_stride, float* lse, int64_t lse_split_stride,
                                 cudaStream_t st) {
  return fwd::launch_forward_pt<fwd::kPF32>(p, qt, kvt, q, q_scale, kc, vc, ks, vs, page_table,
                                            partial, split_stride, lse, lse_split_stride, true,
                                            st);
}

}  // namespace sps
