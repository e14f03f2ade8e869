// forward_p16.cu -- the sparse forward with 16-bit partials ("MSA PR 21: Q8KV4 paged sparse
// prefill", Combine: the pages keep BF16/FP16 partials): BF16 or FP16, nearest even.  The
// kernel is in forward.cuh.
#include "forward.cuh"

namespace sps {

cudaError_t launch_forward_bf16p(const DevPlan& p, sps_dtype qt, sps_dtype kvt, const void* q,
                                 float q_scale, const void* kc, const void* vc, const void* ks,
                                 const void* vs, const int32_t* page_table, void* partial,
                                 int64_t split_stride, float* lse, int64_t lse_split_stride,
                                 cudaStream_t st) {
  return fwd::launch_forward_pt<fwd::kPBF16>(p, qt, kvt, q, q_scale, kc, vc, ks, vs, page_table,
                                             partial, split_stride, lse, lse_split_stride, false,
                                             st);
}

cudaError_t launch_forward_f16p(const DevPlan& p, sps_dtype qt, sps_dtype kvt, const void* q,
                                float q_scale, const void* kc, const void* vc, const void* ks,
                                const void* vs, const int32_t* page_table, void* partial,
                                int64_t split_stride, float* lse, int64_t lse_split_stride,
                                cudaStream_t st) {
  return fwd::launch_forward_pt<fwd::kPF16>(p, qt, kvt, q, q_scale, kc, vc, ks, vs, page_table,
                                            partial, split_stride, lse, lse_split_stride, false,
                                            st);
}

}  // namespace sps
