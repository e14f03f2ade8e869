// sps_internal.h -- plan layout shared by the host library and the kernels (not installed).
#pragma once
#include <cuda_runtime.h>
#include <cstdint>

#include "sparse_prefill.h"

namespace sps {

constexpr int kPage = 128;         // tokens per KV page
constexpr int kMaxTopK = 64;
constexpr int kFwdTaskGroups = 8;  // 128-row query groups per forward work item
constexpr int kChunkWords = 8;     // 32-row words per inversion chunk (one 256-thread block)
constexpr int kInvPages = 64;      // pages per inversion window (one 64-bit row mask)
// Visible pages of one request: 8192 (1M tokens) with top_k <= 16, where the inversion packs a
// page into 16 bits; 1024 (128K tokens) with top_k > 16, whose warp-per-row top-k holds at most
// 32 pages per lane.  The single-launch inversion keeps a 1024-entry offset table per block, so
// longer requests take its three-kernel form.
constexpr int kMaxPagesPerReq = 8192;
constexpr int kMaxPagesWideK = 1024;
constexpr int kInvFusedMaxPages = 1024;
constexpr int kInvScanBuckets = 8;  // buckets per block of the multi-kernel inversion's scan

// One request of the batch, as the kernels see it.
struct ReqInfo {
  int32_t tok0;       // first flat token of the request
  int32_t q_len;      // new tokens
  int32_t ctx;        // cached tokens before them
  int32_t npages;     // visible pages of the request's last token (own page + 1)
  int32_t page_base;  // running sum of npages over earlier requests
  int32_t blk_base;   // first inversion block of the request (blocks: KV head x chunk)
  int32_t words;      // 32-row words of one KV group's rows: ceil(q_len * H/H_kv / 32)
  int32_t ch_base;    // first inversion chunk of the request
  int32_t ch_per_bucket;  // chunks per (page, KV head) bucket: ceil(words / kChunkWords)
  int32_t pad[5];
};

// Indexer work item: query tile (<=128 tokens of one request, 1-2 query heads of one KV
// group) against the page chunk [page_begin, page_end).
struct IdxTask {
  int32_t req, g, h0, nh;
  int32_t tok0, ntok, page_begin, page_end;
};

// Forward work item: up to kFwdTaskGroups x 128 entries of one (request, page, KV head)
// bucket, entries [entry_begin, entry_begin + count).
struct FwdTask {
  int32_t bucket, entry_begin, count, pad;
};

// Everything a kernel needs about the plan, passed by value.
struct DevPlan {
  int32_t batch, T, H, Hkv, Hg, D, K, max_pages, num_phys;
  int32_t num_buckets, max_entries, max_fwd_tasks, n_idx_tasks, total_pages;
  int32_t inv_blocks;       // sum over requests of H_kv * ch_per_bucket
  float sm_scale;
  int32_t* status;
  int32_t* counters;        // [2] fwd task count, [4] [5] inversion grid barrier (arrivals,
                            // generation); [0] [1] [3] unused.  Zeroed by the plan upload;
                            // [4] returns to zero when the barrier completes
  const int32_t* tok_pos;   // [T]
  const int32_t* tok_req;   // [T]
  const ReqInfo* reqs;      // [batch]
  const int32_t* page_req;  // [total_pages]: request of each global page slot
  const IdxTask* idx_tasks; // [n_idx_tasks]
  int32_t num_chunks;       // inversion chunks (buckets x chunks per bucket)
  int32_t* chunk_offsets;   // [num_chunks + 1]: entries before each chunk
  int32_t* bucket_offsets;  // [num_buckets + 1]
  int32_t* bucket_totals;   // [num_buckets]: entries per bucket (single-launch inversion)
  int32_t* range_sums;      // [2][inv_blocks]: entries and work items of each block's range of
                            // buckets (single-launch inversion over many buckets)
  int2* entries;            // [max_entries] (row, t * 64 + slot), t = absolute position
  FwdTask* fwd_tasks;       // [max_fwd_tasks]
  // FP16 copies of quantised inputs (null when the plan has none), each rewritten by the call
  // that reads it: Q [T][H][D]; for an indexer over NVFP4 keys, the key tiles of the batch's
  // visible pages in logical order [total_pages][H_kv][128][D] (global page slot = request's
  // page_base + logical page)
  void* qconv;
  void* kconv;
  // top_k <= 16 over long rows: pass 1 of each row split into topk_nseg segments of topk_segg
  // 16-page groups, each segment's 16 largest scores in topk_lists [rows][topk_nseg][16]
  // (topk_nseg 1: no split, topk_lists null)
  // and, per row, the rule pass 2 applies (need, then the bits of ge and eq): topk_meta
  // [rows][3]; and the largest candidate score of each 16-page group: topk_gmax [groups][rows]
  float* topk_lists;
  int32_t* topk_meta;
  float* topk_gmax;
  int32_t topk_nseg, topk_segg;
  // forward, BF16 K/V: when buckets hold few rows (an item of one group or less, so every group
  // waits for its own K/V tiles), the K/V tiles of the item this many items ahead are
  // prefetched into L2 (0: none; the plan sets 1)
  int32_t fwd_prefetch;
};

// Launch of `kern` that may overlap the previous kernel in the stream (programmatic stream
// serialization): its blocks can start, and run their prologue, as the previous kernel's
// blocks leave the SMs; the kernel calls pdl_wait() before it reads that kernel's results.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// Launchers (one per kernel file).  Return cudaSuccess or the launch error.
cudaError_t launch_combine(int64_t rows, int32_t splits, int32_t D, const float* partial,
                           int64_t split_stride, const float* lse, int64_t lse_split_stride,
                           void* out, int64_t out_row_stride, float* out_lse, int32_t* status,
                           cudaStream_t st);
cudaError_t launch_topk(const DevPlan& p, const float* scores, int64_t pitch, int32_t* idx,
                        cudaStream_t st);
cudaError_t launch_inversion(const DevPlan& p, const int32_t* idx, float* lse,
                             int64_t lse_split_stride, cudaStream_t st);
cudaError_t launch_indexer(const DevPlan& p, sps_dtype qt, sps_dtype kt, const void* q,
                           float q_scale, const void* kc, const void* kscales, float k_scale,
                           const int32_t* page_table, float* scores, int64_t pitch,
                           cudaStream_t st);
cudaError_t launch_forward(const DevPlan& p, sps_dtype qt, sps_dtype kvt, const void* q,
                           float q_scale, const void* kc, const void* vc, const void* ks,
                           const void* vs, const int32_t* page_table, float* partial,
                           int64_t split_stride, float* lse, int64_t lse_split_stride,
                           cudaStream_t st);
// The same forward with BF16 partials (split stride in elements).
cudaError_t launch_forward_bf16p(const DevPlan& p, sps_dtype qt, sps_dtype kvt, const void* q,
                                 float q_scale, const void* kc, const void* vc, const void* ks,
                                 const void* vs, const int32_t* page_table, void* partial,
                                 int64_t split_stride, float* lse, int64_t lse_split_stride,
                                 cudaStream_t st);
// The same forward with FP16 partials (split stride in elements).
cudaError_t launch_forward_f16p(const DevPlan& p, sps_dtype qt, sps_dtype kvt, const void* q,
                                float q_scale, const void* kc, const void* vc, const void* ks,
                                const void* vs, const int32_t* page_table, void* partial,
                                int64_t split_stride, float* lse, int64_t lse_split_stride,
                                cudaStream_t st);
// The pages' Q8KV4 route: K rounded to E4M3, S = Q K^T on the FP8 tensor core (D = 128).
cudaError_t launch_forward_fp8qk(const DevPlan& p, sps_dtype qt, sps_dtype kvt, const void* q,
                                 float q_scale, const void* kc, const void* vc, const void* ks,
                                 const void* vs, const int32_t* page_table, float* partial,
                                 int64_t split_stride, float* lse, int64_t lse_split_stride,
                                 cudaStream_t st);
// The combine over BF16 partials.
cudaError_t launch_combine_bf16p(int64_t rows, int32_t splits, int32_t D, const void* partial,
                                 int64_t split_stride, const float* lse, int64_t lse_split_stride,
                                 void* out, int64_t out_row_stride, float* out_lse,
                                 int32_t* status, cudaStream_t st);

// The combine over FP16 partials.
cudaError_t launch_combine_f16p(int64_t rows, int32_t splits, int32_t D, const void* partial,
                                int64_t split_stride, const float* lse, int64_t lse_split_stride,
                                void* out, int64_t out_row_stride, float* out_lse,
                                int32_t* status, cudaStream_t st);

// Chunked-prefill append of the new tokens' K/V into the paged cache (BF16 copy or NVFP4
// quantisation), per-tensor E4M3 quantisation, and the BF16 absmax behind its scale.
cudaError_t launch_kv_append(const DevPlan& p, bool nvfp4, const void* knew, const void* vnew,
                             const int32_t* page_table, void* kc, void* vc, void* ks, void* vs,
                             cudaStream_t st);
cudaError_t launch_quantize_e4m3(const void* in, int64_t n, float scale, void* out,
                                 cudaStream_t st);
cudaError_t launch_absmax_bf16(const void* in, int64_t n, float* out, cudaStream_t st);

// Copy of n bytes from device-accessible page-locked host memory (src) to device memory (dst),
// both 16-byte aligned, by a kernel rather than the copy engine.
cudaError_t launch_staged_copy(const void* src, void* dst, size_t n, cudaStream_t st);

// One-block kernel whose bounded wait on a never-arrived mbarrier must time out.
cudaError_t launch_wait_timeout(int32_t* status, int64_t limit_ns, cudaStream_t st);
cudaError_t launch_barrier_timeout(unsigned int* bar, int32_t* status, int64_t limit_ns,
                                   cudaStream_t st);

// Exact E4M3 / NVFP4 -> FP16 conversion of n elements (n % 16 == 0).
cudaError_t launch_dequant(sps_dtype dt, const void* in, const void* scales, int64_t n,
                           void* out, cudaStream_t st);
// NVFP4 key tiles of the batch's visible pages, through the page table, into the plan's
// logical-order FP16 copy (DevPlan::kconv).
cudaError_t launch_dequant_pages(const DevPlan& p, const void* codes, const void* scales,
                                 const int32_t* page_table, void* out, cudaStream_t st);
// NVFP4 -> E4M3 codes: each exact code x scale product rounded to nearest even E4M3
// (saturating), the pages' QMUL4 dequant.
cudaError_t launch_dequant_e4m3(const void* in, const void* scales, int64_t n, void* out,
                                cudaStream_t st);

// Tensor-map encoding through the driver entry point (no link against libcuda).
bool encode_tmap_2d(void* map, int dtype_code, void* base, uint64_t inner, uint64_t outer,
                    uint64_t outer_stride_bytes, uint32_t box_inner, uint32_t box_outer,
                    bool swizzle128);
bool encode_tmap_3d(void* map, int dtype_code, void* base, uint64_t d0, uint64_t d1,
                    uint64_t d2, uint64_t s1_bytes, uint64_t s2_bytes, uint32_t b0, uint32_t b1,
                    uint32_t b2, bool swizzle128);
// FP32 elements, 64-byte swizzle (box_inner * 4 == 64): the top-k score tiles.
bool encode_tmap_2d_f32_sw64(void* map, const void* base, uint64_t inner, uint64_t outer,
                             uint64_t outer_stride_bytes, uint32_t box_inner,
                             uint32_t box_outer);
int num_sms();

}  // namespace sps
