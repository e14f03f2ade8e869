/*
 * sparse_prefill.h -- C ABI of the GB300 (sm_103a) paged block-sparse prefill attention
 * library (libsps.so).
 *
 * The method, in four steps (terms as on the pages "MSA PR 21: Q8KV4 paged sparse prefill"
 * and "MSA PR 36: Q8KV8 prefill indexer"):
 *
 *   1. indexer_scores     every causally visible 128-token KV page of every (query token,
 *                         query head) row gets the score max_{visible keys j} q.k_j in FP32.
 *   2. topk_select        each row keeps k pages: its own page always, the others by score
 *                         (ties to the lower page index).
 *   3. sparse_prefill_fwd one pass per (page, KV head, query split): each selected page yields
 *                         a partial attention output plus its log-sum-exp (LSE), written into
 *                         a split-strided FP32 partial buffer.  Only the row's own page is
 *                         causally masked; K/V are read through a page table.
 *   4. partial_combine    every row's k partials are merged by LSE into a BF16 output.
 *
 * Terms.  T = total query tokens of the batch (requests concatenated), H = query heads,
 * H_kv = KV heads (H % H_kv == 0; query head h reads KV head h / (H / H_kv)), D = head_dim,
 * page = 128 tokens.  A ROW is r = token * H + h.  Request b's token i sits at absolute
 * position t = ctx_lens[b] + i; its own page is o = t / 128; it may see pages 0..o and, inside
 * the own page, keys with position <= t.
 *
 * Memory.  The caller owns every buffer.  The library never allocates device memory; device
 * pointers below must be device-accessible allocations on the current device.  "host" marks
 * host pointers.  The plan (sps_plan) is an opaque host object owned by the caller.
 *
 * Errors.  Every call returns an sps_status.  Arguments are validated on the host first
 * (null pointers, dtypes, 16-byte alignment where TMA reads, strides, pitches, limits); a
 * rejected call launches nothing and returns SPS_EINVAL or SPS_EUNSUPPORTED.  A failed CUDA
 * launch returns SPS_ECUDA.  Errors found on the device (a page-table entry out of range, a
 * selected page the row cannot see, a bounded wait that timed out) never trap: the kernel
 * records the first such code in a device status word and exits; read it with
 * sps_read_device_status.  sps_last_error() gives a message for the last failing call on the
 * calling thread.  No C++ exception crosses this interface.
 *
 * Streams.  All device work is asynchronous on the given stream (NULL = legacy default
 * stream).  Calls that share a workspace must be ordered on one stream.
 */
#ifndef SPARSE_PREFILL_H
#define SPARSE_PREFILL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* sps_stream_t; /* a cudaStream_t */

typedef enum {
  SPS_OK = 0,
  SPS_EINVAL = 1,          /* bad argument (message in sps_last_error) */
  SPS_EUNSUPPORTED = 2,    /* valid but not implemented (dtype pair, head_dim, ...) */
  SPS_ENOSPACE = 3,        /* workspace smaller than sparse_prefill_plan asked for */
  SPS_ECUDA = 4,           /* a CUDA runtime/driver call failed */
  SPS_EDEVICE = 5          /* the device status word holds an error */
} sps_status;

typedef enum { SPS_BF16 = 0, SPS_FP16 = 1, SPS_E4M3 = 2, SPS_NVFP4 = 3 } sps_dtype;

/* Device status codes (read with sps_read_device_status). */
enum {
  SPS_DEV_OK = 0,
  SPS_DEV_TIMEOUT = 1,     /* a bounded wait gave up */
  SPS_DEV_BAD_PAGE = 2,    /* page_table entry outside [0, num_phys_pages) */
  SPS_DEV_BAD_INDEX = 3,   /* a selected page outside [0, own page] of its row */
  SPS_DEV_OVERFLOW = 4     /* more work items than the plan sized the workspace for */
};

/*
 * Problem description (host memory; copied by sparse_prefill_plan).
 *
 *   batch              number of requests, >= 1
 *   q_lens, ctx_lens   host arrays [batch]: new query tokens and cached context tokens per
 *                      request (the chunk's own K/V are already in the cache)
 *   num_q_heads        H;  num_kv_heads: H_kv (H % H_kv == 0)
 *   head_dim           D: 64 or 128
 *   page_size          must be 128
 *   top_k              k: 1..64 pages kept per row
 *   max_pages_per_req  row length of the page table, >= every request's visible page count;
 *                      at most 8192 (1M tokens) with top_k <= 16 and 1024 (128K tokens) with
 *                      larger top_k, else SPS_EUNSUPPORTED
 *   num_phys_pages     number of physical pages in the K/V caches
 *   q_dtype / kv_dtype           attention inputs: BF16/BF16 or E4M3/NVFP4
 *   idx_q_dtype / idx_k_dtype    indexer inputs: BF16/BF16, E4M3/E4M3 or E4M3/NVFP4
 *   softmax_scale      multiplier of q.k inside the softmax (typically 1/sqrt(D))
 */
typedef struct {
  int32_t batch;
  const int32_t* q_lens;
  const int32_t* ctx_lens;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t page_size;
  int32_t top_k;
  int32_t max_pages_per_req;
  int32_t num_phys_pages;
  sps_dtype q_dtype;
  sps_dtype kv_dtype;
  sps_dtype idx_q_dtype;
  sps_dtype idx_k_dtype;
  float softmax_scale;
} sps_problem;

typedef struct sps_plan sps_plan;

/* Sizes and workspace offsets of a plan (for inspection and tests).  Offsets are bytes from
 * the workspace base. */
typedef struct {
  int64_t num_tokens;        /* T */
  int64_t num_rows;          /* T * H */
  int64_t num_buckets;       /* (request, visible page, KV head) triples */
  int64_t max_entries;       /* num_rows * top_k */
  int64_t indexer_tasks;     /* indexer work items */
  int64_t max_fwd_tasks;     /* upper bound on forward work items */
  int64_t workspace_bytes;
  int64_t off_status;        /* int32 device status word */
  int64_t off_tok_pos;       /* int32 [T]: absolute position of each token */
  int64_t off_tok_req;       /* int32 [T]: request of each token */
  int64_t off_bucket_offsets;/* int32 [num_buckets + 1]: CSR offsets of the inversion */
  int64_t off_entries;       /* int32 pairs [max_entries]: (row, t*64 + slot), rows ascending per
                                bucket, t = absolute position of the row's token */
  int64_t off_fwd_task_count;/* int32: number of forward work items built on the device */
} sps_plan_info;

/*
 * sparse_prefill_plan -- host only, no device work.
 * Validates the problem, derives per-token metadata, the indexer's work list (query tile x
 * page chunk; the chunk shrinks from 128 to 8 pages until the work fills the GPU, as the
 * adaptive page chunk of "MSA PR 36", Changes) and the workspace layout (one workspace may
 * serve every call of this plan in order on one stream, as the PrefillWorkspace of "MSA PR
 * 21", Place the partials by memory locality domain).
 *   plan            out: new plan, free with sps_plan_destroy
 *   workspace_bytes out: device workspace size the plan's calls need (256-byte aligned)
 * Returns SPS_EINVAL / SPS_EUNSUPPORTED for a problem it cannot run.
 */
sps_status sparse_prefill_plan(const sps_problem* problem, sps_plan** plan,
                               size_t* workspace_bytes);

void sps_plan_destroy(sps_plan* plan);

sps_status sps_plan_get_info(const sps_plan* plan, sps_plan_info* info);

/*
 * sps_plan_upload -- copies the plan's metadata into `workspace` (device, >= workspace_bytes,
 * 256-byte aligned) on `stream` with one copy that also clears the device status word and
 * counters.  Call once per (plan, workspace) before the other plan calls, on the same stream,
 * and outside CUDA graph capture; call it again after the status word has recorded an error.
 * The bytes go through a mapped page-locked staging ring of the library (allocated on the first
 * call; a region is reused only after the event behind its copy has completed) and a small
 * copy kernel on `stream` reads them from there, so the upload never waits for the caller's
 * own host<->device transfers on other streams, and the plan may be destroyed as soon as the
 * call returns.  Where the ring cannot be allocated or mapped it is a plain asynchronous copy.
 */
sps_status sps_plan_upload(const sps_plan* plan, void* workspace, size_t workspace_bytes,
                           sps_stream_t stream);

/*
 * indexer_scores -- step 1 ("MSA PR 36", Changes: per-page max by TMEM load-and-reduce;
 * Wrapper API: caller-owned score buffer).
 *   q_idx        device [T][H][D] in idx_q_dtype (E4M3: one byte per element)
 *   q_scale      per-tensor multiplier of the decoded q (1 for BF16)
 *   k_idx_cache  device [num_phys_pages][H_kv][128][D] in idx_k_dtype; NVFP4: packed codes
 *                [..][128][D/2], the even element in the low nibble
 *   k_idx_scales device [num_phys_pages][H_kv][128][D/16] E4M3 (NVFP4 only, else NULL)
 *   k_scale      per-tensor multiplier of the decoded k (1 for BF16 and NVFP4)
 *   page_table   device int32 [batch][max_pages_per_req], logical -> physical page
 *   scores       device FP32 [T*H][score_pitch]; score_pitch >= max_pages_per_req, 4-aligned
 * Writes scores[r][p] = q_scale * k_scale * max_{j in page p, j <= t} (q_r . k_j) for every
 * p <= o(r); every other entry is left untouched.  Accumulation is FP32.
 */
sps_status indexer_scores(const sps_plan* plan, const void* q_idx, float q_scale,
                          const void* k_idx_cache, const void* k_idx_scales, float k_scale,
                          const int32_t* page_table, float* scores, int64_t score_pitch,
                          void* workspace, sps_stream_t stream);

/*
 * topk_select -- step 2 (the method's page selection, with the row's own page -- the one page
 * "MSA PR 21", K1 Softmax, masks causally -- always kept; bitwise-stable selection, "MSA PR
 * 36", Kernel performance table: top-k bitwise identical).
 *   scores  device FP32 [T*H][score_pitch] as written by indexer_scores (entries p <= o read)
 *   idx     device int32 [T*H][top_k] out: the selected pages of each row in ascending page
 *           order, padded with -1 when the row sees fewer than top_k pages.
 * The own page o is always kept; the other min(top_k, o+1) - 1 are the best by (score
 * descending, page ascending), with -0.0 equal to +0.0.  NaN scores are outside the contract.
 * Any score_pitch >= max_pages_per_req gives the same result; with top_k <= 16 a pitch that is
 * a multiple of 4 on a 16-byte aligned buffer is the fast layout (the rows arrive by tensor
 * copies), other pitches are read by per-thread loads.
 */
sps_status topk_select(const sps_plan* plan, const float* scores, int64_t score_pitch,
                       int32_t* idx, void* workspace, sps_stream_t stream);

/*
 * sparse_prefill_fwd -- step 3 ("MSA PR 21", K1: one CTA per (page, head, query split),
 * groups of 128 query rows, own-page-only causal mask; K1 also reads the split stride).
 *   q            device [T][H][D], q_dtype (BF16, or E4M3 with q_scale)
 *   k_cache, v_cache  device [num_phys_pages][H_kv][128][D] (BF16), or NVFP4 codes
 *                [..][128][D/2] with k_scales / v_scales [..][128][D/16] E4M3
 *   page_table   device int32 [batch][max_pages_per_req]
 *   idx          device int32 [T*H][top_k] from topk_select (or any selection obeying its
 *                contract: ascending, -1 padded, pages <= own page)
 *   partial      device FP32; element (slot s, row r, dim d) at
 *                partial[s * split_stride + r * D + d]; split_stride >= T*H*D, multiple of 4
 *   lse          device FP32; (s, r) at lse[s * lse_split_stride + r]; stride >= T*H
 * For every row r and slot s with page p = idx[r][s] >= 0: the softmax over the page's keys
 * j <= t of softmax_scale * q.k_j gives partial = sum_j p_j v_j / l (FP32) and
 * lse = m + ln(l) (natural log).  Empty slots (idx = -1) get lse = -inf and their partial is
 * not written.  P is rounded to FP16 for the P.V product; V is converted to FP16 (exact for
 * NVFP4 and for BF16 values in the FP16 normal range).
 */
sps_status sparse_prefill_fwd(const sps_plan* plan, const void* q, float q_scale,
                              const void* k_cache, const void* v_cache, const void* k_scales,
                              const void* v_scales, const int32_t* page_table,
                              const int32_t* idx, float* partial, int64_t split_stride,
                              float* lse, int64_t lse_split_stride, void* workspace,
                              sps_stream_t stream);

/*
 * partial_combine -- step 4 ("MSA PR 21", Combine: one streaming kernel; a CTA owns
 * consecutive rows, the splits stream through a shared-memory ring of bulk copies).
 * Plan-free so it can run on any partial buffer.
 *   rows, splits, head_dim  R, S (1..64), D (64 or 128)
 *   partial   device FP32, (s, r, d) at partial[s * split_stride + r * head_dim + d];
 *             16-byte aligned, split_stride a multiple of 4 and >= rows * head_dim
 *   lse       device FP32, (s, r) at lse[s * lse_split_stride + r], lse_split_stride >= rows
 *   out_bf16  device BF16, row r at out_bf16 + r * out_row_stride (elements); 16-byte aligned,
 *             out_row_stride a multiple of 8
 *   out_lse   device FP32 [rows] or NULL
 *   dev_status device int32 status word or NULL (a wait that times out records there)
 * out[r] = sum_s w_s partial_s / sum_s w_s with w_s = exp(lse_s - max_s lse_s); a slot with
 * lse = -inf gets weight 0 by selection (its partial is never read); a row whose slots are
 * all -inf gets out = 0 and out_lse = -inf.  FP32 accumulation, BF16 round-to-nearest output.
 */
sps_status partial_combine(int64_t rows, int32_t splits, int32_t head_dim, const float* partial,
                           int64_t split_stride, const float* lse, int64_t lse_split_stride,
                           void* out_bf16, int64_t out_row_stride, float* out_lse,
                           int32_t* dev_status, sps_stream_t stream);

/*
 * sparse_prefill_fwd_bf16 / partial_combine_bf16 -- the same two steps with the partial
 * outputs stored as BF16, the storage the pages keep ("MSA PR 21", Combine: keep BF16/FP16
 * partials and outputs only).  It halves the forward's writes and the combine's reads.
 *   partial_bf16  device BF16; element (s, r, d) at partial_bf16[s * split_stride + r * D + d]
 *                 (elements); 16-byte aligned, split_stride a multiple of 8 and >= rows * D
 * Every other argument, the LSE and the output are those of sparse_prefill_fwd and
 * partial_combine.  The forward rounds each normalised partial to BF16 (round to nearest
 * even); the combine widens them exactly to FP32 and accumulates in FP32.
 */
sps_status sparse_prefill_fwd_bf16(const sps_plan* plan, const void* q, float q_scale,
                                   const void* k_cache, const void* v_cache,
                                   const void* k_scales, const void* v_scales,
                                   const int32_t* page_table, const int32_t* idx,
                                   void* partial_bf16, int64_t split_stride, float* lse,
                                   int64_t lse_split_stride, void* workspace,
                                   sps_stream_t stream);
sps_status partial_combine_bf16(int64_t rows, int32_t splits, int32_t head_dim,
                                const void* partial_bf16, int64_t split_stride, const float* lse,
                                int64_t lse_split_stride, void* out_bf16, int64_t out_row_stride,
                                float* out_lse, int32_t* dev_status, sps_stream_t stream);

/*
 * sparse_prefill_fwd_f16 / partial_combine_f16 -- the same two steps with the partial outputs
 * stored as FP16, the other 16-bit storage the pages name ("MSA PR 21", Combine: keep
 * BF16/FP16 partials).  FP16 carries 11 significant bits against BF16's 8, so its rounding
 * adds far less to the output error; its range is that of the FP16 V operand the forward
 * already uses (|v| < 65504), which bounds every partial, a convex combination of V rows.
 *   partial_f16  device FP16; element (s, r, d) at partial_f16[s * split_stride + r * D + d]
 *                (elements); 16-byte aligned, split_stride a multiple of 8 and >= rows * D
 * Every other argument, the LSE and the output are those of sparse_prefill_fwd and
 * partial_combine.  The forward rounds each normalised partial to FP16 (nearest even); the
 * combine widens them exactly to FP32 and accumulates in FP32.
 */
sps_status sparse_prefill_fwd_f16(const sps_plan* plan, const void* q, float q_scale,
                                  const void* k_cache, const void* v_cache, const void* k_scales,
                                  const void* v_scales, const int32_t* page_table,
                                  const int32_t* idx, void* partial_f16, int64_t split_stride,
                                  float* lse, int64_t lse_split_stride, void* workspace,
                                  sps_stream_t stream);
sps_status partial_combine_f16(int64_t rows, int32_t splits, int32_t head_dim,
                               const void* partial_f16, int64_t split_stride, const float* lse,
                               int64_t lse_split_stride, void* out_bf16, int64_t out_row_stride,
                               float* out_lse, int32_t* dev_status, sps_stream_t stream);

/*
 * sparse_prefill_fwd_fp8qk -- the pages' own Q8KV4 route ("MSA PR 21: Q8KV4 paged sparse
 * prefill": QMUL4 dequant, whose only rounding is the final conversion of the code x scale
 * product to E4M3, and FP8 UMMA for Q K^T): the same arguments and outputs as
 * sparse_prefill_fwd for a plan with E4M3 Q, NVFP4 K/V and head_dim 128.  K is rounded to
 * E4M3 (nearest even, saturating), S = Q K^T runs on the FP8 tensor core (FP32 accumulation);
 * V stays exact (FP16) for P.V.  Its results match the definition on the E4M3-rounded K, not
 * on the exact products; other plans return SPS_EUNSUPPORTED.
 */
sps_status sparse_prefill_fwd_fp8qk(const sps_plan* plan, const void* q, float q_scale,
                                    const void* k_cache, const void* v_cache,
                                    const void* k_scales, const void* v_scales,
                                    const int32_t* page_table, const int32_t* idx, float* partial,
                                    int64_t split_stride, float* lse, int64_t lse_split_stride,
                                    void* workspace, sps_stream_t stream);

/*
 * sps_kv_append -- the chunked-prefill step before indexer_scores: writes the batch's new
 * tokens' K and V into the paged cache (the formats of "MSA PR 21: Q8KV4 paged sparse
 * prefill": E4M3 query, NVFP4 K/V with an E4M3 scale per 16 elements; the pages fix no
 * rounding for this step).  Token i of request b (position t = ctx_len + i, flat token order
 * of the plan) goes to physical page page_table[b][t / 128], slot t % 128, of every KV head.
 *   k_new, v_new  device BF16 [T][H_kv][D], 16-byte aligned
 *   k_cache, v_cache  the plan's kv_dtype: BF16 [num_phys_pages][H_kv][128][D] (bits copied),
 *                 or NVFP4 codes [..][128][D/2] with k_scales / v_scales [..][128][D/16]:
 *                 per 16-element block scale = E4M3(absmax / 6), code = E2M1(x / scale), both
 *                 divisions in FP32, conversions to nearest even and saturating; a block whose
 *                 scale rounds to zero gets zero codes
 *   workspace     the plan's uploaded workspace (token positions); a page-table entry outside
 *                 [0, num_phys_pages) sets SPS_DEV_BAD_PAGE and skips the row
 * Slots not written keep their contents.
 */
sps_status sps_kv_append(const sps_plan* plan, const void* k_new, const void* v_new,
                         const int32_t* page_table, void* k_cache, void* v_cache, void* k_scales,
                         void* v_scales, void* workspace, sps_stream_t stream);

/*
 * sps_quantize_e4m3 -- per-tensor E4M3 query codes: codes[i] = E4M3(x[i] / scale) (FP32
 * division, nearest even, saturating at 448); x BF16, n a multiple of 16, both 16-byte
 * aligned, scale finite and > 0 (the pages' E4M3 query with its per-tensor scale).
 * sps_absmax_bf16 -- *absmax (device FP32) = max |x[i]| over n BF16 values (n a multiple of
 * 16), e.g. for scale = absmax / 448.
 */
sps_status sps_quantize_e4m3(const void* x_bf16, int64_t n, float scale, void* codes,
                             sps_stream_t stream);
sps_status sps_absmax_bf16(const void* x_bf16, int64_t n, float* absmax, sps_stream_t stream);

/*
 * sps_dequantize -- exact conversion of quantised inputs to FP16 (the dequant step of "MSA PR
 * 21: Q8KV4 paged sparse prefill", Build the prefill for SM107: an E2M1 code times its E4M3
 * scale is exact in FP16).  The indexer and the forward run it internally on quantised plans.
 *   in_dtype  SPS_E4M3: `in` holds n one-byte codes (16-byte aligned);
 *             SPS_NVFP4: `in` holds n/2 bytes of packed E2M1 codes, the even element in the
 *             low nibble (8-byte aligned), and `scales` n/16 E4M3 scales, one per 16
 *             consecutive elements
 *   n         number of elements, a multiple of 16
 *   out_f16   device FP16 [n] (16-byte aligned): code (E4M3), or code x scale (NVFP4), with no
 *             per-tensor scale applied.  Every result is exact (NaN codes give NaN).
 */
sps_status sps_dequantize(sps_dtype in_dtype, const void* in, const void* scales, int64_t n,
                          void* out_f16, sps_stream_t stream);

/*
 * sparse_prefill_fwd_noalloc -- sparse_prefill_fwd for callers that cannot allocate device
 * memory.  (No counterpart on the pages: this is an interface convenience of this library.)
 *
 * Who needs it: code that must not call cudaMalloc or hand out device buffers of its own --
 * for example a plug-in called from inside another runtime whose memory pool it cannot reach,
 * a serving loop that forbids new device allocations once it is warm, or a C caller with a
 * fixed device-memory budget.  Such a caller can still pass its inputs and outputs, but it has
 * no workspace to give; this variant keeps the forward's scratch (the plan's metadata and the
 * page -> row inversion) in a fixed array inside the library instead.
 *
 * Arguments are those of sparse_prefill_fwd without the workspace, plus
 *   dev_status  device int32 or NULL: where the kernels record device-side errors
 *               (SPS_DEV_*; the caller clears it).  With NULL such errors go unreported.
 * The plan needs no sps_plan_upload: this call copies the plan's metadata into the array
 * (through the library's staging ring when an earlier call has allocated it, else as a plain
 * asynchronous copy from the plan's own host memory; it never allocates the ring).
 *
 * Rules.
 *   - The array holds 48 MiB per device and every GPU that loads the library keeps it until
 *     the process exits.  A plan whose workspace_bytes exceeds 48 MiB is rejected with
 *     SPS_ENOSPACE (for example 16K tokens x 32 heads x top-16 needs more); split the batch or
 *     use sparse_prefill_fwd.
 *   - The first call on a device looks up the array's device address (once per device, with
 *     that device current); make that first call before any stream capture on the device.
 *   - All calls on a device share the one array, and it keeps the last call's contents (each
 *     call clears and rewrites what it needs).  Calls whose work overlaps on the GPU -- on
 *     different streams, or from different host threads -- race and corrupt each other; order
 *     them on one stream.
 *   - No cudaMalloc, cudaFree or other allocating routine is called.
 */
sps_status sparse_prefill_fwd_noalloc(const sps_plan* plan, const void* q, float q_scale,
                                      const void* k_cache, const void* v_cache,
                                      const void* k_scales, const void* v_scales,
                                      const int32_t* page_table, const int32_t* idx,
                                      float* partial, int64_t split_stride, float* lse,
                                      int64_t lse_split_stride, int32_t* dev_status,
                                      sps_stream_t stream);

/*
 * sps_check_wait_timeout -- health check of the failure path every kernel relies on: a
 * one-block kernel waits on an mbarrier that nothing ever arrives on, through the same bounded
 * wait the pipelines use (their limit is 2 s; here `limit_ns`, 1 ms .. 10 s).  The wait gives
 * up, records SPS_DEV_TIMEOUT in *dev_status (a device int32 the caller cleared) and the kernel
 * returns; the context stays usable.  Asynchronous on `stream`.  ("MSA PR 36", Changes, notes a
 * hang fixed in the indexer's K loader; here no wait can hang.)
 */
sps_status sps_check_wait_timeout(int64_t limit_ns, int32_t* dev_status, sps_stream_t stream);

/*
 * sps_check_barrier_timeout -- the same check for the grid barrier of the library's
 * cooperative launch (the single-launch inversion inside sparse_prefill_fwd): two blocks, one
 * of which leaves without arriving, so the other's barrier wait must give up after
 * `limit_ns` (1 ms .. 10 s), record SPS_DEV_TIMEOUT in *dev_status and return.
 *   dev_barrier  device uint32[2], zeroed by the caller (the barrier's counters)
 */
sps_status sps_check_barrier_timeout(int64_t limit_ns, uint32_t* dev_barrier,
                                     int32_t* dev_status, sps_stream_t stream);

/*
 * sps_read_device_status -- synchronous: waits for the device, then copies the plan
 * workspace's status word into *code (SPS_DEV_*).  Returns SPS_EDEVICE when it is non-zero.
 */
sps_status sps_read_device_status(const sps_plan* plan, const void* workspace, int32_t* code);

/* Message of the last failing call on the calling thread ("" if none). */
const char* sps_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* SPARSE_PREFILL_H */
