// host.cpp -- C ABI of libsps: problem validation, the plan (per-token metadata, indexer work
// list, workspace layout), the metadata upload (through a page-locked staging ring), and the
// argument checks in front of every kernel launch.  No device memory is ever allocated here.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "sps_internal.h"

using namespace sps;

namespace {

thread_local std::string g_err;

sps_status fail(sps_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_err = buf;
  return st;
}

sps_status cuda_fail(cudaError_t e, const char* what) {
  return fail(SPS_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

inline int64_t align_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }
inline bool aligned(const void* p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

// Page-locked staging for the plan-metadata uploads.  The bytes are written into a mapped
// page-locked ring and a copy kernel on the caller's stream reads them from there: a copy from
// pageable memory makes the GPU wait while the driver stages it, and a DMA on the copy engine
// queues behind the caller's own transfers on other streams (for instance the next batch's
// inputs).  One ring per process, allocated on first use (by the calls that may allocate) and
// never freed; a region is reused only after the event recorded behind its copy has completed.
// Uploads that do not fit, uploads into a stream being captured into a graph (the graph must
// keep reading the plan's own copy), a failed page-locked allocation or mapping, or a call
// that may not allocate while the ring does not exist yet copy from pageable memory instead.
class StagingRing {
 public:
  cudaError_t upload(void* dst, const void* src, size_t n, cudaStream_t s, bool may_alloc) {
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cap) != cudaSuccess || cap != cudaStreamCaptureStatusNone) {
      (void)cudaGetLastError();
      return cudaMemcpyAsync(dst, src, n, cudaMemcpyHostToDevice, s);
    }
    std::lock_guard<std::mutex> lock(mu_);
    if (!buf_ && !failed_ && may_alloc) {
      if (cudaHostAlloc(reinterpret_cast<void**>(&buf_), kBytes,
                        cudaHostAllocPortable | cudaHostAllocMapped) != cudaSuccess) {
        buf_ = nullptr;
        failed_ = true;
        (void)cudaGetLastError();
      } else if (cudaHostGetDevicePointer(reinterpret_cast<void**>(&dbuf_), buf_, 0) !=
                 cudaSuccess) {
        dbuf_ = nullptr;  // not mapped: DMA from the ring instead
        (void)cudaGetLastError();
      }
    }
    if (!buf_ || n > kBytes / 2) return cudaMemcpyAsync(dst, src, n, cudaMemcpyHostToDevice, s);
    size_t off = head_;
    if (off + n > kBytes) off = 0;
    // wait for the copies still reading [off, off + n)
    while (!live_.empty() && overlaps(live_.front(), off, off + n)) {
      cudaError_t e = cudaEventSynchronize(live_.front().ev);
      free_ev_.push_back(live_.front().ev);
      live_.erase(live_.begin());
      if (e != cudaSuccess) return e;
    }
    memcpy(buf_ + off, src, n);
    cudaError_t e = (dbuf_ && aligned(dst, 16))
                        ? launch_staged_copy(dbuf_ + off, dst, n, s)
                        : cudaMemcpyAsync(dst, buf_ + off, n, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return e;
    cudaEvent_t ev;
    if (!free_ev_.empty()) {
      ev = free_ev_.back();
      free_ev_.pop_back();
    } else if ((e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming)) != cudaSuccess) {
      return cudaStreamSynchronize(s);  // no event: the region is safe once the copy is done
    }
    if ((e = cudaEventRecord(ev, s)) != cudaSuccess) {
      cudaEventDestroy(ev);
      return cudaStreamSynchronize(s);
    }
    live_.push_back({off, off + n, ev});
    head_ = (size_t)align_up((int64_t)(off + n), 256);
    return cudaSuccess;
  }

 private:
  struct Live {
    size_t begin, end;
    cudaEvent_t ev;
  };
  static bool overlaps(const Live& l, size_t b, size_t e) { return l.begin < e && b < l.end; }
  static constexpr size_t kBytes = 16u << 20;
  std::mutex mu_;
  uint8_t* buf_ = nullptr;   // host address of the ring
  uint8_t* dbuf_ = nullptr;  // its device address (NULL: not mapped)
  bool failed_ = false;
  size_t head_ = 0;
  std::vector<Live> live_;  // in ring order
  std::vector<cudaEvent_t> free_ev_;
};
StagingRing g_staging;

}  // namespace

struct sps_plan {
  sps_problem pb;                 // copy (host arrays below)
  std::vector<int32_t> q_lens, ctx_lens;
  std::vector<ReqInfo> reqs;
  std::vector<int32_t> page_req;  // [total_pages]
  std::vector<IdxTask> idx_tasks;
  int64_t T = 0, R = 0, num_buckets = 0, max_entries = 0, max_fwd_tasks = 0;
  int64_t total_pages = 0, num_chunks = 0, inv_blocks = 0;
  // workspace layout (bytes)
  int64_t off_status = 0, off_counters = 0, off_tok_pos = 0, off_tok_req = 0, off_reqs = 0,
          off_page_req = 0, off_idx_tasks = 0, off_chunk_offsets = 0, off_bucket_totals = 0,
          off_range_sums = 0,
          off_qconv = -1, off_kconv = -1,
          off_bucket_offsets = 0, off_entries = 0, off_fwd_tasks = 0, off_topk_lists = -1,
          off_topk_meta = -1, off_topk_gmax = -1,
          ws_bytes = 0;
  int64_t fwd_ws_bytes = 0;  // the part the forward uses (the no-allocation forward's need)
  int32_t topk_nseg = 1, topk_segg = 0;
  int32_t fwd_prefetch = 0;
  int64_t upload_bytes = 0;  // [0, upload_bytes) of the workspace comes from `blob`
  std::vector<uint8_t> blob;
};

namespace {

sps_status validate_problem(const sps_problem* p) {
  if (!p) return fail(SPS_EINVAL, "problem is NULL");
  if (p->batch < 1) return fail(SPS_EINVAL, "batch must be >= 1 (got %d)", p->batch);
  if (!p->q_lens || !p->ctx_lens) return fail(SPS_EINVAL, "q_lens/ctx_lens must be host arrays");
  if (p->page_size != kPage) return fail(SPS_EUNSUPPORTED, "page_size must be 128");
  if (p->head_dim != 64 && p->head_dim != 128)
    return fail(SPS_EUNSUPPORTED, "head_dim must be 64 or 128 (got %d)", p->head_dim);
  if (p->num_q_heads < 1 || p->num_kv_heads < 1 || p->num_q_heads % p->num_kv_heads)
    return fail(SPS_EINVAL, "num_q_heads (%d) must be a positive multiple of num_kv_heads (%d)",
                p->num_q_heads, p->num_kv_heads);
  if (p->top_k < 1 || p->top_k > kMaxTopK)
    return fail(SPS_EINVAL, "top_k must be in [1, %d] (got %d)", kMaxTopK, p->top_k);
  if (p->num_phys_pages < 1) return fail(SPS_EINVAL, "num_phys_pages must be >= 1");
  if (!(p->softmax_scale > 0.f) || !std::isfinite(p->softmax_scale))
    return fail(SPS_EINVAL, "softmax_scale must be finite and > 0");
  bool attn_ok = (p->q_dtype == SPS_BF16 && p->kv_dtype == SPS_BF16) ||
                 (p->q_dtype == SPS_E4M3 && p->kv_dtype == SPS_NVFP4);
  if (!attn_ok) return fail(SPS_EUNSUPPORTED, "attention dtypes must be BF16/BF16 or E4M3/NVFP4");
  bool idx_ok = (p->idx_q_dtype == SPS_BF16 && p->idx_k_dtype == SPS_BF16) ||
                (p->idx_q_dtype == SPS_E4M3 && p->idx_k_dtype == SPS_E4M3) ||
                (p->idx_q_dtype == SPS_E4M3 && p->idx_k_dtype == SPS_NVFP4);
  if (!idx_ok)
    return fail(SPS_EUNSUPPORTED, "indexer dtypes must be BF16/BF16, E4M3/E4M3 or E4M3/NVFP4");
  if (p->idx_q_dtype == SPS_E4M3 && p->idx_k_dtype == SPS_E4M3 && p->head_dim != 128)
    return fail(SPS_EUNSUPPORTED, "the E4M3 x E4M3 indexer needs head_dim 128");
  int64_t T = 0;
  for (int b = 0; b < p->batch; ++b) {
    if (p->q_lens[b] < 0 || p->ctx_lens[b] < 0)
      return fail(SPS_EINVAL, "request %d: negative q_len/ctx_len", b);
    int64_t last = (int64_t)p->ctx_lens[b] + p->q_lens[b] - 1;
    if (last >= (int64_t)1 << 24) return fail(SPS_EINVAL, "request %d: sequence too long", b);
    int64_t np = p->q_lens[b] > 0 ? last / kPage + 1 : 0;
    if (np > p->max_pages_per_req)
      return fail(SPS_EINVAL, "request %d needs %lld pages > max_pages_per_req %d", b,
                  (long long)np, p->max_pages_per_req);
    T += p->q_lens[b];
  }
  if (T < 1) return fail(SPS_EINVAL, "the batch has no query tokens");
  int64_t R = T * p->num_q_heads;
  if (R * p->top_k >= ((int64_t)1 << 31) || R * p->head_dim >= ((int64_t)1 << 40))
    return fail(SPS_EUNSUPPORTED, "batch too large (rows x top_k must stay below 2^31)");
  const int page_cap = p->top_k <= 16 ? kMaxPagesPerReq : kMaxPagesWideK;
  if (p->max_pages_per_req > page_cap)
    return fail(SPS_EUNSUPPORTED,
                "max_pages_per_req above %d (%dK tokens of context per request) is not supported "
                "with top_k %d",
                page_cap, page_cap * kPage / 1024, p->top_k);
  return SPS_OK;
}

// Indexer work list: tiles of <= 128 tokens x (1 or 2 heads of one KV group) against page
// chunks; the chunk starts at 128 pages and halves (down to 8) until there are enough items
// for a few waves.  Items are ordered by decreasing page count (largest first), then by
// their natural order, so a static round-robin over CTAs balances well.
void build_indexer_tasks(sps_plan* pl) {
  const sps_problem& p = pl->pb;
  const int Hg = p.num_q_heads / p.num_kv_heads;
  const int nh = (Hg % 2 == 0) ? 2 : 1;
  const int64_t target = 4LL * std::max(1, num_sms());
  int chunk = 128;
  for (;;) {
    std::vector<IdxTask> tasks;
    for (int b = 0; b < p.batch; ++b) {
      const ReqInfo& ri = pl->reqs[b];
      for (int i0 = 0; i0 < ri.q_len; i0 += kPage) {
        int ntok = std::min(kPage, ri.q_len - i0);
        int o_last = (ri.ctx + i0 + ntok - 1) / kPage;
        for (int g = 0; g < p.num_kv_heads; ++g)
          for (int hl = 0; hl < Hg; hl += nh)
            for (int pb = 0; pb <= o_last; pb += chunk) {
              IdxTask t;
              t.req = b;
              t.g = g;
              t.h0 = g * Hg + hl;
              t.nh = nh;
              t.tok0 = ri.tok0 + i0;
              t.ntok = ntok;
              t.page_begin = pb;
              t.page_end = std::min(o_last + 1, pb + chunk);
              tasks.push_back(t);
            }
      }
    }
    if ((int64_t)tasks.size() >= target || chunk <= 8) {
      std::stable_sort(tasks.begin(), tasks.end(), [](const IdxTask& a, const IdxTask& b) {
        return (a.page_end - a.page_begin) > (b.page_end - b.page_begin);
      });
      pl->idx_tasks.swap(tasks);
      return;
    }
    chunk /= 2;
  }
}

}  // namespace

extern "C" {

const char* sps_last_error(void) { return g_err.c_str(); }

sps_status sparse_prefill_plan(const sps_problem* problem, sps_plan** out,
                               size_t* workspace_bytes) {
  if (!out || !workspace_bytes) return fail(SPS_EINVAL, "plan/workspace_bytes out-pointers NULL");
  *out = nullptr;
  sps_status st = validate_problem(problem);
  if (st != SPS_OK) return st;
  sps_plan* pl = new (std::nothrow) sps_plan();
  if (!pl) return fail(SPS_EINVAL, "out of host memory");
  pl->pb = *problem;
  const sps_problem& p = pl->pb;
  pl->q_lens.assign(problem->q_lens, problem->q_lens + p.batch);
  pl->ctx_lens.assign(problem->ctx_lens, problem->ctx_lens + p.batch);
  pl->pb.q_lens = pl->q_lens.data();
  pl->pb.ctx_lens = pl->ctx_lens.data();
  const int Hg = p.num_q_heads / p.num_kv_heads;

  // per-request info, per-token metadata
  std::vector<int32_t> tok_pos, tok_req;
  int32_t tok = 0, page_base = 0;
  for (int b = 0; b < p.batch; ++b) {
    ReqInfo ri{};
    ri.tok0 = tok;
    ri.q_len = pl->q_lens[b];
    ri.ctx = pl->ctx_lens[b];
    ri.npages = ri.q_len > 0 ? (ri.ctx + ri.q_len - 1) / kPage + 1 : 0;
    ri.page_base = page_base;
    ri.words = (int32_t)((int64_t(ri.q_len) * Hg + 31) / 32);
    ri.ch_per_bucket = (ri.words + kChunkWords - 1) / kChunkWords;
    ri.blk_base = (int32_t)pl->inv_blocks;
    pl->inv_blocks += (int64_t)p.num_kv_heads * ri.ch_per_bucket;
    ri.ch_base = (int32_t)pl->num_chunks;
    pl->num_chunks += (int64_t)ri.npages * p.num_kv_heads * ri.ch_per_bucket;
    for (int i = 0; i < ri.q_len; ++i) {
      tok_pos.push_back(ri.ctx + i);
      tok_req.push_back(b);
    }
    for (int pg = 0; pg < ri.npages; ++pg) pl->page_req.push_back(b);
    page_base += ri.npages;
    tok += ri.q_len;
    pl->reqs.push_back(ri);
  }
  pl->T = tok;
  pl->R = (int64_t)tok * p.num_q_heads;
  pl->total_pages = page_base;
  pl->num_buckets = (int64_t)page_base * p.num_kv_heads;
  pl->max_entries = pl->R * p.top_k;
  const int64_t per_task = (int64_t)kFwdTaskGroups * 128;
  pl->max_fwd_tasks = pl->max_entries / per_task + pl->num_buckets + 1;
  build_indexer_tasks(pl);

  // workspace layout
  int64_t off = 0;
  auto take = [&](int64_t bytes) {
    int64_t o = off;
    off = align_up(off + std::max<int64_t>(bytes, 4), 256);
    return o;
  };
  pl->off_status = take(4);
  pl->off_counters = take(16 * 4);
  pl->off_tok_pos = take(4 * pl->T);
  pl->off_tok_req = take(4 * pl->T);
  pl->off_reqs = take(sizeof(ReqInfo) * p.batch);
  pl->off_page_req = take(4 * std::max<int64_t>(1, pl->total_pages));
  pl->off_idx_tasks = take(sizeof(IdxTask) * std::max<size_t>(1, pl->idx_tasks.size()));
  int64_t upload_end = off;
  pl->off_chunk_offsets = take(4 * (pl->num_chunks + 1));
  pl->off_bucket_totals = take(4 * pl->num_buckets);
  // per block of the single-launch inversion, or of the multi-kernel one's scan: its range's
  // entries and work items
  pl->off_range_sums = take(8 * std::max<int64_t>(
      {int64_t(1), pl->inv_blocks, (pl->num_buckets + kInvScanBuckets - 1) / kInvScanBuckets}));
  pl->off_bucket_offsets = take(4 * (pl->num_buckets + 1));
  pl->off_entries = take(8 * std::max<int64_t>(1, pl->max_entries));
  pl->off_fwd_tasks = take(sizeof(FwdTask) * pl->max_fwd_tasks);
  // FP16 staging of quantised inputs for the tensor-core paths: an exact FP16 copy of E4M3 Q;
  // an indexer over NVFP4 keys also takes FP16 copies of the key tiles of the pages the batch
  // sees (every one of them is read by the indexer), so the workspace grows with the batch,
  // not with the physical pool.  The forward dequantises NVFP4 K/V inside its loader, and
  // E4M3 x E4M3 indexing runs on the FP8 tensor core directly; neither needs a copy.
  const bool idx_fp16 = p.idx_k_dtype == SPS_NVFP4;
  if (p.q_dtype == SPS_E4M3 || (idx_fp16 && p.idx_q_dtype == SPS_E4M3))
    pl->off_qconv = take(2 * pl->R * p.head_dim);
  if (idx_fp16)
    pl->off_kconv = take(2 * std::max<int64_t>(1, pl->total_pages) * p.num_kv_heads * kPage *
                         p.head_dim);
  pl->fwd_ws_bytes = off;
  // at most 128 entries per bucket on average: most work items are a single group
  pl->fwd_prefetch = pl->max_entries <= 128 * std::max<int64_t>(1, pl->num_buckets) ? 1 : 0;
  // Top-k with top_k <= 16 runs a thread per row, so long rows of a small batch leave few
  // warps, each walking hundreds of 16-page groups one after another.  From 64 groups on, pass
  // 1 is split into segments of at least 32 groups, enough of them for ~24 warps per SM of a
  // 152-SM GPU; each segment's 16 largest scores go to this area and merge per row, and the
  // largest score of each 16-page group lets pass 2 read only the groups that can hold a
  // chosen page.
  const int64_t groups = (p.max_pages_per_req + 15) / 16;
  if (p.top_k > 1 && p.top_k <= 16 && groups >= 64) {
    const int64_t warps = (pl->R + 31) / 32, target = 24 * 152;
    const int64_t nseg = std::min<int64_t>(groups / 32, (target + warps - 1) / warps);
    if (nseg >= 2) {
      pl->topk_nseg = (int32_t)nseg;
      pl->topk_segg = (int32_t)((groups + nseg - 1) / nseg);
      pl->off_topk_lists = take(4 * 16 * pl->R * nseg);
      pl->off_topk_meta = take(4 * 3 * pl->R);
      pl->off_topk_gmax = take(4 * groups * pl->R);
    }
  }
  pl->ws_bytes = off;

  // the host image of [0, upload_end): the status word and counters (zero), then the metadata
  pl->upload_bytes = upload_end;
  pl->blob.assign(pl->upload_bytes, 0);
  auto put = [&](int64_t o, const void* src, size_t n) {
    if (n) memcpy(pl->blob.data() + o, src, n);
  };
  put(pl->off_tok_pos, tok_pos.data(), 4 * tok_pos.size());
  put(pl->off_tok_req, tok_req.data(), 4 * tok_req.size());
  put(pl->off_reqs, pl->reqs.data(), sizeof(ReqInfo) * pl->reqs.size());
  put(pl->off_page_req, pl->page_req.data(), 4 * pl->page_req.size());
  put(pl->off_idx_tasks, pl->idx_tasks.data(), sizeof(IdxTask) * pl->idx_tasks.size());

  *out = pl;
  *workspace_bytes = (size_t)pl->ws_bytes;
  return SPS_OK;
}

void sps_plan_destroy(sps_plan* plan) { delete plan; }

sps_status sps_plan_get_info(const sps_plan* pl, sps_plan_info* info) {
  if (!pl || !info) return fail(SPS_EINVAL, "plan/info NULL");
  info->num_tokens = pl->T;
  info->num_rows = pl->R;
  info->num_buckets = pl->num_buckets;
  info->max_entries = pl->max_entries;
  info->indexer_tasks = (int64_t)pl->idx_tasks.size();
  info->max_fwd_tasks = pl->max_fwd_tasks;
  info->workspace_bytes = pl->ws_bytes;
  info->off_status = pl->off_status;
  info->off_tok_pos = pl->off_tok_pos;
  info->off_tok_req = pl->off_tok_req;
  info->off_bucket_offsets = pl->off_bucket_offsets;
  info->off_entries = pl->off_entries;
  info->off_fwd_task_count = pl->off_counters + 2 * 4;
  return SPS_OK;
}

}  // extern "C"

namespace {

DevPlan make_dev_plan(const sps_plan* pl, void* ws) {
  uint8_t* base = static_cast<uint8_t*>(ws);
  const sps_problem& p = pl->pb;
  DevPlan d{};
  d.batch = p.batch;
  d.T = (int32_t)pl->T;
  d.H = p.num_q_heads;
  d.Hkv = p.num_kv_heads;
  d.Hg = p.num_q_heads / p.num_kv_heads;
  d.D = p.head_dim;
  d.K = p.top_k;
  d.max_pages = p.max_pages_per_req;
  d.num_phys = p.num_phys_pages;
  d.num_buckets = (int32_t)pl->num_buckets;
  d.max_entries = (int32_t)pl->max_entries;
  d.max_fwd_tasks = (int32_t)pl->max_fwd_tasks;
  d.n_idx_tasks = (int32_t)pl->idx_tasks.size();
  d.total_pages = (int32_t)pl->total_pages;
  d.inv_blocks = (int32_t)pl->inv_blocks;
  d.sm_scale = p.softmax_scale;
  d.status = reinterpret_cast<int32_t*>(base + pl->off_status);
  d.counters = reinterpret_cast<int32_t*>(base + pl->off_counters);
  d.tok_pos = reinterpret_cast<const int32_t*>(base + pl->off_tok_pos);
  d.tok_req = reinterpret_cast<const int32_t*>(base + pl->off_tok_req);
  d.reqs = reinterpret_cast<const ReqInfo*>(base + pl->off_reqs);
  d.page_req = reinterpret_cast<const int32_t*>(base + pl->off_page_req);
  d.idx_tasks = reinterpret_cast<const IdxTask*>(base + pl->off_idx_tasks);
  d.num_chunks = (int32_t)pl->num_chunks;
  d.chunk_offsets = reinterpret_cast<int32_t*>(base + pl->off_chunk_offsets);
  d.bucket_offsets = reinterpret_cast<int32_t*>(base + pl->off_bucket_offsets);
  d.bucket_totals = reinterpret_cast<int32_t*>(base + pl->off_bucket_totals);
  d.range_sums = reinterpret_cast<int32_t*>(base + pl->off_range_sums);
  d.entries = reinterpret_cast<int2*>(base + pl->off_entries);
  d.fwd_tasks = reinterpret_cast<FwdTask*>(base + pl->off_fwd_tasks);
  d.qconv = pl->off_qconv >= 0 ? base + pl->off_qconv : nullptr;
  d.kconv = pl->off_kconv >= 0 ? base + pl->off_kconv : nullptr;
  d.topk_lists = pl->off_topk_lists >= 0 ? reinterpret_cast<float*>(base + pl->off_topk_lists)
                                         : nullptr;
  d.topk_meta = pl->off_topk_meta >= 0 ? reinterpret_cast<int32_t*>(base + pl->off_topk_meta)
                                       : nullptr;
  d.topk_gmax = pl->off_topk_gmax >= 0 ? reinterpret_cast<float*>(base + pl->off_topk_gmax)
                                       : nullptr;
  d.topk_nseg = pl->topk_nseg;
  d.fwd_prefetch = pl->fwd_prefetch;
  d.topk_segg = pl->topk_segg;
  return d;
}

sps_status check_plan_ws(const sps_plan* pl, const void* ws) {
  if (!pl) return fail(SPS_EINVAL, "plan is NULL");
  if (!ws) return fail(SPS_EINVAL, "workspace is NULL");
  if (!aligned(ws, 256)) return fail(SPS_EINVAL, "workspace must be 256-byte aligned");
  return SPS_OK;
}

sps_status launched(cudaError_t e, const char* what) {
  if (e == cudaErrorNotSupported)
    return fail(SPS_EUNSUPPORTED, "%s: not implemented for this dtype combination / head_dim",
                what);
  if (e != cudaSuccess) return cuda_fail(e, what);
  return SPS_OK;
}

}  // namespace

extern "C" {

sps_status sps_plan_upload(const sps_plan* pl, void* ws, size_t ws_bytes, sps_stream_t stream) {
  sps_status st = check_plan_ws(pl, ws);
  if (st != SPS_OK) return st;
  if ((int64_t)ws_bytes < pl->ws_bytes)
    return fail(SPS_ENOSPACE, "workspace of %zu bytes < %lld required", ws_bytes,
                (long long)pl->ws_bytes);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* base = static_cast<uint8_t*>(ws);
  // one copy: zeroed status word and counters, then the plan metadata
  cudaError_t e = g_staging.upload(base, pl->blob.data(), pl->upload_bytes, s, true);
  if (e != cudaSuccess) return cuda_fail(e, "plan upload");
  return SPS_OK;
}

sps_status indexer_scores(const sps_plan* pl, const void* q_idx, float q_scale,
                          const void* k_idx_cache, const void* k_idx_scales, float k_scale,
                          const int32_t* page_table, float* scores, int64_t score_pitch,
                          void* ws, sps_stream_t stream) {
  sps_status st = check_plan_ws(pl, ws);
  if (st != SPS_OK) return st;
  const sps_problem& p = pl->pb;
  if (!q_idx || !k_idx_cache || !page_table || !scores)
    return fail(SPS_EINVAL, "indexer_scores: NULL input/output pointer");
  if (p.idx_k_dtype == SPS_NVFP4 && !k_idx_scales)
    return fail(SPS_EINVAL, "indexer_scores: NVFP4 keys need k_idx_scales");
  if (score_pitch < p.max_pages_per_req)
    return fail(SPS_EINVAL, "score_pitch %lld < max_pages_per_req %d", (long long)score_pitch,
                p.max_pages_per_req);
  if (!aligned(q_idx, 16) || !aligned(k_idx_cache, 16) || (k_idx_scales && !aligned(k_idx_scales, 16)))
    return fail(SPS_EINVAL, "indexer_scores: q/k buffers must be 16-byte aligned");
  if (!aligned(scores, 4)) return fail(SPS_EINVAL, "scores must be 4-byte aligned");
  if (!std::isfinite(q_scale) || !std::isfinite(k_scale))
    return fail(SPS_EINVAL, "indexer_scores: scales must be finite");
  DevPlan d = make_dev_plan(pl, ws);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  return launched(launch_indexer(d, p.idx_q_dtype, p.idx_k_dtype, q_idx, q_scale, k_idx_cache,
                                 k_idx_scales, k_scale, page_table, scores, score_pitch, s),
                  "indexer launch");
}

sps_status topk_select(const sps_plan* pl, const float* scores, int64_t score_pitch,
                       int32_t* idx, void* ws, sps_stream_t stream) {
  sps_status st = check_plan_ws(pl, ws);
  if (st != SPS_OK) return st;
  if (!scores || !idx) return fail(SPS_EINVAL, "topk_select: NULL scores/idx");
  if (score_pitch < pl->pb.max_pages_per_req)
    return fail(SPS_EINVAL, "score_pitch %lld < max_pages_per_req %d", (long long)score_pitch,
                pl->pb.max_pages_per_req);
  if (!aligned(scores, 4) || !aligned(idx, 4)) return fail(SPS_EINVAL, "misaligned scores/idx");
  DevPlan d = make_dev_plan(pl, ws);
  return launched(launch_topk(d, scores, score_pitch, idx, reinterpret_cast<cudaStream_t>(stream)),
                  "top-k launch");
}

namespace {

// The forward with FP32, BF16 or FP16 partials, or the FP8-QK route: the same checks and
// launches.
enum class FwdKind { kFP32, kBF16Partials, kF16Partials, kFP8QK };
sps_status fwd_common(const sps_plan* pl, const void* q, float q_scale, const void* k_cache,
                      const void* v_cache, const void* k_scales, const void* v_scales,
                      const int32_t* page_table, const int32_t* idx, void* partial,
                      int64_t split_stride, float* lse, int64_t lse_split_stride, void* ws,
                      sps_stream_t stream, FwdKind kind) {
  const bool p16 = kind == FwdKind::kBF16Partials || kind == FwdKind::kF16Partials;
  sps_status st = check_plan_ws(pl, ws);
  if (st != SPS_OK) return st;
  const sps_problem& p = pl->pb;
  if (!q || !k_cache || !v_cache || !page_table || !idx || !partial || !lse)
    return fail(SPS_EINVAL, "sparse_prefill_fwd: NULL input/output pointer");
  if (p.kv_dtype == SPS_NVFP4 && (!k_scales || !v_scales))
    return fail(SPS_EINVAL, "sparse_prefill_fwd: NVFP4 K/V need k_scales and v_scales");
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      (k_scales && !aligned(k_scales, 16)) || (v_scales && !aligned(v_scales, 16)))
    return fail(SPS_EINVAL, "sparse_prefill_fwd: q/k/v buffers must be 16-byte aligned");
  if (!aligned(partial, 16)) return fail(SPS_EINVAL, "partial must be 16-byte aligned");
  const int64_t qa = p16 ? 8 : 4;  // elements per 16 bytes
  if (split_stride < pl->R * p.head_dim || split_stride % qa)
    return fail(SPS_EINVAL, "split_stride must be >= rows*head_dim and a multiple of %lld",
                (long long)qa);
  if (lse_split_stride < pl->R) return fail(SPS_EINVAL, "lse_split_stride must be >= rows");
  if (!std::isfinite(q_scale)) return fail(SPS_EINVAL, "q_scale must be finite");
  if (kind == FwdKind::kFP8QK &&
      (p.q_dtype != SPS_E4M3 || p.kv_dtype != SPS_NVFP4 || p.head_dim != 128))
    return fail(SPS_EUNSUPPORTED, "sparse_prefill_fwd_fp8qk: needs E4M3 Q, NVFP4 K/V, D = 128");
  DevPlan d = make_dev_plan(pl, ws);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // no counter needs clearing here: the inversion writes the task count, and its grid barrier
  // returns to zero when it completes (the plan upload clears it first)
  cudaError_t e = launch_inversion(d, idx, lse, lse_split_stride, s);
  if (e != cudaSuccess) return cuda_fail(e, "inversion launch");
  if (kind == FwdKind::kFP8QK)
    return launched(launch_forward_fp8qk(d, p.q_dtype, p.kv_dtype, q, q_scale, k_cache, v_cache,
                                         k_scales, v_scales, page_table,
                                         static_cast<float*>(partial), split_stride, lse,
                                         lse_split_stride, s),
                    "forward launch");
  if (kind == FwdKind::kBF16Partials)
    return launched(launch_forward_bf16p(d, p.q_dtype, p.kv_dtype, q, q_scale, k_cache, v_cache,
                                         k_scales, v_scales, page_table, partial, split_stride,
                                         lse, lse_split_stride, s),
                    "forward launch");
  if (kind == FwdKind::kF16Partials)
    return launched(launch_forward_f16p(d, p.q_dtype, p.kv_dtype, q, q_scale, k_cache, v_cache,
                                        k_scales, v_scales, page_table, partial, split_stride,
                                        lse, lse_split_stride, s),
                    "forward launch");
  return launched(launch_forward(d, p.q_dtype, p.kv_dtype, q, q_scale, k_cache, v_cache, k_scales,
                                 v_scales, page_table, static_cast<float*>(partial),
                                 split_stride, lse, lse_split_stride, s),
                  "forward launch");
}

sps_status combine_common(int64_t rows, int32_t splits, int32_t head_dim, const void* partial,
                          int64_t split_stride, const float* lse, int64_t lse_split_stride,
                          void* out_bf16, int64_t out_row_stride, float* out_lse,
                          int32_t* dev_status, sps_stream_t stream, int ptype) {
  const bool p16 = ptype != 0;  // 0: FP32, 1: BF16, 2: FP16 partials
  if (rows < 0) return fail(SPS_EINVAL, "rows must be >= 0");
  if (splits < 1 || splits > kMaxTopK) return fail(SPS_EINVAL, "splits must be in [1, 64]");
  if (head_dim != 64 && head_dim != 128) return fail(SPS_EUNSUPPORTED, "head_dim must be 64 or 128");
  if (rows == 0) return SPS_OK;
  if (!partial || !lse || !out_bf16) return fail(SPS_EINVAL, "partial_combine: NULL pointer");
  if (!aligned(partial, 16) || !aligned(out_bf16, 16) || !aligned(lse, 4))
    return fail(SPS_EINVAL, "partial/out must be 16-byte aligned, lse 4-byte aligned");
  const int64_t qa = p16 ? 8 : 4;  // elements per 16 bytes
  if (split_stride % qa || split_stride < rows * head_dim)
    return fail(SPS_EINVAL, "split_stride must be a multiple of %lld and >= rows*head_dim",
                (long long)qa);
  if (lse_split_stride < rows) return fail(SPS_EINVAL, "lse_split_stride must be >= rows");
  if (out_row_stride < head_dim || out_row_stride % 8)
    return fail(SPS_EINVAL, "out_row_stride must be >= head_dim and a multiple of 8");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (ptype == 1)
    return launched(launch_combine_bf16p(rows, splits, head_dim, partial, split_stride, lse,
                                         lse_split_stride, out_bf16, out_row_stride, out_lse,
                                         dev_status, s),
                    "combine launch");
  if (ptype == 2)
    return launched(launch_combine_f16p(rows, splits, head_dim, partial, split_stride, lse,
                                        lse_split_stride, out_bf16, out_row_stride, out_lse,
                                        dev_status, s),
                    "combine launch");
  return launched(launch_combine(rows, splits, head_dim, static_cast<const float*>(partial),
                                 split_stride, lse, lse_split_stride, out_bf16, out_row_stride,
                                 out_lse, dev_status, s),
                  "combine launch");
}

}  // namespace

sps_status sparse_prefill_fwd(const sps_plan* pl, const void* q, float q_scale,
                              const void* k_cache, const void* v_cache, const void* k_scales,
                              const void* v_scales, const int32_t* page_table,
                              const int32_t* idx, float* partial, int64_t split_stride,
                              float* lse, int64_t lse_split_stride, void* ws,
                              sps_stream_t stream) {
  return fwd_common(pl, q, q_scale, k_cache, v_cache, k_scales, v_scales, page_table, idx,
                    partial, split_stride, lse, lse_split_stride, ws, stream, FwdKind::kFP32);
}

sps_status sparse_prefill_fwd_fp8qk(const sps_plan* pl, const void* q, float q_scale,
                                    const void* k_cache, const void* v_cache,
                                    const void* k_scales, const void* v_scales,
                                    const int32_t* page_table, const int32_t* idx, float* partial,
                                    int64_t split_stride, float* lse, int64_t lse_split_stride,
                                    void* ws, sps_stream_t stream) {
  return fwd_common(pl, q, q_scale, k_cache, v_cache, k_scales, v_scales, page_table, idx,
                    partial, split_stride, lse, lse_split_stride, ws, stream, FwdKind::kFP8QK);
}

sps_status sparse_prefill_fwd_bf16(const sps_plan* pl, const void* q, float q_scale,
                                   const void* k_cache, const void* v_cache,
                                   const void* k_scales, const void* v_scales,
                                   const int32_t* page_table, const int32_t* idx,
                                   void* partial_bf16, int64_t split_stride, float* lse,
                                   int64_t lse_split_stride, void* ws, sps_stream_t stream) {
  return fwd_common(pl, q, q_scale, k_cache, v_cache, k_scales, v_scales, page_table, idx,
                    partial_bf16, split_stride, lse, lse_split_stride, ws, stream,
                    FwdKind::kBF16Partials);
}

sps_status partial_combine(int64_t rows, int32_t splits, int32_t head_dim, const float* partial,
                           int64_t split_stride, const float* lse, int64_t lse_split_stride,
                           void* out_bf16, int64_t out_row_stride, float* out_lse,
                           int32_t* dev_status, sps_stream_t stream) {
  return combine_common(rows, splits, head_dim, partial, split_stride, lse, lse_split_stride,
                        out_bf16, out_row_stride, out_lse, dev_status, stream, 0);
}

sps_status partial_combine_bf16(int64_t rows, int32_t splits, int32_t head_dim,
                                const void* partial_bf16, int64_t split_stride, const float* lse,
                                int64_t lse_split_stride, void* out_bf16, int64_t out_row_stride,
                                float* out_lse, int32_t* dev_status, sps_stream_t stream) {
  return combine_common(rows, splits, head_dim, partial_bf16, split_stride, lse,
                        lse_split_stride, out_bf16, out_row_stride, out_lse, dev_status, stream,
                        1);
}

sps_status sparse_prefill_fwd_f16(const sps_plan* pl, const void* q, float q_scale,
                                  const void* k_cache, const void* v_cache, const void* k_scales,
                                  const void* v_scales, const int32_t* page_table,
                                  const int32_t* idx, void* partial_f16, int64_t split_stride,
                                  float* lse, int64_t lse_split_stride, void* ws,
                                  sps_stream_t stream) {
  return fwd_common(pl, q, q_scale, k_cache, v_cache, k_scales, v_scales, page_table, idx,
                    partial_f16, split_stride, lse, lse_split_stride, ws, stream,
                    FwdKind::kF16Partials);
}

sps_status partial_combine_f16(int64_t rows, int32_t splits, int32_t head_dim,
                               const void* partial_f16, int64_t split_stride, const float* lse,
                               int64_t lse_split_stride, void* out_bf16, int64_t out_row_stride,
                               float* out_lse, int32_t* dev_status, sps_stream_t stream) {
  return combine_common(rows, splits, head_dim, partial_f16, split_stride, lse, lse_split_stride,
                        out_bf16, out_row_stride, out_lse, dev_status, stream, 2);
}

sps_status sps_kv_append(const sps_plan* pl, const void* k_new, const void* v_new,
                         const int32_t* page_table, void* k_cache, void* v_cache, void* k_scales,
                         void* v_scales, void* ws, sps_stream_t stream) {
  sps_status st = check_plan_ws(pl, ws);
  if (st != SPS_OK) return st;
  const sps_problem& p = pl->pb;
  const bool nvfp4 = p.kv_dtype == SPS_NVFP4;
  if (p.kv_dtype != SPS_BF16 && !nvfp4)
    return fail(SPS_EUNSUPPORTED, "sps_kv_append: the cache must be BF16 or NVFP4");
  if (!k_new || !v_new || !page_table || !k_cache || !v_cache)
    return fail(SPS_EINVAL, "sps_kv_append: NULL pointer");
  if (nvfp4 && (!k_scales || !v_scales))
    return fail(SPS_EINVAL, "sps_kv_append: an NVFP4 cache needs k_scales and v_scales");
  if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_cache, 16) ||
      !aligned(v_cache, 16) || !aligned(page_table, 4))
    return fail(SPS_EINVAL, "sps_kv_append: buffers must be 16-byte aligned");
  DevPlan d = make_dev_plan(pl, ws);
  return launched(launch_kv_append(d, nvfp4, k_new, v_new, page_table, k_cache, v_cache, k_scales,
                                   v_scales, reinterpret_cast<cudaStream_t>(stream)),
                  "kv append launch");
}

sps_status sps_quantize_e4m3(const void* x_bf16, int64_t n, float scale, void* codes,
                             sps_stream_t stream) {
  if (n < 0 || n % 16) return fail(SPS_EINVAL, "sps_quantize_e4m3: n must be a multiple of 16");
  if (!(scale > 0.f) || !std::isfinite(scale))
    return fail(SPS_EINVAL, "sps_quantize_e4m3: scale must be finite and > 0");
  if (n == 0) return SPS_OK;
  if (!x_bf16 || !codes || !aligned(x_bf16, 16) || !aligned(codes, 16))
    return fail(SPS_EINVAL, "sps_quantize_e4m3: buffers must be non-NULL and 16-byte aligned");
  return launched(launch_quantize_e4m3(x_bf16, n, scale, codes,
                                       reinterpret_cast<cudaStream_t>(stream)),
                  "quantize launch");
}

sps_status sps_absmax_bf16(const void* x_bf16, int64_t n, float* absmax, sps_stream_t stream) {
  if (n < 0 || n % 16) return fail(SPS_EINVAL, "sps_absmax_bf16: n must be a multiple of 16");
  if (!absmax || !aligned(absmax, 4)) return fail(SPS_EINVAL, "sps_absmax_bf16: bad output");
  if (n > 0 && (!x_bf16 || !aligned(x_bf16, 16)))
    return fail(SPS_EINVAL, "sps_absmax_bf16: input must be non-NULL and 16-byte aligned");
  return launched(launch_absmax_bf16(x_bf16, n, absmax, reinterpret_cast<cudaStream_t>(stream)),
                  "absmax launch");
}

sps_status sps_dequantize(sps_dtype in_dtype, const void* in, const void* scales, int64_t n,
                          void* out_f16, sps_stream_t stream) {
  if (in_dtype != SPS_E4M3 && in_dtype != SPS_NVFP4)
    return fail(SPS_EUNSUPPORTED, "sps_dequantize: input must be E4M3 or NVFP4");
  if (n < 0 || n % 16) return fail(SPS_EINVAL, "sps_dequantize: n must be a multiple of 16");
  if (n == 0) return SPS_OK;
  if (!in || !out_f16 || (in_dtype == SPS_NVFP4 && !scales))
    return fail(SPS_EINVAL, "sps_dequantize: NULL pointer");
  if (!aligned(in, in_dtype == SPS_E4M3 ? 16 : 8) || !aligned(out_f16, 16))
    return fail(SPS_EINVAL, "sps_dequantize: input must be %d-byte and output 16-byte aligned",
                in_dtype == SPS_E4M3 ? 16 : 8);
  return launched(launch_dequant(in_dtype, in, scales, n, out_f16,
                                 reinterpret_cast<cudaStream_t>(stream)),
                  "dequant launch");
}

sps_status sps_check_wait_timeout(int64_t limit_ns, int32_t* dev_status, sps_stream_t stream) {
  if (!dev_status || !aligned(dev_status, 4))
    return fail(SPS_EINVAL, "sps_check_wait_timeout: dev_status must be a device int32");
  if (limit_ns < 1000000 || limit_ns > 10000000000LL)
    return fail(SPS_EINVAL, "sps_check_wait_timeout: limit_ns must be in [1e6, 1e10]");
  return launched(launch_wait_timeout(dev_status, limit_ns, reinterpret_cast<cudaStream_t>(stream)),
                  "wait-timeout check launch");
}

sps_status sps_check_barrier_timeout(int64_t limit_ns, uint32_t* dev_barrier,
                                     int32_t* dev_status, sps_stream_t stream) {
  if (!dev_status || !aligned(dev_status, 4) || !dev_barrier || !aligned(dev_barrier, 4))
    return fail(SPS_EINVAL, "sps_check_barrier_timeout: dev_barrier/dev_status must be device words");
  if (limit_ns < 1000000 || limit_ns > 10000000000LL)
    return fail(SPS_EINVAL, "sps_check_barrier_timeout: limit_ns must be in [1e6, 1e10]");
  return launched(launch_barrier_timeout(dev_barrier, dev_status, limit_ns,
                                         reinterpret_cast<cudaStream_t>(stream)),
                  "barrier timeout check launch");
}

sps_status sps_read_device_status(const sps_plan* pl, const void* ws, int32_t* code) {
  if (!code) return fail(SPS_EINVAL, "code is NULL");
  sps_status st = check_plan_ws(pl, ws);
  if (st != SPS_OK) return st;
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
  e = cudaMemcpy(code, static_cast<const uint8_t*>(ws) + pl->off_status, 4,
                 cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy(status)");
  if (*code != 0) return fail(SPS_EDEVICE, "device status %d", *code);
  return SPS_OK;
}

}  // extern "C"

// ------------------------------------------------------------------ driver helpers
namespace sps {

namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
void load_encode() {
  cudaDriverEntryPointQueryResult q;
  void* fn = nullptr;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
}
CUtensorMapDataType tm_type(int code) {
  switch (code) {
    case 0: return CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    case 1: return CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    default: return CU_TENSOR_MAP_DATA_TYPE_UINT8;
  }
}
int tm_size(int code) { return code <= 1 ? 2 : 1; }
}  // namespace

bool encode_tmap_2d(void* map, int dtype_code, void* base, uint64_t inner, uint64_t outer,
                    uint64_t outer_stride_bytes, uint32_t box_inner, uint32_t box_outer,
                    bool swizzle128) {
  std::call_once(g_encode_once, load_encode);
  if (!g_encode) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {outer_stride_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  (void)tm_size;
  return g_encode(reinterpret_cast<CUtensorMap*>(map), tm_type(dtype_code), 2, base, dims,
                  strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_tmap_3d(void* map, int dtype_code, void* base, uint64_t d0, uint64_t d1,
                    uint64_t d2, uint64_t s1_bytes, uint64_t s2_bytes, uint32_t b0, uint32_t b1,
                    uint32_t b2, bool swizzle128) {
  std::call_once(g_encode_once, load_encode);
  if (!g_encode) return false;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {s1_bytes, s2_bytes};
  cuuint32_t box[3] = {b0, b1, b2};
  cuuint32_t es[3] = {1, 1, 1};
  return g_encode(reinterpret_cast<CUtensorMap*>(map), tm_type(dtype_code), 3, base, dims,
                  strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_tmap_2d_f32_sw64(void* map, const void* base, uint64_t inner, uint64_t outer,
                             uint64_t outer_stride_bytes, uint32_t box_inner,
                             uint32_t box_outer) {
  std::call_once(g_encode_once, load_encode);
  if (!g_encode) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {outer_stride_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  return g_encode(reinterpret_cast<CUtensorMap*>(map), CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
                  const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int num_sms() {
  static int n = -1;
  if (n < 0) {
    int dev = 0, v = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0)
      n = v;
    else
      n = 152;  // planning without a device: the GB300 SM count
  }
  return n;
}

}  // namespace sps

// ------------------------------------------------------------------ scratch-array forward
// Used by sparse_prefill_fwd_noalloc (noalloc.cu), which owns the scratch array: the same
// checks and launches as sparse_prefill_fwd, with the plan's metadata copied into the given
// scratch area first (the caller has no workspace to upload into).
sps_status sps_internal_cuda_fail(cudaError_t e, const char* what) { return cuda_fail(e, what); }

sps_status sps_internal_fwd_noalloc(const sps_plan* pl, const void* q, float q_scale,
                                    const void* k_cache, const void* v_cache, const void* k_scales,
                                    const void* v_scales, const int32_t* page_table,
                                    const int32_t* idx, float* partial, int64_t split_stride,
                                    float* lse, int64_t lse_split_stride, void* scratch,
                                    size_t scratch_bytes, int32_t* dev_status,
                                    sps_stream_t stream) {
  if (!pl) return fail(SPS_EINVAL, "plan is NULL");
  const sps_problem& p = pl->pb;
  if (!q || !k_cache || !v_cache || !page_table || !idx || !partial || !lse)
    return fail(SPS_EINVAL, "sparse_prefill_fwd_noalloc: NULL input/output pointer");
  if (p.kv_dtype == SPS_NVFP4 && (!k_scales || !v_scales))
    return fail(SPS_EINVAL, "sparse_prefill_fwd_noalloc: NVFP4 K/V need k_scales and v_scales");
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      (k_scales && !aligned(k_scales, 16)) || (v_scales && !aligned(v_scales, 16)))
    return fail(SPS_EINVAL, "sparse_prefill_fwd_noalloc: q/k/v buffers must be 16-byte aligned");
  if (!aligned(partial, 16)) return fail(SPS_EINVAL, "partial must be 16-byte aligned");
  if (split_stride < pl->R * p.head_dim || split_stride % 4)
    return fail(SPS_EINVAL, "split_stride must be >= rows*head_dim and a multiple of 4");
  if (lse_split_stride < pl->R) return fail(SPS_EINVAL, "lse_split_stride must be >= rows");
  if (!std::isfinite(q_scale)) return fail(SPS_EINVAL, "q_scale must be finite");
  if (dev_status && !aligned(dev_status, 4)) return fail(SPS_EINVAL, "dev_status misaligned");
  if ((int64_t)scratch_bytes < pl->fwd_ws_bytes)
    return fail(SPS_ENOSPACE,
                "sparse_prefill_fwd_noalloc: this batch needs %lld bytes of scratch, the built-in "
                "array holds %zu; split the batch or use sparse_prefill_fwd with a workspace",
                (long long)pl->fwd_ws_bytes, scratch_bytes);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* base = static_cast<uint8_t*>(scratch);
  // the array keeps the previous call's contents: one copy zeroes the status word and
  // counters and writes this plan's metadata over the old one
  cudaError_t e = g_staging.upload(base, pl->blob.data(), pl->upload_bytes, s, false);
  if (e != cudaSuccess) return cuda_fail(e, "plan metadata -> scratch");
  DevPlan d = make_dev_plan(pl, scratch);
  if (dev_status) d.status = dev_status;
  e = launch_inversion(d, idx, lse, lse_split_stride, s);
  if (e != cudaSuccess) return cuda_fail(e, "inversion launch");
  return launched(launch_forward(d, p.q_dtype, p.kv_dtype, q, q_scale, k_cache, v_cache,
                                 k_scales, v_scales, page_table, partial, split_stride, lse,
                                 lse_split_stride, s),
                  "forward launch");
}
