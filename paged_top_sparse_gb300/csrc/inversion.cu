// inversion.cu -- page -> (row, slot) inversion of the top-k selection, deterministic.
//
// The forward runs one work item per (page, KV head, query split) ("MSA PR 21: Q8KV4 paged
// sparse prefill", K1), so the row-major selection idx[row][slot] is turned around: for every
// bucket (request, logical page, KV head) the (row, slot) pairs that chose it, in ascending row
// order.  Nothing depends on the timing of atomics:
//
//   1. mark     a warp per 32 consecutive rows of one (request, KV head) sets one bit per
//               (bucket, row) in a selection bitmap (each bucket owns a run of words, bit b
//               of word w = row 32 w + b); warp-aggregated atomicOr; empty slots get
//               lse = -inf here.
//   2. count    a block per 2048-word chunk of a bucket: popcount of the chunk.
//   3. scan     one block: exclusive scan over chunks (buckets are runs of chunks) gives each
//               chunk's first entry and each bucket's CSR offset; then the forward's work
//               list (chunks of up to kFwdTaskGroups x 128 entries per bucket).
//   4. prefix   a block per chunk: exclusive popcount scan -> first entry of every word.
//   5. emit     a warp per 32 rows again: for every (row, slot) the entry position is the
//               word's first entry plus the set bits below the row's bit.  An entry is
//               (row, t * 64 + slot), t the row's absolute position, so the forward needs no
//               further lookup to find the row's own page and visible key count.
#include "ptx.cuh"
#include "sps_internal.h"

namespace sps {
namespace {

// Warp wid of the mark/emit grids -> request, KV head and bitmap word index.
__device__ __forceinline__ int find_word(const DevPlan& p, int64_t wid, int* w_in_req, int* g) {
  int64_t acc = 0;
  for (int b = 0; b < p.batch; ++b) {
    const int nw = p.reqs[b].bm_words;
    const int64_t n = (int64_t)p.Hkv * nw;
    if (wid < acc + n) {
      const int64_t local = wid - acc;
      *g = (int)(local / nw);
      *w_in_req = (int)(local % nw);
      return b;
    }
    acc += n;
  }
  return -1;
}

// Chunk id -> request, bucket, bucket-local (page, kv head) and chunk-within-bucket.
__device__ __forceinline__ int find_chunk(const DevPlan& p, int chunk, int* bucket, int* pg,
                                          int* g, int* c) {
  for (int b = p.batch - 1; b >= 0; --b) {
    const ReqInfo& ri = p.reqs[b];
    if (ri.npages > 0 && chunk >= ri.ch_base) {
      const int lc = chunk - ri.ch_base;
      const int bl = lc / ri.ch_per_bucket;
      *c = lc % ri.ch_per_bucket;
      *pg = bl / p.Hkv;
      *g = bl % p.Hkv;
      *bucket = (ri.page_base + *pg) * p.Hkv + *g;
      return b;
    }
  }
  return -1;
}

struct RowCtx {
  bool valid;
  int64_t r;
  int t;  // absolute position of the row's token
  int o;  // its own page
};

__device__ __forceinline__ RowCtx row_of(const DevPlan& p, const ReqInfo& ri, int g, int w,
                                         int lane) {
  RowCtx rc;
  const int row_local = w * 32 + lane;
  rc.valid = row_local < ri.q_len * p.Hg;
  rc.r = 0;
  rc.t = 0;
  rc.o = -1;
  if (rc.valid) {
    const int i = row_local / p.Hg, hl = row_local % p.Hg;
    rc.r = (int64_t)(ri.tok0 + i) * p.H + g * p.Hg + hl;
    rc.t = ri.ctx + i;
    rc.o = rc.t >> 7;
  }
  return rc;
}

__global__ void __launch_bounds__(256)
mark_kernel(DevPlan p, const int32_t* __restrict__ idx, float* __restrict__ lse,
            int64_t lse_split_stride) {
  const int64_t wid = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (wid >= p.mark_warps) return;
  int w, g;
  const int b = find_word(p, wid, &w, &g);
  if (b < 0) return;
  const ReqInfo ri = p.reqs[b];
  const RowCtx rc = row_of(p, ri, g, w, lane);
  for (int s = 0; s < p.K; ++s) {
    int pg = rc.valid ? __ldg(idx + rc.r * p.K + s) : -1;
    if (rc.valid && pg < 0) lse[s * lse_split_stride + rc.r] = -INFINITY;
    if (rc.valid && pg > rc.o) {
      set_status(p.status, DEV_BAD_INDEX);
      pg = -1;
    }
    // unique negative keys for inactive lanes so they only match themselves
    const int key = pg >= 0 ? pg : -1 - lane;
    const uint32_t mask = __match_any_sync(0xffffffffu, key);
    if (pg >= 0 && lane == __ffs(mask) - 1)
      atomicOr(p.bitmap + ri.bm_base + (int64_t)(pg * p.Hkv + g) * ri.bm_words + w, mask);
  }
}

__global__ void __launch_bounds__(256) count_kernel(DevPlan p) {
  __shared__ int sh[8];
  int bucket, pg, g, c;
  const int b = find_chunk(p, blockIdx.x, &bucket, &pg, &g, &c);
  if (b < 0) return;
  const ReqInfo ri = p.reqs[b];
  const uint32_t* words = p.bitmap + ri.bm_base + (int64_t)(pg * p.Hkv + g) * ri.bm_words;
  const int w0 = c * kChunkWords, w1 = min(ri.bm_words, w0 + kChunkWords);
  int n = 0;
  for (int w = w0 + threadIdx.x; w < w1; w += blockDim.x) n += __popc(words[w]);
  n = __reduce_add_sync(0xffffffffu, n);
  if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = n;
  __syncthreads();
  if (threadIdx.x == 0) {
    int t = 0;
    for (int i = 0; i < 8; ++i) t += sh[i];
    p.chunk_offsets[blockIdx.x] = t;  // a count here; the scan turns it into an offset
  }
}

// Block-wide exclusive scan of one int per thread; returns the block total.
__device__ __forceinline__ int block_exclusive_scan(int v, int* out, int* sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  int x = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, d);
    if (lane >= d) x += y;
  }
  if (lane == 31) sh[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int s = lane < nwarps ? sh[lane] : 0;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, s, d);
      if (lane >= d) s += y;
    }
    sh[lane] = s;
  }
  __syncthreads();
  const int total = sh[nwarps - 1];
  *out = (warp ? sh[warp - 1] : 0) + x - v;
  __syncthreads();
  return total;
}

// First chunk of bucket `bucket` (buckets are laid out request by request, page-major).
__device__ __forceinline__ int first_chunk(const DevPlan& p, int bucket) {
  const int gp = bucket / p.Hkv, g = bucket % p.Hkv;
  const ReqInfo& ri = p.reqs[p.page_req[gp]];
  return ri.ch_base + ((gp - ri.page_base) * p.Hkv + g) * ri.ch_per_bucket;
}

__global__ void __launch_bounds__(1024) scan_kernel(DevPlan p) {
  __shared__ int sh[32];
  const int nc = p.num_chunks;
  {  // chunk counts -> exclusive offsets (in place)
    const int per = (nc + 1023) / 1024;
    const int c0 = threadIdx.x * per;
    int cnt = 0;
    for (int c = c0; c < c0 + per && c < nc; ++c) cnt += p.chunk_offsets[c];
    int off;
    const int total = block_exclusive_scan(cnt, &off, sh);
    for (int c = c0; c < c0 + per && c < nc; ++c) {
      const int x = p.chunk_offsets[c];
      p.chunk_offsets[c] = off;
      off += x;
    }
    if (threadIdx.x == 0) {
      p.chunk_offsets[nc] = total;
      if (total > p.max_entries) set_status(p.status, DEV_OVERFLOW);
    }
  }
  __syncthreads();
  // bucket offsets and the forward work list
  const int nb = p.num_buckets;
  const int per = (nb + 1023) / 1024;
  const int b0 = threadIdx.x * per;
  const int per_task = kFwdTaskGroups * 128;
  int ntask = 0;
  for (int b = b0; b < b0 + per && b < nb; ++b) {
    const int beg = p.chunk_offsets[first_chunk(p, b)];
    const int end = b + 1 < nb ? p.chunk_offsets[first_chunk(p, b + 1)] : p.chunk_offsets[nc];
    ntask += (end - beg + per_task - 1) / per_task;
  }
  int toff;
  const int ttotal = block_exclusive_scan(ntask, &toff, sh);
  for (int b = b0; b < b0 + per && b < nb; ++b) {
    const int beg = p.chunk_offsets[first_chunk(p, b)];
    const int end = b + 1 < nb ? p.chunk_offsets[first_chunk(p, b + 1)] : p.chunk_offsets[nc];
    p.bucket_offsets[b] = beg;
    for (int e = beg; e < end; e += per_task) {
      if (toff < p.max_fwd_tasks) {
        FwdTask t;
        t.bucket = b;
        t.entry_begin = e;
        t.count = min(per_task, end - e);
        t.pad = 0;
        p.fwd_tasks[toff] = t;
      }
      ++toff;
    }
  }
  if (threadIdx.x == 0) {
    p.bucket_offsets[nb] = p.chunk_offsets[nc];
    p.counters[2] = min(ttotal, p.max_fwd_tasks);
    if (ttotal > p.max_fwd_tasks) set_status(p.status, DEV_OVERFLOW);
  }
}

__global__ void __launch_bounds__(256) prefix_kernel(DevPlan p) {
  __shared__ int sh[32];
  constexpr int WPT = kChunkWords / 256;  // words per thread
  int bucket, pg, g, c;
  const int b = find_chunk(p, blockIdx.x, &bucket, &pg, &g, &c);
  if (b < 0) return;
  const ReqInfo ri = p.reqs[b];
  const int64_t wbase = ri.bm_base + (int64_t)(pg * p.Hkv + g) * ri.bm_words;
  const int w0 = c * kChunkWords + threadIdx.x * WPT;
  int n = 0;
  uint32_t bits[WPT];
#pragma unroll
  for (int i = 0; i < WPT; ++i) {
    const int w = w0 + i;
    bits[i] = w < ri.bm_words ? p.bitmap[wbase + w] : 0u;
    n += __popc(bits[i]);
  }
  int off;
  block_exclusive_scan(n, &off, sh);
  off += p.chunk_offsets[blockIdx.x];
#pragma unroll
  for (int i = 0; i < WPT; ++i) {
    const int w = w0 + i;
    if (w < ri.bm_words) p.word_pos[wbase + w] = off;
    off += __popc(bits[i]);
  }
}

__global__ void __launch_bounds__(256)
emit_kernel(DevPlan p, const int32_t* __restrict__ idx) {
  const int64_t wid = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (wid >= p.mark_warps) return;
  int w, g;
  const int b = find_word(p, wid, &w, &g);
  if (b < 0) return;
  const ReqInfo ri = p.reqs[b];
  const RowCtx rc = row_of(p, ri, g, w, lane);
  if (!rc.valid) return;
  const uint32_t below = (1u << lane) - 1u;
  for (int s = 0; s < p.K; ++s) {
    const int pg = __ldg(idx + rc.r * p.K + s);
    if (pg < 0 || pg > rc.o) continue;
    const int64_t wi = ri.bm_base + (int64_t)(pg * p.Hkv + g) * ri.bm_words + w;
    const int pos = p.word_pos[wi] + __popc(p.bitmap[wi] & below);
    p.entries[pos] = make_int2((int)rc.r, (rc.t << 6) | s);
  }
}

}  // namespace

cudaError_t launch_inversion(const DevPlan& p, const int32_t* idx, float* lse,
                             int64_t lse_split_stride, cudaStream_t st) {
  cudaError_t e;
  e = cudaMemsetAsync(p.bitmap, 0, sizeof(uint32_t) * (size_t)p.bm_total_words, st);
  if (e != cudaSuccess) return e;
  const unsigned wgrid = (unsigned)((p.mark_warps + 7) / 8);
  if (wgrid > 0) {
    mark_kernel<<<wgrid, 256, 0, st>>>(p, idx, lse, lse_split_stride);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (p.num_chunks > 0) {
    count_kernel<<<(unsigned)p.num_chunks, 256, 0, st>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  scan_kernel<<<1, 1024, 0, st>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (p.num_chunks > 0) {
    prefix_kernel<<<(unsigned)p.num_chunks, 256, 0, st>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (wgrid > 0) {
    emit_kernel<<<wgrid, 256, 0, st>>>(p, idx);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace sps
