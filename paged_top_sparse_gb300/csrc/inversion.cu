// inversion.cu -- page -> (row, slot) inversion of the top-k selection, deterministic.
//
// The forward runs one work item per (page, KV head, query split) ("MSA PR 21: Q8KV4 paged
// sparse prefill", K1), so the row-major selection idx[row][slot] is turned around: for every
// bucket (request, logical page, KV head) the (row, slot) pairs that chose it, in ascending row
// order.  Nothing depends on the timing of atomics, and no global atomics touch the data:
//
//   1. count    a 256-thread block per (request, KV head, chunk of 256 consecutive rows of
//               the group), a thread per row.  Per window of 64 pages each thread turns its
//               row's selection (read as 16-byte vectors when top_k allows) into a 64-bit page
//               mask, and 64 ballots turn a warp's 32 masks around into one 32-bit row mask per
//               page; the block sums the popcounts of each page's 8 warp masks into that
//               (bucket, chunk)'s entry count.  Empty slots get lse = -inf here.
//   2. chunks   per bucket: exclusive scan over the bucket's chunks (bucket-local offsets)
//               and the bucket's total.
//   3. buckets  exclusive scan over the bucket totals, which gives the CSR offsets, and the
//               forward's work list (chunks of up to kFwdTaskGroups x 128 entries per bucket).
//   4. emit     a page's entries of the chunk start at the bucket's offset plus the chunk's
//               plus the rows of earlier warps, and a row's entry at that plus the set bits of
//               lower lanes.  An entry is (row, t * 64 + slot), t the row's absolute position,
//               so the forward needs no further lookup to find the row's own page and visible
//               key count.
//
// When every chunk's block fits on the GPU at once (the usual case), one cooperative launch
// runs all four steps (fused_kernel): the masks stay in shared memory and the selections in
// registers from step 1 to step 4, and bounded grid barriers separate the steps: with few
// buckets two (every block then does step 3 for all buckets itself), with many three (each
// block scans the buckets of its own range in step 2 and sums them, a barrier, each block
// offsets its range from the range sums, a barrier).  Otherwise (or when a request sees more
// than 1024 pages) four kernels run: count and emit (which rebuilds the masks) with a block per
// chunk and group of eight 64-page windows, so that a long request's windows are spread over
// the grid; between them the scan (step 2, a block per eight buckets, which also sums each
// block's range) and the offsets (step 3 on the same grid: each block offsets its buckets by
// the range sums before it).
#include "ptx.cuh"
#include "sps_internal.h"

namespace sps {
namespace {

// Block of steps 1 and 3 -> request, KV head and chunk of the bucket.  Returns -1 if none.
__device__ __forceinline__ int find_block(const DevPlan& p, int blk, int* g, int* c) {
  for (int b = 0; b < p.batch; ++b) {
    const ReqInfo& ri = p.reqs[b];
    const int n = p.Hkv * ri.ch_per_bucket;
    if (blk < ri.blk_base + n) {
      if (blk < ri.blk_base) return -1;
      const int local = blk - ri.blk_base;
      *g = local / ri.ch_per_bucket;
      *c = local % ri.ch_per_bucket;
      return b;
    }
  }
  return -1;
}

// Chunk c of bucket (page pg of request ri, KV head g).
__device__ __forceinline__ int chunk_id(const DevPlan& p, const ReqInfo& ri, int pg, int g,
                                        int c) {
  return ri.ch_base + (pg * p.Hkv + g) * ri.ch_per_bucket + c;
}

struct RowCtx {
  bool valid;
  int64_t r;
  int t;  // absolute position of the row's token
  int o;  // its own page
};

// Row of lane `lane` in 32-row word w of KV group g of request ri.
__device__ __forceinline__ RowCtx row_of(const DevPlan& p, const ReqInfo& ri, int g, int w,
                                         int lane) {
  RowCtx rc;
  const int row_local = w * 32 + lane;
  rc.valid = w < ri.words && row_local < ri.q_len * p.Hg;
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

// The selections of one row, held by its thread.  KV > 0: the first K of KV slots (K a
// multiple of 4, read as 16-byte vectors, the rest -1), two 16-bit values per register; a
// value outside [-1, 32767] is stored as -1 (negative: empty) or 32767 (past every own page:
// invalid), which keeps its meaning.  KV == 0: read from global memory at each use (any K).
template <int KV>
struct RowSel {
  uint32_t v[KV > 0 ? KV / 2 : 1];
  const int32_t* row;
  int K;
  static __device__ __forceinline__ uint32_t pack(int a, int b) {
    a = min(max(a, -1), 32767);
    b = min(max(b, -1), 32767);
    return ((uint32_t)a & 0xffffu) | ((uint32_t)b << 16);
  }
  __device__ __forceinline__ void load(const int32_t* idx, const RowCtx& rc, int k) {
    K = k;
    row = idx + rc.r * k;
    if (KV > 0) {
#pragma unroll
      for (int q = 0; q < KV / 4; ++q) {
        int4 x = make_int4(-1, -1, -1, -1);
        if (rc.valid && 4 * q < k) x = __ldg(reinterpret_cast<const int4*>(row) + q);
        v[2 * q] = pack(x.x, x.y);
        v[2 * q + 1] = pack(x.z, x.w);
      }
    }
  }
  __device__ __forceinline__ int n() const { return KV > 0 ? KV : K; }
  __device__ __forceinline__ int get(int s) const {
    if (KV > 0) return (int)(int16_t)(v[s >> 1] >> (16 * (s & 1)));
    return __ldg(row + s);
  }
};

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

static_assert(kChunkWords * 32 == 256, "a chunk is one 256-thread block, a warp per 32 rows");

// The row's valid selections in pages [p0, p0 + 64) as a bit mask (bit d: page p0 + d).
template <int KV>
__device__ __forceinline__ uint64_t row_mask(const RowSel<KV>& sel, const RowCtx& rc, int p0) {
  uint64_t m = 0;
  if (rc.valid) {
#pragma unroll
    for (int s = 0; s < sel.n(); ++s) {
      const int pg = sel.get(s);
      const int d = pg - p0;
      if (d >= 0 && d < kInvPages && pg <= rc.o) m |= 1ull << d;
    }
  }
  return m;
}

// Page masks of the block's rows for the windows w0 <= w < w1: tm[w - w0][d][v] bit l is set
// when row l of warp v selected page 64 w + d.  One window: each warp turns its 32 row masks
// around with 64 ballots.  Several: the masks are cleared and every selection ORs its lane's
// bit into its page's word (a row has at most top_k selections, while the ballots cost 64 per
// window; with one window the ballots win, since many lanes of a warp share pages, the own
// page above all, and their ORs to one word serialise).  Every thread of the block calls it.
template <int KV>
__device__ __forceinline__ void build_masks(uint32_t (*tm)[kInvPages][kChunkWords + 1], int w0,
                                            int w1, const RowSel<KV>& sel, const RowCtx& rc,
                                            int warp, int lane) {
  if (w1 - w0 == 1) {
    const uint64_t m = row_mask(sel, rc, w0 * kInvPages);
    uint32_t lo = 0, hi = 0;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const uint32_t b0 = __ballot_sync(0xffffffffu, (uint32_t)(m >> j) & 1u);
      const uint32_t b1 = __ballot_sync(0xffffffffu, (uint32_t)(m >> (j + 32)) & 1u);
      if (lane == j) {
        lo = b0;
        hi = b1;
      }
    }
    tm[0][lane][warp] = lo;
    tm[0][lane + 32][warp] = hi;
    __syncthreads();
    return;
  }
  uint32_t* flat = &tm[0][0][0];
  const int n = (w1 - w0) * kInvPages * (kChunkWords + 1);
  for (int i = threadIdx.x; i < n; i += blockDim.x) flat[i] = 0u;
  __syncthreads();
  if (rc.valid) {
#pragma unroll
    for (int s = 0; s < sel.n(); ++s) {
      const int pg = sel.get(s);
      if (pg < 0 || pg > rc.o) continue;
      const int w = pg / kInvPages;
      if (w < w0 || w >= w1) continue;
      atomicOr(&tm[w - w0][pg % kInvPages][warp], 1u << lane);
    }
  }
  __syncthreads();
}

// Windows of one block of the three-kernel form (blockIdx.y picks the group of the chunk's
// request's windows), so that a long request's windows are spread over the grid.
constexpr int kInvGroupWins = 8;

template <int KV>
__global__ void __launch_bounds__(256, 4)
count_kernel(DevPlan p, const int32_t* __restrict__ idx, float* __restrict__ lse,
             int64_t lse_split_stride) {
  __shared__ uint32_t tm[kInvGroupWins][kInvPages][kChunkWords + 1];
  int g, c;
  const int b = find_block(p, blockIdx.x, &g, &c);
  if (b < 0) return;  // uniform over the block
  const ReqInfo& ri = p.reqs[b];
  const int nwin = (ri.npages + kInvPages - 1) / kInvPages;
  const int w0 = (int)blockIdx.y * kInvGroupWins;
  if (w0 >= nwin) return;  // uniform
  const int w1 = min(nwin, w0 + kInvGroupWins);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const RowCtx rc = row_of(p, ri, g, c * kChunkWords + warp, lane);
  RowSel<KV> sel;
  sel.load(idx, rc, p.K);
  if (rc.valid && blockIdx.y == 0) {
#pragma unroll
    for (int s = 0; s < sel.n(); ++s) {
      if (s >= p.K) break;
      const int pg = sel.get(s);
      if (pg < 0) lse[s * lse_split_stride + rc.r] = -INFINITY;
      else if (pg > rc.o) set_status(p.status, DEV_BAD_INDEX);
    }
  }
  build_masks(tm, w0, w1, sel, rc, warp, lane);
  for (int i = threadIdx.x; i < (w1 - w0) * kInvPages; i += blockDim.x) {
    const int wi = i / kInvPages, d = i % kInvPages, pg = (w0 + wi) * kInvPages + d;
    if (pg < ri.npages) {
      int n = 0;
#pragma unroll 8
      for (int v = 0; v < kChunkWords; ++v) n += __popc(tm[wi][d][v]);
      p.chunk_offsets[chunk_id(p, ri, pg, g, c)] = n;  // a count until step 2
    }
  }
}

// Step 2: a block per eight buckets turns their chunk counts into bucket-local exclusive
// offsets (a warp per bucket of at most 32 chunks, the block for larger ones) and leaves each
// bucket's total in bucket_offsets[bucket]; the last block to finish runs step 3.
constexpr int kScanBuckets = kInvScanBuckets;

__global__ void __launch_bounds__(256) scan_kernel(DevPlan p) {
  __shared__ int sh[32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bk0 = (int)blockIdx.x * kScanBuckets;
  // a bucket of at most 32 chunks: one warp, lane i holding chunk i
  if (bk0 + warp < p.num_buckets) {
    const int bk = bk0 + warp, gp = bk / p.Hkv, g = bk % p.Hkv;
    const ReqInfo& ri = p.reqs[p.page_req[gp]];
    const int n = ri.ch_per_bucket;
    if (n <= 32) {
      int32_t* cnt = p.chunk_offsets + chunk_id(p, ri, gp - ri.page_base, g, 0);
      const int x = lane < n ? cnt[lane] : 0;
      int incl = x;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += y;
      }
      if (lane < n) cnt[lane] = incl - x;
      const int total = __shfl_sync(0xffffffffu, incl, 31);
      if (lane == 0) p.bucket_offsets[bk] = total;
    }
  }
  // larger buckets: the whole block, one after another (the same test for every thread)
  for (int j = 0; j < kScanBuckets && bk0 + j < p.num_buckets; ++j) {
    const int bk = bk0 + j, gp = bk / p.Hkv, g = bk % p.Hkv;
    const ReqInfo& ri = p.reqs[p.page_req[gp]];
    const int n = ri.ch_per_bucket;
    if (n <= 32) continue;
    int32_t* cnt = p.chunk_offsets + chunk_id(p, ri, gp - ri.page_base, g, 0);
    const int per = (n + 255) / 256;
    const int i0 = threadIdx.x * per, i1 = min(n, i0 + per);
    int x = 0;
    for (int i = i0; i < i1; ++i) x += cnt[i];
    int off;
    const int total = block_exclusive_scan(x, &off, sh);
    for (int i = i0; i < i1; ++i) {
      const int v = cnt[i];
      cnt[i] = off;
      off += v;
    }
    if (threadIdx.x == 0) p.bucket_offsets[bk] = total;
  }
  __syncthreads();
  // this block's range: its buckets' entries and work items
  if (warp == 0) {
    const int bk = bk0 + lane;
    const int per_task = kFwdTaskGroups * 128;
    const int t = lane < kScanBuckets && bk < p.num_buckets ? p.bucket_offsets[bk] : 0;
    int c = t, n = (t + per_task - 1) / per_task;
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) {
      c += __shfl_xor_sync(0xffffffffu, c, d);
      n += __shfl_xor_sync(0xffffffffu, n, d);
    }
    if (lane == 0) {
      p.range_sums[blockIdx.x] = c;
      p.range_sums[gridDim.x + blockIdx.x] = n;
    }
  }
}

// Step 3 of the multi-kernel form, on the scan's grid: each block offsets its buckets by the
// range sums of the blocks before it and writes their CSR offsets and work items; block 0 also
// the total.
__global__ void __launch_bounds__(256) offsets_kernel(DevPlan p) {
  __shared__ int sh[32];
  const int G = gridDim.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int cnt = 0, ntask = 0, tot = 0, ttot = 0;
  for (int b = threadIdx.x; b < G; b += blockDim.x) {
    const int c = p.range_sums[b], t = p.range_sums[G + b];
    tot += c;
    ttot += t;
    if (b < (int)blockIdx.x) {
      cnt += c;
      ntask += t;
    }
  }
  int unused;
  cnt = block_exclusive_scan(cnt, &unused, sh);
  ntask = block_exclusive_scan(ntask, &unused, sh);
  tot = block_exclusive_scan(tot, &unused, sh);
  ttot = block_exclusive_scan(ttot, &unused, sh);
  if (warp != 0) return;
  const int per_task = kFwdTaskGroups * 128;
  const int bk = (int)blockIdx.x * kScanBuckets + lane;
  const bool mine = lane < kScanBuckets && bk < p.num_buckets;
  const int t = mine ? p.bucket_offsets[bk] : 0;
  const int nt = (t + per_task - 1) / per_task;
  int o = t, to = nt;  // inclusive scans over the block's buckets
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, o, d), z = __shfl_up_sync(0xffffffffu, to, d);
    if (lane >= d) {
      o += y;
      to += z;
    }
  }
  o += cnt - t;
  to += ntask - nt;
  if (mine) {
    p.bucket_offsets[bk] = o;
    for (int j = 0; j < nt; ++j) {
      if (to + j < p.max_fwd_tasks) {
        FwdTask ft;
        ft.bucket = bk;
        ft.entry_begin = o + j * per_task;
        ft.count = min(per_task, t - j * per_task);
        ft.pad = 0;
        p.fwd_tasks[to + j] = ft;
      }
    }
  }
  if (blockIdx.x == 0 && lane == 0) {
    p.bucket_offsets[p.num_buckets] = tot;
    if (tot > p.max_entries) set_status(p.status, DEV_OVERFLOW);
    p.counters[2] = min(ttot, p.max_fwd_tasks);
    if (ttot > p.max_fwd_tasks) set_status(p.status, DEV_OVERFLOW);
  }
}

template <int KV>
__global__ void __launch_bounds__(256, 4)
emit_kernel(DevPlan p, const int32_t* __restrict__ idx) {
  __shared__ uint32_t tm[kInvGroupWins][kInvPages][kChunkWords + 1];
  __shared__ int pos0[kInvGroupWins][kInvPages][kChunkWords + 1];  // first entry of (page, warp)
  pdl_trigger();  // the forward that follows may start its prologue
  int g, c;
  const int b = find_block(p, blockIdx.x, &g, &c);
  if (b < 0) return;  // uniform over the block
  const ReqInfo& ri = p.reqs[b];
  const int nwin = (ri.npages + kInvPages - 1) / kInvPages;
  const int w0 = (int)blockIdx.y * kInvGroupWins;
  if (w0 >= nwin) return;  // uniform
  const int w1 = min(nwin, w0 + kInvGroupWins);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const RowCtx rc = row_of(p, ri, g, c * kChunkWords + warp, lane);
  RowSel<KV> sel;
  sel.load(idx, rc, p.K);
  const uint32_t below = (1u << lane) - 1u;
  build_masks(tm, w0, w1, sel, rc, warp, lane);
  for (int i = threadIdx.x; i < (w1 - w0) * kInvPages; i += blockDim.x) {
    const int wi = i / kInvPages, d = i % kInvPages, pg = (w0 + wi) * kInvPages + d;
    if (pg < ri.npages) {
      const int bk = (ri.page_base + pg) * p.Hkv + g;
      int acc = p.bucket_offsets[bk] + p.chunk_offsets[chunk_id(p, ri, pg, g, c)];
      for (int v = 0; v < kChunkWords; ++v) {
        pos0[wi][d][v] = acc;
        acc += __popc(tm[wi][d][v]);
      }
    }
  }
  __syncthreads();
  if (rc.valid) {
#pragma unroll
    for (int s = 0; s < sel.n(); ++s) {
      const int pg = sel.get(s);
      if (pg < 0 || pg > rc.o) continue;
      const int w = pg / kInvPages;
      if (w < w0 || w >= w1) continue;
      const int wi = w - w0, d = pg % kInvPages;
      const int pos = pos0[wi][d][warp] + __popc(tm[wi][d][warp] & below);
      p.entries[pos] = make_int2((int)rc.r, (rc.t << 6) | s);
    }
  }
}

// Step 2 for one bucket, by the whole block: its chunk counts (written by other blocks, so read
// past L1) become bucket-local exclusive offsets, and its total goes to bucket_totals.
__device__ __forceinline__ void scan_bucket_block(const DevPlan& p, int bk, int* sh) {
  const int gp = bk / p.Hkv, gg = bk % p.Hkv;
  const ReqInfo& rb = p.reqs[p.page_req[gp]];
  int32_t* cnt = p.chunk_offsets + chunk_id(p, rb, gp - rb.page_base, gg, 0);
  const int n = rb.ch_per_bucket;
  const int per = (n + 255) / 256;
  const int i0 = threadIdx.x * per, i1 = min(n, i0 + per);
  int x = 0;
  for (int i = i0; i < i1; ++i) x += __ldcg(cnt + i);
  int off;
  const int total = block_exclusive_scan(x, &off, sh);
  for (int i = i0; i < i1; ++i) {
    const int v = __ldcg(cnt + i);
    cnt[i] = off;
    off += v;
  }
  if (threadIdx.x == 0) p.bucket_totals[bk] = total;
}

// The same by one warp, for a bucket of at most 32 chunks (lane i holds chunk i).
__device__ __forceinline__ void scan_bucket_warp(const DevPlan& p, int bk, int lane) {
  const int gp = bk / p.Hkv, gg = bk % p.Hkv;
  const ReqInfo& rb = p.reqs[p.page_req[gp]];
  int32_t* cnt = p.chunk_offsets + chunk_id(p, rb, gp - rb.page_base, gg, 0);
  const int n = rb.ch_per_bucket;
  const int x = lane < n ? __ldcg(cnt + lane) : 0;
  int incl = x;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += y;
  }
  if (lane < n) cnt[lane] = incl - x;
  const int total = __shfl_sync(0xffffffffu, incl, 31);
  if (lane == 0) p.bucket_totals[bk] = total;
}

// All the steps in one cooperative launch, one block per chunk (as count_kernel): the page
// masks of every window stay in shared memory and the row's selections in registers from
// the count to the emit, and two grid barriers replace the kernel boundaries.  After the
// second, every block scans the bucket totals itself, so no single block has to publish the
// bucket offsets before the others can emit.
template <int KV>
__global__ void __launch_bounds__(256, 8)
fused_kernel(DevPlan p, const int32_t* __restrict__ idx, float* __restrict__ lse,
             int64_t lse_split_stride, int nwin) {
  extern __shared__ uint32_t dyn[];
  uint32_t (*tmw)[kInvPages][kChunkWords + 1] =
      reinterpret_cast<uint32_t (*)[kInvPages][kChunkWords + 1]>(dyn);  // [nwin]
  int (*pos0)[kInvPages][kChunkWords + 1] =  // [nwin]: first entry of (page, warp)
      reinterpret_cast<int (*)[kInvPages][kChunkWords + 1]>(
          dyn + (size_t)nwin * kInvPages * (kChunkWords + 1));
  __shared__ int sh[32];
  __shared__ int flag;
  unsigned int* bar = reinterpret_cast<unsigned int*>(p.counters + 4);
  pdl_trigger();  // the forward that follows may start its prologue
  int g = 0, c = 0;
  const int b = find_block(p, blockIdx.x, &g, &c);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int per_task = kFwdTaskGroups * 128;
  // ---- 1. count
  RowCtx rc{};
  RowSel<KV> sel;
  const ReqInfo* ri = b >= 0 ? &p.reqs[b] : nullptr;
  if (ri) {
    rc = row_of(p, *ri, g, c * kChunkWords + warp, lane);
    sel.load(idx, rc, p.K);
    if (rc.valid) {
#pragma unroll
      for (int s = 0; s < sel.n(); ++s) {
        if (s >= p.K) break;
        const int pg = sel.get(s);
        if (pg < 0) lse[s * lse_split_stride + rc.r] = -INFINITY;
        else if (pg > rc.o) set_status(p.status, DEV_BAD_INDEX);
      }
    }
    build_masks(tmw, 0, (ri->npages + kInvPages - 1) / kInvPages, sel, rc, warp, lane);
    for (int wi = 0; wi * kInvPages < ri->npages; ++wi) {
      const int d = threadIdx.x, p0 = wi * kInvPages;
      if (d < kInvPages && p0 + d < ri->npages) {
        int n = 0;
#pragma unroll 8
        for (int v = 0; v < kChunkWords; ++v) n += __popc(tmw[wi][d][v]);
        p.chunk_offsets[chunk_id(p, *ri, p0 + d, g, c)] = n;
      }
    }
  }
  if (!grid_barrier(bar, p.status, &flag)) return;
  // ---- 2. chunk offsets within each bucket, bucket totals.  Few buckets: a block per bucket,
  // then a grid barrier.  Many: each block takes the buckets of its own range of step 3 (a
  // warp per bucket of at most 32 chunks, the whole block for larger ones), so that its range
  // sums (3a) follow without a grid barrier between them.
  const int nb = p.num_buckets;
  const bool few = nb <= 2 * (int)blockDim.x;
  const int G = gridDim.x;
  const int rper = (nb + G - 1) / G;  // buckets of each block's range (many buckets)
  const int r0 = few ? 0 : min(nb, blockIdx.x * rper), r1 = few ? 0 : min(nb, r0 + rper);
  if (few) {
    for (int bk = blockIdx.x; bk < nb; bk += G) scan_bucket_block(p, bk, sh);
    if (!grid_barrier(bar, p.status, &flag)) return;
  } else {
    for (int bk = r0 + warp; bk < r1; bk += blockDim.x / 32)
      if (p.reqs[p.page_req[bk / p.Hkv]].ch_per_bucket <= 32) scan_bucket_warp(p, bk, lane);
    for (int bk = r0; bk < r1; ++bk)  // the same condition for every thread of the block
      if (p.reqs[p.page_req[bk / p.Hkv]].ch_per_bucket > 32) scan_bucket_block(p, bk, sh);
    __syncthreads();  // the range's totals are written
  }
  // ---- 3. exclusive scans over the bucket totals (entries and work items), which give every
  // bucket's CSR offset and its work items.  Few buckets: every block scans them all and keeps
  // the offsets of its own buckets (its request and KV head, every page) for the emit.  Many
  // buckets (more than two per thread): each block sums its own range of buckets (the ones it
  // scanned in step 2), a grid barrier, then each block scans the ranges' sums (one per block),
  // writes its range's offsets and work items, and after another barrier reads its own
  // buckets' offsets.
  __shared__ int s_boff[kInvFusedMaxPages];  // CSR offset of page pg's bucket of this block's KV head
  const int own0 = ri ? ri->page_base * p.Hkv + g : -1;  // this block's bucket of page 0
  if (few) {
    const int per = (nb + 255) / 256;
    const int b0 = threadIdx.x * per, b1 = min(nb, b0 + per);
    int cnt = 0, ntask = 0;
    for (int bk = b0; bk < b1; ++bk) {
      const int t = __ldcg(p.bucket_totals + bk);
      cnt += t;
      ntask += (t + per_task - 1) / per_task;
    }
    int o, to;
    const int total = block_exclusive_scan(cnt, &o, sh);
    const int ttotal = block_exclusive_scan(ntask, &to, sh);
    for (int bk = b0; bk < b1; ++bk) {
      const int t = __ldcg(p.bucket_totals + bk);
      const int nt = (t + per_task - 1) / per_task;
      if (bk % (int)gridDim.x == (int)blockIdx.x) {
        p.bucket_offsets[bk] = o;
        for (int j = 0; j < nt; ++j) {
          if (to + j < p.max_fwd_tasks) {
            FwdTask ft;
            ft.bucket = bk;
            ft.entry_begin = o + j * per_task;
            ft.count = min(per_task, t - j * per_task);
            ft.pad = 0;
            p.fwd_tasks[to + j] = ft;
          }
        }
      }
      if (ri && bk >= own0 && (bk - own0) % p.Hkv == 0 && (bk - own0) / p.Hkv < ri->npages)
        s_boff[(bk - own0) / p.Hkv] = o;
      o += t;
      to += nt;
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) {
      p.bucket_offsets[nb] = total;
      if (total > p.max_entries) set_status(p.status, DEV_OVERFLOW);
      p.counters[2] = min(ttotal, p.max_fwd_tasks);
      if (ttotal > p.max_fwd_tasks) set_status(p.status, DEV_OVERFLOW);
    }
  } else {
    // 3a. this block's range: its sums of entries and of work items
    {
      int cnt = 0, ntask = 0;
      for (int bk = r0 + threadIdx.x; bk < r1; bk += blockDim.x) {
        const int t = __ldcg(p.bucket_totals + bk);
        cnt += t;
        ntask += (t + per_task - 1) / per_task;
      }
      int unused;
      const int rc = block_exclusive_scan(cnt, &unused, sh);
      const int rt = block_exclusive_scan(ntask, &unused, sh);
      if (threadIdx.x == 0) {
        p.range_sums[blockIdx.x] = rc;
        p.range_sums[G + blockIdx.x] = rt;
      }
    }
    if (!grid_barrier(bar, p.status, &flag)) return;
    // 3b. the ranges before this one give its first offset and first work item
    {
      int cnt = 0, ntask = 0, tot = 0, ttot = 0;
      for (int b = threadIdx.x; b < G; b += blockDim.x) {
        const int c = __ldcg(p.range_sums + b), t = __ldcg(p.range_sums + G + b);
        tot += c;
        ttot += t;
        if (b < (int)blockIdx.x) {
          cnt += c;
          ntask += t;
        }
      }
      int unused;
      const int base = block_exclusive_scan(cnt, &unused, sh);
      const int tbase = block_exclusive_scan(ntask, &unused, sh);
      const int total = block_exclusive_scan(tot, &unused, sh);
      const int ttotal = block_exclusive_scan(ttot, &unused, sh);
      // the range's own scan: thread i takes buckets r0 + i per .. (a few each)
      const int per = (r1 - r0 + (int)blockDim.x - 1) / (int)blockDim.x;
      const int b0 = r0 + threadIdx.x * per, b1 = min(r1, b0 + per);
      int c2 = 0, n2 = 0;
      for (int bk = b0; bk < b1; ++bk) {
        const int t = __ldcg(p.bucket_totals + bk);
        c2 += t;
        n2 += (t + per_task - 1) / per_task;
      }
      int o, to;
      block_exclusive_scan(c2, &o, sh);
      block_exclusive_scan(n2, &to, sh);
      o += base;
      to += tbase;
      for (int bk = b0; bk < b1; ++bk) {
        const int t = __ldcg(p.bucket_totals + bk);
        const int nt = (t + per_task - 1) / per_task;
        p.bucket_offsets[bk] = o;
        for (int j = 0; j < nt; ++j) {
          if (to + j < p.max_fwd_tasks) {
            FwdTask ft;
            ft.bucket = bk;
            ft.entry_begin = o + j * per_task;
            ft.count = min(per_task, t - j * per_task);
            ft.pad = 0;
            p.fwd_tasks[to + j] = ft;
          }
        }
        o += t;
        to += nt;
      }
      if (blockIdx.x == 0 && threadIdx.x == 0) {
        p.bucket_offsets[nb] = total;
        if (total > p.max_entries) set_status(p.status, DEV_OVERFLOW);
        p.counters[2] = min(ttotal, p.max_fwd_tasks);
        if (ttotal > p.max_fwd_tasks) set_status(p.status, DEV_OVERFLOW);
      }
    }
    if (!grid_barrier(bar, p.status, &flag)) return;
    // 3c. this block's own buckets' offsets, for the emit
    if (ri)
      for (int pg = threadIdx.x; pg < ri->npages; pg += blockDim.x)
        s_boff[pg] = __ldcg(p.bucket_offsets + own0 + pg * p.Hkv);
  }
  __syncthreads();
  // ---- 4. emit: every (page, warp) start of the request's windows in one pass, then each
  // selection's entry
  if (!ri) return;
  for (int pg = threadIdx.x; pg < ri->npages; pg += blockDim.x) {
    const int wi = pg / kInvPages, d = pg % kInvPages;
    int acc = s_boff[pg] + __ldcg(p.chunk_offsets + chunk_id(p, *ri, pg, g, c));
    for (int v = 0; v < kChunkWords; ++v) {
      pos0[wi][d][v] = acc;
      acc += __popc(tmw[wi][d][v]);
    }
  }
  __syncthreads();
  if (rc.valid) {
    const uint32_t below = (1u << lane) - 1u;
#pragma unroll
    for (int s = 0; s < sel.n(); ++s) {
      const int pg = sel.get(s);
      if (pg < 0 || pg > rc.o) continue;
      const int wi = pg / kInvPages, d = pg % kInvPages;
      const int pos = pos0[wi][d][warp] + __popc(tmw[wi][d][warp] & below);
      p.entries[pos] = make_int2((int)rc.r, (rc.t << 6) | s);
    }
  }
}

template <int KV>
bool try_fused(const DevPlan& p, const int32_t* idx, float* lse, int64_t lse_split_stride,
               cudaStream_t st, cudaError_t* err) {
  // max_pages bounds every request's page count, so it sizes the 64-page windows and must fit
  // the per-block offset table
  if (p.max_pages > kInvFusedMaxPages) return false;
  const int nwin = (p.max_pages + kInvPages - 1) / kInvPages;
  const size_t dsmem = (size_t)2 * nwin * kInvPages * (kChunkWords + 1) * sizeof(uint32_t);
  auto kern = fused_kernel<KV>;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 256, dsmem) != cudaSuccess) {
    (void)cudaGetLastError();
    return false;
  }
  if ((int64_t)per_sm * num_sms() < p.inv_blocks || p.inv_blocks < 1) return false;
  DevPlan pc = p;
  int64_t lss = lse_split_stride;
  int nw = nwin;
  void* args[] = {&pc, const_cast<int32_t**>(&idx), &lse, &lss, &nw};
  *err = cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(kern), dim3(p.inv_blocks),
                                     dim3(256), args, dsmem, st);
  if (*err == cudaErrorCooperativeLaunchTooLarge) {
    (void)cudaGetLastError();
    return false;
  }
  return true;
}

}  // namespace

cudaError_t launch_inversion(const DevPlan& p, const int32_t* idx, float* lse,
                             int64_t lse_split_stride, cudaStream_t st) {
  cudaError_t e;
  // selections held in registers when top_k is a multiple of 4 up to 16
  const int kv = (p.K % 4 == 0 && p.K <= 16) ? 16 : 0;
  // one cooperative launch when every chunk's block fits on the GPU at once
  if (kv == 16 ? try_fused<16>(p, idx, lse, lse_split_stride, st, &e)
               : try_fused<0>(p, idx, lse, lse_split_stride, st, &e))
    return e;
  // a block per (chunk, group of kInvGroupWins windows of the chunk's request)
  const dim3 grid((unsigned)p.inv_blocks,
                  (unsigned)((p.max_pages + kInvPages * kInvGroupWins - 1) / (kInvPages * kInvGroupWins)));
  const unsigned nblk = (unsigned)p.inv_blocks;
  if (nblk > 0) {
    if (kv == 16) count_kernel<16><<<grid, 256, 0, st>>>(p, idx, lse, lse_split_stride);
    else count_kernel<0><<<grid, 256, 0, st>>>(p, idx, lse, lse_split_stride);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  const unsigned nscan = (unsigned)((p.num_buckets + kScanBuckets - 1) / kScanBuckets);
  scan_kernel<<<nscan, 256, 0, st>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  offsets_kernel<<<nscan, 256, 0, st>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (nblk > 0) {
    if (kv == 16) emit_kernel<16><<<grid, 256, 0, st>>>(p, idx);
    else emit_kernel<0><<<grid, 256, 0, st>>>(p, idx);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace sps
