// inversion.cu -- page -> (row, slot) inversion of the top-k selection, deterministic.
//
// The forward runs one work item per (page, KV head, query split) ("MSA PR 21: Q8KV4 paged
// sparse prefill", K1), so the row-major selection idx[row][slot] is turned around: for every
// bucket (request, logical page, KV head) the (row, slot) pairs that chose it, in ascending row
// order.  The order never depends on atomic timing:
//
//   1. mark     a warp per 32 consecutive rows of one (request, KV head) sets one bit per
//               (bucket, row) in a selection bitmap (warp-aggregated atomicOr of the lanes'
//               own bits); empty slots get lse = -inf here.
//   2. count    a block per bucket: popcount of its bitmap words.
//   3. scan     one block: exclusive scan of the bucket counts -> CSR offsets, then the list
//               of forward work items (chunks of up to kFwdTaskGroups x 128 entries).
//   4. fill     a block per bucket: popcount prefix over the bucket's bitmap words gives each
//               set bit its rank; its slot is found by binary search in the row's ascending
//               selection.
#include "ptx.cuh"
#include "sps_internal.h"

namespace sps {
namespace {

__device__ __forceinline__ int find_request(const DevPlan& p, int64_t warp_id, int* w_in_req,
                                            int* g) {
  // warps of request b: H_kv * bm_words consecutive warp ids
  int64_t acc = 0;
  for (int b = 0; b < p.batch; ++b) {
    const int nw = p.reqs[b].bm_words;
    const int64_t n = (int64_t)p.Hkv * nw;
    if (warp_id < acc + n) {
      const int64_t local = warp_id - acc;
      *g = (int)(local / nw);
      *w_in_req = (int)(local % nw);
      return b;
    }
    acc += n;
  }
  return -1;
}

__global__ void __launch_bounds__(256)
mark_kernel(DevPlan p, const int32_t* __restrict__ idx, float* __restrict__ lse,
            int64_t lse_split_stride, int64_t total_warps) {
  const int64_t wid = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (wid >= total_warps) return;
  int w, g;
  const int b = find_request(p, wid, &w, &g);
  if (b < 0) return;
  const ReqInfo ri = p.reqs[b];
  const int row_local = w * 32 + lane;
  const bool valid = row_local < ri.q_len * p.Hg;
  int64_t r = 0;
  int o = -1;
  if (valid) {
    const int i = row_local / p.Hg, hl = row_local % p.Hg;
    r = (int64_t)(ri.tok0 + i) * p.H + g * p.Hg + hl;
    o = (ri.ctx + i) >> 7;
  }
  for (int s = 0; s < p.K; ++s) {
    int pg = valid ? __ldg(idx + r * p.K + s) : -1;
    if (valid && pg < 0) lse[s * lse_split_stride + r] = -INFINITY;
    if (valid && pg > o) {
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

// Block-wide exclusive scan of one int per thread (1024 threads); returns the block total.
__device__ __forceinline__ int block_exclusive_scan(int v, int* out, int* sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, d);
    if (lane >= d) x += y;
  }
  if (lane == 31) sh[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int s = lane < (int)(blockDim.x >> 5) ? sh[lane] : 0;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, s, d);
      if (lane >= d) s += y;
    }
    sh[lane] = s;  // inclusive warp totals
  }
  __syncthreads();
  const int warp_prefix = warp ? sh[warp - 1] : 0;
  const int total = sh[(blockDim.x >> 5) - 1];
  *out = warp_prefix + x - v;
  __syncthreads();
  return total;
}

__global__ void __launch_bounds__(1024) scan_kernel(DevPlan p) {
  __shared__ int sh[32];
  const int nb = p.num_buckets;
  const int per = (nb + 1023) / 1024;
  const int b0 = threadIdx.x * per;
  const int per_task = kFwdTaskGroups * 128;
  int cnt = 0, ntask = 0;
  for (int b = b0; b < b0 + per && b < nb; ++b) {
    const int c = p.bucket_count[b];
    cnt += c;
    ntask += (c + per_task - 1) / per_task;
  }
  int off, toff;
  const int total = block_exclusive_scan(cnt, &off, sh);
  const int ttotal = block_exclusive_scan(ntask, &toff, sh);
  for (int b = b0; b < b0 + per && b < nb; ++b) {
    const int c = p.bucket_count[b];
    p.bucket_offsets[b] = off;
    for (int e = 0; e < c; e += per_task) {
      if (toff < p.max_fwd_tasks) {
        FwdTask t;
        t.bucket = b;
        t.entry_begin = off + e;
        t.count = min(per_task, c - e);
        t.pad = 0;
        p.fwd_tasks[toff] = t;
      }
      ++toff;
    }
    off += c;
  }
  if (threadIdx.x == 0) {
    p.bucket_offsets[nb] = total;
    p.counters[2] = min(ttotal, p.max_fwd_tasks);
    if (ttotal > p.max_fwd_tasks || total > p.max_entries) set_status(p.status, DEV_OVERFLOW);
  }
}

// Bitmap words of bucket `bucket` and its request.
__device__ __forceinline__ const uint32_t* bucket_words(const DevPlan& p, int bucket, ReqInfo* ri,
                                                       int* pg, int* g) {
  const int gp = bucket / p.Hkv;
  *g = bucket % p.Hkv;
  *ri = p.reqs[p.page_req[gp]];
  *pg = gp - ri->page_base;
  return p.bitmap + ri->bm_base + (int64_t)(*pg * p.Hkv + *g) * ri->bm_words;
}

__global__ void __launch_bounds__(256) count_kernel(DevPlan p) {
  __shared__ int sh[8];
  ReqInfo ri;
  int pg, g;
  const uint32_t* words = bucket_words(p, blockIdx.x, &ri, &pg, &g);
  int c = 0;
  for (int w = threadIdx.x; w < ri.bm_words; w += blockDim.x) c += __popc(words[w]);
  c = __reduce_add_sync(0xffffffffu, c);
  if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = c;
  __syncthreads();
  if (threadIdx.x == 0) {
    int t = 0;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) t += sh[i];
    p.bucket_count[blockIdx.x] = t;
  }
}

__global__ void __launch_bounds__(256)
fill_kernel(DevPlan p, const int32_t* __restrict__ idx) {
  __shared__ int sh[32];
  const int bucket = blockIdx.x;
  ReqInfo ri;
  int pg, g;
  const uint32_t* words = bucket_words(p, bucket, &ri, &pg, &g);
  const int nw = ri.bm_words;
  const int per = (nw + blockDim.x - 1) / blockDim.x;
  const int w0 = threadIdx.x * per;
  int cnt = 0;
  for (int w = w0; w < w0 + per && w < nw; ++w) cnt += __popc(words[w]);
  int rank;
  // block_exclusive_scan expects up to 32 warps; 256 threads = 8 warps
  block_exclusive_scan(cnt, &rank, sh);
  int2* dst = p.entries + p.bucket_offsets[bucket];
  for (int w = w0; w < w0 + per && w < nw; ++w) {
    uint32_t bits = words[w];
    while (bits) {
      const int bit = __ffs(bits) - 1;
      bits &= bits - 1;
      const int row_local = w * 32 + bit;
      const int i = row_local / p.Hg, hl = row_local % p.Hg;
      const int64_t r = (int64_t)(ri.tok0 + i) * p.H + g * p.Hg + hl;
      // slot of pg in the row's ascending selection (entries past n_sel are -1)
      const int o = (ri.ctx + i) >> 7;
      int lo = 0, hi = min(p.K, o + 1) - 1;
      const int32_t* row = idx + r * p.K;
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (__ldg(row + mid) < pg) lo = mid + 1;
        else hi = mid;
      }
      dst[rank++] = make_int2((int)r, lo);
    }
  }
}

}  // namespace

cudaError_t launch_inversion(const DevPlan& p, const int32_t* idx, float* lse,
                             int64_t lse_split_stride, cudaStream_t st) {
  cudaError_t e;
  e = cudaMemsetAsync(p.bitmap, 0, sizeof(uint32_t) * (size_t)p.bm_total_words, st);
  if (e != cudaSuccess) return e;
  if (p.mark_warps > 0) {
    mark_kernel<<<(unsigned)((p.mark_warps + 7) / 8), 256, 0, st>>>(p, idx, lse, lse_split_stride,
                                                                   p.mark_warps);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (p.num_buckets > 0) {
    count_kernel<<<(unsigned)p.num_buckets, 256, 0, st>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  scan_kernel<<<1, 1024, 0, st>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (p.num_buckets > 0) {
    fill_kernel<<<(unsigned)p.num_buckets, 256, 0, st>>>(p, idx);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace sps
