// topk.cu -- per-row top-k page selection, one warp per row.
//
// Contract (the method's page selection: every row attends its own page, the one page the
// forward of "MSA PR 21: Q8KV4 paged sparse prefill", K1 Softmax, masks causally; "MSA PR 36:
// Q8KV8 prefill indexer", Kernel performance, relies on a bitwise-stable selection): the row's
// own page o is always kept; the other
// n_sel - 1 = min(k, o+1) - 1 pages are the best by (score descending, page ascending), with
// -0.0 equal to +0.0; output in ascending page order, padded with -1.
//
// Scores become 32-bit order-preserving keys.  Lane l holds the E adjacent pages E l .. E l + E-1,
// sorted best-first once (bitonic network in registers), so any page of a lower lane is lower
// than every page of a higher lane.  A selection round is then one warp max-reduction
// (redux.sync) of the lanes' head keys: the lane whose head holds the maximum takes that page
// and shifts its next candidate up.  The rounds first run as if no two heads were ever equal
// (no ballot); the lanes' take counts then sum to n_sel - 1 exactly when no round had a tie,
// and otherwise the rounds run again with ties going to the lowest such lane (the lower page).
// The kernel is bound by ALU issue, so the tie-free pass is what most rows pay.  After the
// rounds a popc prefix writes the chosen pages in ascending order.  Rows of more than 128 pages
// first filter their keys down to at most 64 candidates (see topk_filter_kernel: pages dealt
// to the lanes round-robin, so that every lane is busy and loads are contiguous) and run the
// rounds on those.
#include "ptx.cuh"
#include "sps_internal.h"

namespace sps {
namespace {

// Order-preserving map of a non-NaN float to uint32 (larger float -> larger key, never 0);
// -0.0 is first turned into +0.0 so the two compare equal.
__device__ __forceinline__ uint32_t score_key(float f) {
  uint32_t u = __float_as_uint(f + 0.0f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Sorts a lane's E candidates (key, page offset) best-first: larger key, then lower page.
template <int E>
__device__ __forceinline__ void sort_best_first(uint32_t (&k)[E], uint32_t (&pg)[E]) {
#pragma unroll
  for (int size = 2; size <= E; size <<= 1)
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1)
#pragma unroll
      for (int i = 0; i < E; ++i) {
        const int l = i ^ stride;
        if (l > i) {
          const bool l_better = k[l] > k[i] || (k[l] == k[i] && pg[l] < pg[i]);
          if (l_better == ((i & size) == 0)) {  // best-first runs where bit `size` of i is 0
            const uint32_t tk = k[i], tp = pg[i];
            k[i] = k[l]; pg[i] = pg[l];
            k[l] = tk; pg[l] = tp;
          }
        }
      }
}

// K - 1 selection rounds over the lanes' best-first candidate lists, assuming no two lanes
// ever show equal heads: the lane whose head equals the warp maximum takes it.  Returns how
// many of its candidates this lane took; the counts sum to K - 1 exactly when no round had a
// tie (a tie makes every holder advance), which the caller checks.  `key` is not modified.
template <int E, int KC>
__device__ __forceinline__ int rounds_distinct_heads(const uint32_t (&key)[E], int K) {
  uint32_t h[E];
#pragma unroll
  for (int j = 0; j < E; ++j) h[j] = key[j];
  int c = 0;
#pragma unroll (KC ? KC : 4)
  for (int round = 1; round < K; ++round) {
    const uint32_t m = __reduce_max_sync(0xffffffffu, h[0]);
    if (h[0] == m) {
      ++c;
#pragma unroll
      for (int j = 0; j + 1 < E; ++j) h[j] = h[j + 1];
      h[E - 1] = 0u;
    }
  }
  return c;
}

// The same rounds with ties resolved: of the lanes whose head equals the maximum, the lowest
// (it holds the lowest page) takes it.
template <int E, int KC>
__device__ __forceinline__ int rounds_lowest_lane(const uint32_t (&key)[E], int K, int lane) {
  uint32_t h[E];
#pragma unroll
  for (int j = 0; j < E; ++j) h[j] = key[j];
  const uint32_t lt = (1u << lane) - 1u;
  int c = 0;
#pragma unroll 4
  for (int round = 1; round < K; ++round) {
    const uint32_t m = __reduce_max_sync(0xffffffffu, h[0]);
    const uint32_t tie = __ballot_sync(0xffffffffu, h[0] == m);
    if (h[0] == m && (tie & lt) == 0) {
      ++c;
#pragma unroll
      for (int j = 0; j + 1 < E; ++j) h[j] = h[j + 1];
      h[E - 1] = 0u;
    }
  }
  return c;
}

// KC: top_k fixed at compile time (the rounds unroll completely), or 0 for any top_k.
template <int E, int KC = 0>  // pages per lane: max_pages <= 32 * E
__global__ void __launch_bounds__(256)
topk_kernel(DevPlan p, const float* __restrict__ scores, int64_t pitch, int32_t* __restrict__ idx) {
  pdl_wait();  // the scores come from the indexer just before
  const int lane = threadIdx.x & 31;
  const uint32_t r = blockIdx.x * 8u + (threadIdx.x >> 5);
  if (r >= (uint32_t)p.T * (uint32_t)p.H) return;
  const int o = __ldg(p.tok_pos + r / (uint32_t)p.H) >> 7;
  const int n = o + 1, K = KC ? KC : p.K;
  int32_t* out = idx + (int64_t)r * K;
  if (n <= K) {  // every visible page is kept
    for (int s = lane; s < K; s += 32) out[s] = s < n ? s : -1;
    return;
  }
  const float* row = scores + (int64_t)r * pitch;
  const int base = lane * E;
  uint32_t key[E], pg[E];
#pragma unroll
  for (int j = 0; j < E; ++j) {
    const int page = base + j;
    pg[j] = (uint32_t)j;
    key[j] = (page < n && page != o) ? score_key(__ldg(row + page)) : 0u;
  }
  sort_best_first<E>(key, pg);
  int c = rounds_distinct_heads<E, KC>(key, K);
  if (__reduce_add_sync(0xffffffffu, (uint32_t)c) != (uint32_t)(K - 1))
    c = rounds_lowest_lane<E, KC>(key, K, lane);
  uint32_t taken = 0;  // bit j: page base + j selected
#pragma unroll
  for (int j = 0; j < E; ++j)
    if (j < c) taken |= 1u << pg[j];
  if (o / E == lane) taken |= 1u << (o % E);
  // ascending output: pages before this lane's are those of lower lanes
  int before = __popc(taken);
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, before, d);
    if (lane >= d) before += y;
  }
  before -= __popc(taken);
#pragma unroll
  for (int j = 0; j < E; ++j)
    if ((taken >> j) & 1u) out[before++] = base + j;
}

// Long rows: a filter first.  Lane l holds the pages l, l + 32, l + 64, ... (E of them), so
// every lane has work and each load instruction reads 128 contiguous bytes.  The (k-1)-th
// largest of the 32 lane maxima, t0 (read off a bitonic sort of the maxima across the warp), is
// at most the row's (k-1)-th largest key (those k-1 maxima are k-1 distinct keys >= t0), so
// every page of the answer has key >= t0.  The keys >= t0 are compacted in page order (one
// ballot per stride of 32 pages) into two per lane (shared memory, at most 64 of them) and the
// rounds above run on those; the row's own page, its last visible page, goes last.  A row with
// more than 64 such keys (heavy ties) reloads its keys with EH adjacent pages per lane and runs
// the rounds on all of them.
template <int E, int EH>  // E * 32 >= max_pages, EH * 32 >= max_pages (EH a power of two)
__global__ void __launch_bounds__(256)
topk_filter_kernel(DevPlan p, const float* __restrict__ scores, int64_t pitch,
                   int32_t* __restrict__ idx) {
  __shared__ uint2 cand[8][64];  // per warp: (key, page) of the compacted candidates
  pdl_wait();  // the scores come from the indexer just before
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t r = blockIdx.x * 8u + warp;  // rows x top_k < 2^31
  if (r >= (uint32_t)p.T * (uint32_t)p.H) return;
  const int o = __ldg(p.tok_pos + r / (uint32_t)p.H) >> 7;
  const int n = o + 1, K = p.K;
  int32_t* out = idx + (int64_t)r * K;
  if (n <= K) {  // every visible page is kept
    for (int s = lane; s < K; s += 32) out[s] = s < n ? s : -1;
    return;
  }
  const float* row = scores + (int64_t)r * pitch;
  uint32_t key[E];
  uint32_t lm = 0;  // the lane's largest key
#pragma unroll
  for (int j = 0; j < E; ++j) {
    const int page = j * 32 + lane;
    key[j] = (page < n && page != o) ? score_key(__ldg(row + page)) : 0u;
    lm = max(lm, key[j]);
  }
  // t0: the (K-1)-th largest lane maximum (0 when fewer lanes hold candidates), from a
  // bitonic sort of the 32 lane maxima into descending lane order
  uint32_t v = lm;
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1)
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const uint32_t w = __shfl_xor_sync(0xffffffffu, v, stride);
      // descending runs where bit `size` of the lane is 0; the lower lane of a pair keeps
      // the larger key in a descending run
      const bool keep_max = ((lane & stride) == 0) == ((lane & size) == 0);
      v = keep_max ? max(v, w) : min(v, w);
    }
  const uint32_t t0 = K - 2 < 32 ? __shfl_sync(0xffffffffu, v, K - 2) : 0u;
  // compaction in page order: stride j holds the pages 32 j .. 32 j + 31, lane order
  const uint32_t lt = (1u << lane) - 1u;
  int total = 0;  // warp-uniform
#pragma unroll
  for (int j = 0; j < E; ++j) {
    const bool keep = key[j] != 0u && key[j] >= t0;
    const uint32_t b = __ballot_sync(0xffffffffu, keep);
    const int at = total + __popc(b & lt);
    if (keep && at < 64) cand[warp][at] = make_uint2(key[j], (uint32_t)(j * 32 + lane));
    total += __popc(b);
  }
  if (total <= 64) {
    __syncwarp();
    uint32_t ck[2], cp[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int i = 2 * lane + j;
      ck[j] = i < total ? cand[warp][i].x : 0u;
      cp[j] = (uint32_t)j;
    }
    const uint32_t page0 = 2 * lane < total ? cand[warp][2 * lane].y : 0u;
    const uint32_t page1 = 2 * lane + 1 < total ? cand[warp][2 * lane + 1].y : 0u;
    sort_best_first<2>(ck, cp);
    int c = rounds_distinct_heads<2, 0>(ck, K);
    if (__reduce_add_sync(0xffffffffu, (uint32_t)c) != (uint32_t)(K - 1))
      c = rounds_lowest_lane<2, 0>(ck, K, lane);
    uint32_t taken = 0;  // bit j: compacted candidate 2 lane + j selected
#pragma unroll
    for (int j = 0; j < 2; ++j)
      if (j < c) taken |= 1u << cp[j];
    int before = __popc(taken);
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, before, d);
      if (lane >= d) before += y;
    }
    before -= __popc(taken);
    if (taken & 1u) out[before++] = (int32_t)page0;
    if (taken & 2u) out[before++] = (int32_t)page1;
    if (lane == 0) out[K - 1] = o;  // the own page is the row's last visible page
    return;
  }
  // heavy ties: the rounds on every key of the row, EH adjacent pages per lane
  const int base = lane * EH;
  uint32_t hk[EH], pg[EH];
#pragma unroll
  for (int j = 0; j < EH; ++j) {
    const int page = base + j;
    hk[j] = (page < n && page != o) ? score_key(__ldg(row + page)) : 0u;
    pg[j] = (uint32_t)j;
  }
  sort_best_first<EH>(hk, pg);
  const int c = rounds_lowest_lane<EH, 0>(hk, K, lane);
  uint32_t taken = 0;
#pragma unroll
  for (int j = 0; j < EH; ++j)
    if (j < c) taken |= 1u << pg[j];
  if (o / EH == lane) taken |= 1u << (o % EH);
  int before = __popc(taken);
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, before, d);
    if (lane >= d) before += y;
  }
  before -= __popc(taken);
#pragma unroll
  for (int j = 0; j < EH; ++j)
    if ((taken >> j) & 1u) out[before++] = base + j;
}

}  // namespace

cudaError_t launch_topk(const DevPlan& p, const float* scores, int64_t pitch, int32_t* idx,
                        cudaStream_t st) {
  const int64_t R = (int64_t)p.T * p.H;
  const unsigned grid = (unsigned)((R + 7) / 8);
  if (grid == 0) return cudaSuccess;
  // top_k = 16 (the common case) runs instances whose rounds unroll completely (the filtered
  // long rows do better with the rolled loop)
  const bool k16 = p.K == 16;
  cudaError_t e;
  if (p.max_pages <= 32) {
    if (k16) e = launch_pdl(topk_kernel<1, 16>, dim3(grid), dim3(256), 0, st, p, scores, pitch, idx);
    else e = launch_pdl(topk_kernel<1>, dim3(grid), dim3(256), 0, st, p, scores, pitch, idx);
  } else if (p.max_pages <= 64) {
    if (k16) e = launch_pdl(topk_kernel<2, 16>, dim3(grid), dim3(256), 0, st, p, scores, pitch, idx);
    else e = launch_pdl(topk_kernel<2>, dim3(grid), dim3(256), 0, st, p, scores, pitch, idx);
  } else if (p.max_pages <= 128) {
    if (k16) e = launch_pdl(topk_kernel<4, 16>, dim3(grid), dim3(256), 0, st, p, scores, pitch, idx);
    else e = launch_pdl(topk_kernel<4>, dim3(grid), dim3(256), 0, st, p, scores, pitch, idx);
  } else if (p.max_pages <= 256) {
    e = launch_pdl(topk_filter_kernel<8, 8>, dim3(grid), dim3(256), 0, st, p, scores, pitch, idx);
  } else if (p.max_pages <= 320) {
    e = launch_pdl(topk_filter_kernel<10, 16>, dim3(grid), dim3(256), 0, st, p, scores, pitch, idx);
  } else if (p.max_pages <= 384) {
    e = launch_pdl(topk_filter_kernel<12, 16>, dim3(grid), dim3(256), 0, st, p, scores, pitch, idx);
  } else if (p.max_pages <= 512) {
    e = launch_pdl(topk_filter_kernel<16, 16>, dim3(grid), dim3(256), 0, st, p, scores, pitch, idx);
  } else if (p.max_pages <= 768) {
    e = launch_pdl(topk_filter_kernel<24, 32>, dim3(grid), dim3(256), 0, st, p, scores, pitch, idx);
  } else {
    static_assert(kMaxPagesPerReq <= 32 * 32, "the widest lane layouts hold 32 x 32 pages");
    e = launch_pdl(topk_filter_kernel<32, 32>, dim3(grid), dim3(256), 0, st, p, scores, pitch, idx);
  }
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace sps
