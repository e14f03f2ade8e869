// topk.cu -- per-row top-k page selection, one warp per row.
//
// Contract (north-star definition of the method; "MSA PR 36: Q8KV8 prefill indexer" relies on
// a bitwise-stable selection): the row's own page o is always kept; the other
// n_sel - 1 = min(k, o+1) - 1 pages are the best by (score descending, page ascending), with
// -0.0 equal to +0.0; output in ascending page order, padded with -1.
//
// Each lane holds pages lane, lane+32, ... as 32-bit order-preserving keys of their scores.
// A selection round is two warp reductions (redux.sync): the maximum key, then the lowest
// page among the lanes that hold it; the winner is marked taken.  n_sel - 1 rounds, then a
// ballot/popc prefix writes the chosen pages in ascending order.
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

template <int E>  // pages per lane: max_pages <= 32 * E
__global__ void __launch_bounds__(256)
topk_kernel(DevPlan p, const float* __restrict__ scores, int64_t pitch, int32_t* __restrict__ idx) {
  const int lane = threadIdx.x & 31;
  const int64_t r = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int64_t R = (int64_t)p.T * p.H;
  if (r >= R) return;
  const int tok = (int)(r / p.H);
  const int t = __ldg(p.tok_pos + tok);
  const int o = t >> 7;
  const int n = o + 1;
  const int K = p.K;
  int32_t* out = idx + r * K;
  if (n <= K) {  // every visible page is kept
    for (int s = lane; s < K; s += 32) out[s] = s < n ? s : -1;
    return;
  }
  const float* row = scores + r * pitch;
  uint32_t key[E];
#pragma unroll
  for (int j = 0; j < E; ++j) {
    int pg = lane + 32 * j;
    key[j] = (pg < n && pg != o) ? score_key(__ldg(row + pg)) : 0u;
  }
  uint32_t taken = 0;  // bit j: page lane + 32 j selected
  for (int round = 1; round < K; ++round) {
    // best remaining key of this lane; equal keys keep the lower page (lower j)
    uint32_t bk = 0;
    int bj = 0;
#pragma unroll
    for (int j = 0; j < E; ++j)
      if (key[j] > bk) { bk = key[j]; bj = j; }
    const uint32_t wmax = __reduce_max_sync(0xffffffffu, bk);
    const uint32_t cand = (bk == wmax) ? (uint32_t)(lane + 32 * bj) : 0xffffffffu;
    const uint32_t win = __reduce_min_sync(0xffffffffu, cand);
    if ((int)(win & 31) == lane) {
      const int wj = (int)(win >> 5);
#pragma unroll
      for (int j = 0; j < E; ++j)
        if (j == wj) { taken |= 1u << j; key[j] = 0u; }
    }
  }
  if ((o & 31) == lane) taken |= 1u << (o >> 5);
  // ascending output through ballot prefix counts
  int before = 0;
  const uint32_t lt = (1u << lane) - 1u;
#pragma unroll
  for (int j = 0; j < E; ++j) {
    const uint32_t bal = __ballot_sync(0xffffffffu, (taken >> j) & 1u);
    if ((taken >> j) & 1u) out[before + __popc(bal & lt)] = lane + 32 * j;
    before += __popc(bal);
  }
  // before == K here (n > K): no padding needed
}

}  // namespace

cudaError_t launch_topk(const DevPlan& p, const float* scores, int64_t pitch, int32_t* idx,
                        cudaStream_t st) {
  const int64_t R = (int64_t)p.T * p.H;
  const unsigned grid = (unsigned)((R + 7) / 8);
  if (grid == 0) return cudaSuccess;
  if (p.max_pages <= 32) topk_kernel<1><<<grid, 256, 0, st>>>(p, scores, pitch, idx);
  else if (p.max_pages <= 64) topk_kernel<2><<<grid, 256, 0, st>>>(p, scores, pitch, idx);
  else if (p.max_pages <= 128) topk_kernel<4><<<grid, 256, 0, st>>>(p, scores, pitch, idx);
  else if (p.max_pages <= 256) topk_kernel<8><<<grid, 256, 0, st>>>(p, scores, pitch, idx);
  else topk_kernel<16><<<grid, 256, 0, st>>>(p, scores, pitch, idx);
  return cudaGetLastError();
}

}  // namespace sps
