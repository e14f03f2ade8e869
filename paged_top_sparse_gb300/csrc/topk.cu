// topk.cu -- per-row top-k page selection.
//
// Contract (the method's page selection: every row attends its own page, the one page the
// forward of "MSA PR 21: Q8KV4 paged sparse prefill", K1 Softmax, masks causally; "MSA PR 36:
// Q8KV8 prefill indexer", Kernel performance, relies on a bitwise-stable selection): the row's
// own page o is always kept; the other
// n_sel - 1 = min(k, o+1) - 1 pages are the best by (score descending, page ascending), with
// -0.0 equal to +0.0; output in ascending page order, padded with -1.
//
// top_k <= 16: one thread per row.  The thread streams its row in groups of 16 pages and keeps
// the 16 largest scores seen so far as a descending list: a group is sorted by Batcher's
// odd-even merge network (63 comparators), the list takes the larger of list[i] and
// group[15 - i] (a bitonic sequence that holds the 16 largest of both) and a bitonic merge
// sorts it again.  The (k-1)-th largest score t then decides: every candidate above t is taken,
// and of those equal to t the lowest pages fill the rest (the list's k-th entry shows whether
// t is shared; the entries above t give how many equal ones are needed).  A second pass over
// the row writes the chosen pages in ascending order into shared memory, and each warp stores
// its 32 rows' outputs, which are contiguous, with coalesced stores.  The list never carries
// page numbers, so the network is plain FP32 min/max on the scores themselves: -0.0 and +0.0
// compare equal, as the contract wants, and pages outside the candidates enter as -inf (a
// finite input never scores -inf; NaN scores are outside the contract).  With 16-byte rows
// the scores reach shared memory by TMA tile loads, one warp's 32 rows x 16 pages per tile
// (topk_tma_kernel); other layouts are read by per-thread loads (topk_thread_kernel).  Long
// rows of a small batch, which would leave few warps each walking hundreds of groups, run
// pass 1 in segments of a row (topk_seg_kernel: each segment's 16 largest scores, merged per
// row by the bitonic merge, and each group's largest score), and pass 2 reads again only the
// groups whose largest score reaches the row's threshold (topk_emit_rows_kernel).
//
// Larger top_k (the warp kernels below): one warp per row.
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

__device__ __forceinline__ void cmpx_desc(float& a, float& b) {  // a <- max, b <- min
  const float hi = fmaxf(a, b);
  b = fminf(a, b);
  a = hi;
}

// The least float above t (t finite; either zero gives the least positive subnormal).
__device__ __forceinline__ float next_up(float t) {
  const uint32_t u = __float_as_uint(t);
  if ((u & 0x7fffffffu) == 0u) return __uint_as_float(1u);
  return __uint_as_float(t > 0.f ? u + 1u : u - 1u);
}

// Sorts 16 scores in descending order: Batcher's odd-even merge sort (K. E. Batcher, "Sorting
// networks and their applications", AFIPS 1968), 63 comparators in its ten layers, written
// out so that every index is a constant.
__device__ __forceinline__ void sort16_desc(float (&x)[16]) {
#define C(a, b) cmpx_desc(x[a], x[b])
  C(0, 1); C(2, 3); C(4, 5); C(6, 7); C(8, 9); C(10, 11); C(12, 13); C(14, 15);
  C(0, 2); C(1, 3); C(4, 6); C(5, 7); C(8, 10); C(9, 11); C(12, 14); C(13, 15);
  C(1, 2); C(5, 6); C(9, 10); C(13, 14);
  C(0, 4); C(1, 5); C(2, 6); C(3, 7); C(8, 12); C(9, 13); C(10, 14); C(11, 15);
  C(2, 4); C(3, 5); C(10, 12); C(11, 13);
  C(1, 2); C(3, 4); C(5, 6); C(9, 10); C(11, 12); C(13, 14);
  C(0, 8); C(1, 9); C(2, 10); C(3, 11); C(4, 12); C(5, 13); C(6, 14); C(7, 15);
  C(4, 8); C(5, 9); C(6, 10); C(7, 11);
  C(2, 4); C(3, 5); C(6, 8); C(7, 9); C(10, 12); C(11, 13);
  C(1, 2); C(3, 4); C(5, 6); C(7, 8); C(9, 10); C(11, 12); C(13, 14);
#undef C
}

// best <- the 16 largest of best and g (both descending), descending.
__device__ __forceinline__ void merge16_desc(float (&best)[16], const float (&g)[16]) {
#pragma unroll
  for (int i = 0; i < 16; ++i) best[i] = fmaxf(best[i], g[15 - i]);
#pragma unroll
  for (int s = 8; s >= 1; s >>= 1)
#pragma unroll
    for (int i = 0; i < 16; ++i)
      if ((i & s) == 0) cmpx_desc(best[i], best[i + s]);
}

// Scores of pages c .. c+3 (c < o); entries of pages at or past o are unspecified.  VEC: the
// row is 16-byte aligned and its pitch a multiple of 4, so the four floats lie inside the row.
template <bool VEC>
__device__ __forceinline__ float4 load4_raw(const float* row, int c, int o) {
  if (VEC) return __ldg(reinterpret_cast<const float4*>(row + c));
  float4 f;
  f.x = __ldg(row + c);
  f.y = c + 1 < o ? __ldg(row + c + 1) : 0.f;
  f.z = c + 2 < o ? __ldg(row + c + 2) : 0.f;
  f.w = c + 3 < o ? __ldg(row + c + 3) : 0.f;
  return f;
}

// The 16 scores of pages base .. base+15 (base < o) as four float4; entries of pages at or past
// o are unspecified.  All loads are issued before any is used.
template <bool VEC>
__device__ __forceinline__ void load_group(const float* row, int base, int o, float4 (&f)[4]) {
#pragma unroll
  for (int q = 0; q < 4; ++q)
    f[q] = base + 4 * q < o ? load4_raw<VEC>(row, base + 4 * q, o) : make_float4(0.f, 0.f, 0.f, 0.f);
}

// Pass 1 of a row: the scores of pages base .. base+15 that lie below o join the running list
// of the 16 largest.  Returns the largest of them.
__device__ __forceinline__ float take_group(float (&best)[16], const float4 (&f)[4], int base,
                                            int o) {
  float g[16];
  if (base + 16 <= o) {  // a full group: every page is a candidate
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      g[4 * q + 0] = f[q].x;
      g[4 * q + 1] = f[q].y;
      g[4 * q + 2] = f[q].z;
      g[4 * q + 3] = f[q].w;
    }
  } else {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int c = base + 4 * q;
      g[4 * q + 0] = c + 0 < o ? f[q].x : -INFINITY;
      g[4 * q + 1] = c + 1 < o ? f[q].y : -INFINITY;
      g[4 * q + 2] = c + 2 < o ? f[q].z : -INFINITY;
      g[4 * q + 3] = c + 3 < o ? f[q].w : -INFINITY;
    }
  }
  sort16_desc(g);
  merge16_desc(best, g);
  return g[0];
}

// The selection rule read off the list (o >= K >= 2 candidates, so the (K-1)-th and K-th
// largest scores both exist), t being the (K-1)-th largest.  When the K-th differs from t, the
// chosen candidates are exactly those with score >= t.  When it equals t (shared), every
// candidate above t is taken and `need` of those equal to it, the lowest pages first.
struct TopkRule {
  float ge;  // while need == 0 the pages with score >= ge are taken
  float eq;  // t: with need > 0, the pages above it and `need` more equal to it are taken
  int need;
};

__device__ __forceinline__ TopkRule selection_rule(const float (&best)[16], int K) {
  // the list is descending: t = best[K-2] is the least of the first K-1 entries, t_next =
  // best[K-1] the largest of the rest (reductions, so that no entry is picked by a run-time index)
  float t = INFINITY, t_next = -INFINITY;
  int above = 0;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    t = i < K - 1 ? fminf(t, best[i]) : t;
    t_next = i >= K - 1 ? fmaxf(t_next, best[i]) : t_next;
  }
#pragma unroll
  for (int i = 0; i < 16; ++i) above += best[i] > t ? 1 : 0;
  TopkRule rule;
  const bool shared = t_next == t;
  rule.eq = t;
  // shared: once the equal pages are in, the threshold is the least score above t's
  rule.ge = shared ? next_up(t) : t;
  rule.need = shared ? K - 1 - above : 0;
  return rule;
}

// Pass 2 of a row: the chosen pages among base .. base+15 (those below o), in ascending order,
// into the row's staging so[pos ...].  While no equal page is still needed the group becomes a
// 16-bit mask of the taken pages, walked lowest bit first; otherwise page by page.  pos is
// masked by 15: the staging row stays in bounds whatever the scores.
__device__ __forceinline__ void emit_group(const float4 (&f)[4], int base, int o, TopkRule& rule,
                                           int32_t* so, int& pos) {
  float v[16];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    v[4 * q + 0] = f[q].x;
    v[4 * q + 1] = f[q].y;
    v[4 * q + 2] = f[q].z;
    v[4 * q + 3] = f[q].w;
  }
  const int nb = o - base < 16 ? o - base : 16;  // candidate pages in the group
  if (rule.need == 0) {
    uint32_t bits = 0u;
#pragma unroll
    for (int e = 0; e < 16; ++e) bits |= v[e] >= rule.ge ? 1u << e : 0u;
    if (nb < 16) bits &= (1u << nb) - 1u;
    while (bits) {
      so[pos++ & 15] = base + __ffs(bits) - 1;
      bits &= bits - 1u;
    }
  } else {
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      if (e >= nb) break;
      const bool eq = v[e] == rule.eq && rule.need > 0;
      if (v[e] > rule.eq || eq) so[pos++ & 15] = base + e;
      rule.need -= eq ? 1 : 0;
    }
  }
}

// The rows that keep every visible page (o < K), and K = 1 (the own page alone).
__device__ __forceinline__ void stage_short_row(int32_t* so, int o, int K) {
  if (K == 1) {
    so[0] = o;
  } else {
    for (int s = 0; s < K; ++s) so[s] = s <= o ? s : -1;
  }
}

// A warp's 32 rows are consecutive, so their outputs are one contiguous run of nrow * K ints;
// the warp stores it from the staging rows (pitch OP) with coalesced stores.
template <int OP>
__device__ __forceinline__ void store_staged(const int32_t* s_warp, int32_t* dst, int nrow, int K,
                                             int lane) {
  const int dr = 32 / K, dc = 32 % K;
  int row = lane / K, col = lane % K;
  for (int w = lane; w < nrow * K; w += 32) {
    dst[w] = s_warp[row * OP + col];
    row += dr;
    col += dc;
    if (col >= K) {
      col -= K;
      ++row;
    }
  }
}

constexpr int kTopkOP = 17;  // staging row pitch (ints): conflict-free per-thread writes

// top_k <= 16, any row pitch: every thread loads its own row (VEC: 16-byte loads).
template <bool VEC>
__global__ void __launch_bounds__(256)
topk_thread_kernel(DevPlan p, const float* __restrict__ scores, int64_t pitch,
                   int32_t* __restrict__ idx) {
  __shared__ int32_t s_out[256 * kTopkOP];
  pdl_wait();  // the scores come from the indexer just before
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t R = (int64_t)p.T * p.H;
  const int64_t r0 = (int64_t)blockIdx.x * 256 + warp * 32;  // the warp's first row
  if (r0 >= R) return;                                       // warp-uniform
  const int64_t r = r0 + lane;
  const int K = p.K;
  int32_t* so = s_out + threadIdx.x * kTopkOP;
  if (r < R) {
    // own page o; the pages 0 .. o-1 are the candidates
    const int o = __ldg(p.tok_pos + (uint32_t)r / (uint32_t)p.H) >> 7;
    if (o < K || K == 1) {
      stage_short_row(so, o, K);
    } else {
      const float* row = scores + r * pitch;
      float best[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) best[i] = -INFINITY;
      float4 f[4];
      load_group<VEC>(row, 0, o, f);
      for (int base = 0; base < o; base += 16) {
        float4 cur[4] = {f[0], f[1], f[2], f[3]};
        if (base + 16 < o) load_group<VEC>(row, base + 16, o, f);  // in flight meanwhile
        take_group(best, cur, base, o);
      }
      TopkRule rule = selection_rule(best, K);
      int pos = 0;
      load_group<VEC>(row, 0, o, f);
      for (int base = 0; base < o; base += 16) {
        float4 cur[4] = {f[0], f[1], f[2], f[3]};
        if (base + 16 < o) load_group<VEC>(row, base + 16, o, f);
        emit_group(cur, base, o, rule, so, pos);
      }
      so[K - 1] = o;  // the own page is the row's last visible page
    }
  }
  __syncwarp();
  const int nrow = R - r0 < 32 ? (int)(R - r0) : 32;
  store_staged<kTopkOP>(s_out + warp * 32 * kTopkOP, idx + r0 * K, nrow, K, lane);
}

// top_k <= 16, row pitch a multiple of 4 floats, at least 16 pages and 32 rows: the same
// per-row work, with each warp's 32 rows x 16 scores brought into shared memory by one TMA
// tile load (64-byte swizzle: the 16-byte chunk c of tile row t sits at chunk c ^ ((t >> 1) & 3),
// so the 32 threads' reads of their own rows hit distinct banks).  Each warp runs its own ring
// of S tiles: its pass 1 over groups 0 .. G-1 and its pass 2 over them again are one sequence
// of 2G tile loads, issued S ahead by lane 0.  G is the largest group count of the warp's
// rows.  Waits are bounded; a warp that gives up raises DEV_TIMEOUT and leaves its rows
// unwritten.
constexpr int kTopkTile = 32 * 16 * 4;  // bytes of one tile
template <int S>
constexpr size_t topk_smem() {
  return 1024 + 8 * S * kTopkTile + 8 * S * 8 + 256 * kTopkOP * 4;
}

// Lane 0 of a warp: the tile load of item n of its sequence, 16-page group `group`, into
// stage n % S.
template <int S>
__device__ __forceinline__ void topk_issue_group(const CUtensorMap* tm, uint32_t tiles,
                                                 uint32_t bars, int n, int group, int r0) {
  const int s = n % S;
  mbar_expect_tx(bars + 8 * s, kTopkTile);
  tma_load_2d(tiles + s * kTopkTile, tm, 16 * group, r0, bars + 8 * s);
}

// The same for a sequence of pass 1 over groups 0 .. G-1, then pass 2 over them again.
template <int S>
__device__ __forceinline__ void topk_issue_tile(const CUtensorMap* tm, uint32_t tiles,
                                                uint32_t bars, int n, int G, int r0) {
  topk_issue_group<S>(tm, tiles, bars, n, n < G ? n : n - G, r0);
}

// Every lane waits for item n's tile (stage n % S); true on all lanes when it landed.
template <int S>
__device__ __forceinline__ bool topk_tile_ready(uint32_t bar, int n, int32_t* status) {
  const bool got = mbar_wait(bar, (uint32_t)(n / S) & 1u, nullptr, status);
  return __all_sync(0xffffffffu, got);
}

// This lane's row (tile row `lane`) of a landed tile: chunk c at 16 (c ^ ((lane >> 1) & 3)).
__device__ __forceinline__ void topk_read_tile(const uint8_t* tile, int lane, float4 (&f)[4]) {
  const uint8_t* row = tile + lane * 64;
  const int sw = (lane >> 1) & 3;
#pragma unroll
  for (int c = 0; c < 4; ++c) f[c] = *reinterpret_cast<const float4*>(row + 16 * (c ^ sw));
}

// A segment's stored list: 16 floats, descending.
__device__ __forceinline__ void load_list(const float* src, float (&g)[16]) {
  const float4* s4 = reinterpret_cast<const float4*>(src);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float4 v = __ldg(s4 + q);
    g[4 * q] = v.x;
    g[4 * q + 1] = v.y;
    g[4 * q + 2] = v.z;
    g[4 * q + 3] = v.w;
  }
}

// Pass 1 of long rows split into segments (DevPlan::topk_nseg): warp w of block (x, y) runs
// pass 1 of its 32 rows over the 16-page groups [y * segg, (y + 1) * segg), through the same
// per-warp tile ring, stores each full row's 16 largest scores of the segment (descending) to
// topk_lists[row][y] (a segment past a row's last candidate stores nothing) and the largest
// candidate score of each of its groups to topk_gmax[group][row].
template <int S>
__global__ void __launch_bounds__(256)
topk_seg_kernel(const __grid_constant__ CUtensorMap tmS, DevPlan p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* tiles = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(tiles + 8 * S * kTopkTile);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t my_tiles = smem_u32(tiles + warp * S * kTopkTile);
  const uint32_t my_bars = smem_u32(bars + warp * S);
  if (lane == 0) {
    tma_prefetch_desc(&tmS);
    for (int s = 0; s < S; ++s) mbar_init(my_bars + 8 * s, 1);
    fence_mbar_init();
  }
  __syncwarp();
  pdl_wait();  // the scores come from the indexer just before
  const int64_t R = (int64_t)p.T * p.H;
  const int64_t r0 = (int64_t)blockIdx.x * 256 + warp * 32;
  if (r0 >= R) return;  // warp-uniform; this warp issued no copy
  const int64_t r = r0 + lane;
  const int K = p.K;
  int o = 0;
  bool full = false;
  if (r < R) {
    o = __ldg(p.tok_pos + (uint32_t)r / (uint32_t)p.H) >> 7;
    full = o >= K && K > 1;
  }
  const int Gw = (int)__reduce_max_sync(0xffffffffu, full ? (uint32_t)(o + 15) / 16u : 0u);
  const int g0 = (int)blockIdx.y * p.topk_segg;
  const int g1 = min(Gw, g0 + p.topk_segg);
  const int items = g1 > g0 ? g1 - g0 : 0;
  if (lane == 0)  // item n of this warp's sequence is group g0 + n
    for (int n = 0; n < S && n < items; ++n)
      topk_issue_group<S>(&tmS, my_tiles, my_bars, n, g0 + n, (int)r0);
  float best[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) best[i] = -INFINITY;
  bool ok = true;
  for (int n = 0; n < items; ++n) {
    const int s = n % S;
    if (!topk_tile_ready<S>(my_bars + 8 * s, n, p.status)) {
      ok = false;
      break;
    }
    const int base = 16 * (g0 + n);
    if (full && base < o) {
      float4 f[4];
      topk_read_tile(tiles + (warp * S + s) * kTopkTile, lane, f);
      p.topk_gmax[(int64_t)(g0 + n) * R + r] = take_group(best, f, base, o);
    }
    __syncwarp();
    if (lane == 0 && n + S < items)
      topk_issue_group<S>(&tmS, my_tiles, my_bars, n + S, g0 + n + S, (int)r0);
  }
  if (!ok) {  // let the copies already issued land before the block's shared memory is reused
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < kSettleNs) __nanosleep(1000);
    return;
  }
  if (full && 16 * g0 < o) {
    float4* dst = reinterpret_cast<float4*>(p.topk_lists + (r * p.topk_nseg + blockIdx.y) * 16);
#pragma unroll
    for (int q = 0; q < 4; ++q)
      dst[q] = make_float4(best[4 * q], best[4 * q + 1], best[4 * q + 2], best[4 * q + 3]);
  }
}

// Pass 2 of long rows after topk_tma_kernel<S, true> (rows of 16-byte pitch), eight threads
// per row, each over one eighth of the row's 16-page groups in page order: of its groups only
// those whose largest candidate reaches the threshold (topk_gmax: a taken page, or a page
// equal to the threshold, lies in no other) are read.  A first walk counts the pages each
// thread takes (those above the threshold, and of those equal to it as many as the row still
// needs, lowest pages first); a prefix over the eight gives each its start in the row's
// output, and a second walk writes them.
constexpr int kEmitSub = 8;  // threads per row

// Groups g0 .. g1-1 of a row whose largest candidate reaches thr, in order: f(g).
template <typename F>
__device__ __forceinline__ void for_hit_groups(const DevPlan& p, int64_t R, int64_t r, int g0,
                                               int g1, float thr, F&& f) {
  for (int b = g0; b < g1; b += 8) {  // eight group maxima in flight, then the hits in order
    float gm[8];
#pragma unroll
    for (int u = 0; u < 8; ++u)
      gm[u] = b + u < g1 ? __ldcg(p.topk_gmax + (int64_t)(b + u) * R + r) : -INFINITY;
    uint32_t hit = 0u;
#pragma unroll
    for (int u = 0; u < 8; ++u) hit |= gm[u] >= thr ? 1u << u : 0u;
    while (hit) {
      f(b + __ffs(hit) - 1);
      hit &= hit - 1u;
    }
  }
}

__global__ void __launch_bounds__(256)
topk_emit_rows_kernel(DevPlan p, const float* __restrict__ scores, int64_t pitch,
                      int32_t* __restrict__ idx) {
  pdl_wait();  // the rows' rules from the kernel before
  const int64_t R = (int64_t)p.T * p.H;
  const int64_t r = (int64_t)blockIdx.x * (256 / kEmitSub) + threadIdx.x / kEmitSub;
  const int sub = threadIdx.x % kEmitSub;
  const int K = p.K;
  bool full = false;
  int o = 0;
  if (r < R) {
    o = __ldg(p.tok_pos + (uint32_t)r / (uint32_t)p.H) >> 7;
    full = o >= K && K > 1;  // other rows were written whole by the kernel before
  }
  int need = 0;
  float ge = 0.f, eq = 0.f;
  if (full) {
    const int32_t* meta = p.topk_meta + r * 3;
    need = meta[0];
    ge = __int_as_float(meta[1]);
    eq = __int_as_float(meta[2]);
  }
  const float thr = need > 0 ? eq : ge;
  const float* row = scores + r * pitch;
  const int G = (o + 15) / 16, per = (G + kEmitSub - 1) / kEmitSub;
  const int g0 = min(G, sub * per), g1 = min(G, g0 + per);
  // walk 1: the pages above the threshold (need 0: at or above it) and those equal to it
  int above = 0, equal = 0;
  if (full)
    for_hit_groups(p, R, r, g0, g1, thr, [&](int g) {
      float4 f[4];
      load_group<true>(row, 16 * g, o, f);
      const float v[16] = {f[0].x, f[0].y, f[0].z, f[0].w, f[1].x, f[1].y, f[1].z, f[1].w,
                           f[2].x, f[2].y, f[2].z, f[2].w, f[3].x, f[3].y, f[3].z, f[3].w};
      const int nb = o - 16 * g < 16 ? o - 16 * g : 16;
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        if (e < nb) {
          above += (need > 0 ? v[e] > eq : v[e] >= ge) ? 1 : 0;
          equal += need > 0 && v[e] == eq ? 1 : 0;
        }
      }
    });
  // the equal pages of lower threads come first; then this thread's start in the output
  int eq_before = equal;
#pragma unroll
  for (int d = 1; d < kEmitSub; d <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, eq_before, d, kEmitSub);
    if (sub >= d) eq_before += y;
  }
  eq_before -= equal;
  int my_eq = need - eq_before;
  my_eq = my_eq < 0 ? 0 : (my_eq > equal ? equal : my_eq);
  int start = above + my_eq;
#pragma unroll
  for (int d = 1; d < kEmitSub; d <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, start, d, kEmitSub);
    if (sub >= d) start += y;
  }
  start -= above + my_eq;
  // walk 2: write them
  int32_t* out = idx + r * K;
  if (full) {
    int pos = start;
    for_hit_groups(p, R, r, g0, g1, thr, [&](int g) {
      float4 f[4];
      load_group<true>(row, 16 * g, o, f);
      const float v[16] = {f[0].x, f[0].y, f[0].z, f[0].w, f[1].x, f[1].y, f[1].z, f[1].w,
                           f[2].x, f[2].y, f[2].z, f[2].w, f[3].x, f[3].y, f[3].z, f[3].w};
      const int nb = o - 16 * g < 16 ? o - 16 * g : 16;
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        if (e < nb) {
          bool take = need > 0 ? v[e] > eq : v[e] >= ge;
          if (need > 0 && v[e] == eq && my_eq > 0) {
            take = true;
            --my_eq;
          }
          if (take) {
            if (pos < K - 1) out[pos] = 16 * g + e;  // in bounds whatever the scores
            ++pos;
          }
        }
      }
    });
    if (sub == 0) out[K - 1] = o;
  }
}

// SEG: pass 1 comes from topk_seg_kernel's per-segment lists, merged here into each row's rule
// for topk_emit_rows_kernel; this kernel then writes the short rows (and the own page) only.
template <int S, bool SEG>
__global__ void __launch_bounds__(256)
topk_tma_kernel(const __grid_constant__ CUtensorMap tmS, DevPlan p, int32_t* __restrict__ idx) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* tiles = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(tiles + 8 * S * kTopkTile);
  int32_t* s_out = reinterpret_cast<int32_t*>(bars + 8 * S);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t my_tiles = smem_u32(tiles + warp * S * kTopkTile);
  const uint32_t my_bars = smem_u32(bars + warp * S);
  if (lane == 0) {
    tma_prefetch_desc(&tmS);
    for (int s = 0; s < S; ++s) mbar_init(my_bars + 8 * s, 1);
    fence_mbar_init();
  }
  __syncwarp();
  pdl_wait();  // the scores come from the indexer just before
  const int64_t R = (int64_t)p.T * p.H;
  const int64_t r0 = (int64_t)blockIdx.x * 256 + warp * 32;
  if (r0 >= R) return;  // warp-uniform; this warp issued no copy
  const int64_t r = r0 + lane;
  const int K = p.K;
  int32_t* so = s_out + threadIdx.x * kTopkOP;
  int o = 0;
  bool full = false;  // the row runs both passes
  if (r < R) {
    o = __ldg(p.tok_pos + (uint32_t)r / (uint32_t)p.H) >> 7;
    full = o >= K && K > 1;
    if (!full) stage_short_row(so, o, K);
  }
  const int G = (int)__reduce_max_sync(0xffffffffu, full ? (uint32_t)(o + 15) / 16u : 0u);
  float best[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) best[i] = -INFINITY;
  TopkRule rule{};
  bool ok = true;
  int pos = 0;
  if (SEG && full) {
    // pass 1 from the segments' lists (descending), merged; the rule for topk_emit_rows_kernel,
    // which runs pass 2
    const int nseg = p.topk_nseg;
    for (int sg = 0; sg < nseg && 16 * sg * p.topk_segg < o; ++sg) {
      float g[16];
      load_list(p.topk_lists + (r * nseg + sg) * 16, g);
      merge16_desc(best, g);
    }
    rule = selection_rule(best, K);
    int32_t* meta = p.topk_meta + r * 3;
    meta[0] = rule.need;
    meta[1] = __float_as_int(rule.ge);
    meta[2] = __float_as_int(rule.eq);
  }
  const int p2 = SEG ? 0 : G;  // first item of pass 2
  const int items = SEG ? 0 : p2 + G;
  if (lane == 0)
    for (int n = 0; n < S && n < items; ++n)
      topk_issue_tile<S>(&tmS, my_tiles, my_bars, n, G, (int)r0);
  // pass 1: groups 0 .. G-1 into the running list
  int n = 0;
  for (; n < p2; ++n) {
    const int s = n % S;
    if (!topk_tile_ready<S>(my_bars + 8 * s, n, p.status)) {
      ok = false;
      break;
    }
    if (full && 16 * n < o) {
      float4 f[4];
      topk_read_tile(tiles + (warp * S + s) * kTopkTile, lane, f);
      take_group(best, f, 16 * n, o);
    }
    __syncwarp();  // every lane is done with stage s
    if (lane == 0 && n + S < items)
      topk_issue_tile<S>(&tmS, my_tiles, my_bars, n + S, G, (int)r0);
  }
  if (!SEG && full) rule = selection_rule(best, K);
  // pass 2: the same groups again, the chosen pages in ascending order
  for (; ok && n < items; ++n) {
    const int s = n % S;
    if (!topk_tile_ready<S>(my_bars + 8 * s, n, p.status)) {
      ok = false;
      break;
    }
    if (full && 16 * (n - p2) < o) {
      float4 f[4];
      topk_read_tile(tiles + (warp * S + s) * kTopkTile, lane, f);
      emit_group(f, 16 * (n - p2), o, rule, so, pos);
    }
    __syncwarp();
    if (lane == 0 && n + S < items)
      topk_issue_tile<S>(&tmS, my_tiles, my_bars, n + S, G, (int)r0);
  }
  if (!ok) {  // let the copies already issued land before the block's shared memory is reused
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < kSettleNs) __nanosleep(1000);
    return;
  }
  if (full) so[K - 1] = o;  // the own page is the row's last visible page
  __syncwarp();
  const int nrow = R - r0 < 32 ? (int)(R - r0) : 32;
  store_staged<kTopkOP>(s_out + warp * 32 * kTopkOP, idx + r0 * K, nrow, K, lane);
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

template <int S>
cudaError_t launch_topk_tma(const CUtensorMap& tm, const DevPlan& p, const float* scores,
                            int64_t pitch, int32_t* idx, unsigned grid, cudaStream_t st) {
  if (p.topk_nseg > 1 && p.topk_lists) {
    // long rows: pass 1 by segments, the merge into each row's rule, pass 2 per row over the
    // groups that can hold a chosen page
    cudaError_t e = cudaFuncSetAttribute(topk_seg_kernel<S>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)topk_smem<S>());
    if (e != cudaSuccess) return e;
    e = launch_pdl(topk_seg_kernel<S>, dim3(grid, (unsigned)p.topk_nseg), dim3(256),
                   topk_smem<S>(), st, tm, p);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(topk_tma_kernel<S, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)topk_smem<S>());
    if (e != cudaSuccess) return e;
    e = launch_pdl(topk_tma_kernel<S, true>, dim3(grid), dim3(256), topk_smem<S>(), st, tm, p,
                   idx);
    if (e != cudaSuccess) return e;
    const int64_t R = (int64_t)p.T * p.H, rows_per_block = 256 / kEmitSub;
    return launch_pdl(topk_emit_rows_kernel,
                      dim3((unsigned)((R + rows_per_block - 1) / rows_per_block)), dim3(256), 0,
                      st, p, scores, pitch, idx);
  }
  cudaError_t e = cudaFuncSetAttribute(topk_tma_kernel<S, false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)topk_smem<S>());
  if (e != cudaSuccess) return e;
  return launch_pdl(topk_tma_kernel<S, false>, dim3(grid), dim3(256), topk_smem<S>(), st, tm, p,
                    idx);
}

cudaError_t launch_topk(const DevPlan& p, const float* scores, int64_t pitch, int32_t* idx,
                        cudaStream_t st) {
  const int64_t R = (int64_t)p.T * p.H;
  if (R == 0) return cudaSuccess;
  cudaError_t e;
  if (p.K <= 16) {
    const unsigned grid = (unsigned)((R + 255) / 256);
    const bool vec = pitch % 4 == 0 && reinterpret_cast<uintptr_t>(scores) % 16 == 0;
    alignas(64) CUtensorMap tm;
    if (vec && p.max_pages >= 16 && R >= 32 &&
        encode_tmap_2d_f32_sw64(&tm, scores, (uint64_t)p.max_pages, (uint64_t)R,
                                (uint64_t)pitch * 4, 16, 32)) {
      // rows of many groups need a deeper ring per warp to cover the tile latency (4 stages: two
      // blocks per SM); short rows do better with three blocks per SM (3 stages)
      if (p.max_pages <= 128) e = launch_topk_tma<3>(tm, p, scores, pitch, idx, grid, st);
      else e = launch_topk_tma<4>(tm, p, scores, pitch, idx, grid, st);
    } else if (vec) {
      e = launch_pdl(topk_thread_kernel<true>, dim3(grid), dim3(256), 0, st, p, scores, pitch, idx);
    } else {
      e = launch_pdl(topk_thread_kernel<false>, dim3(grid), dim3(256), 0, st, p, scores, pitch, idx);
    }
    return e != cudaSuccess ? e : cudaGetLastError();
  }
  const unsigned grid = (unsigned)((R + 7) / 8);
  if (p.max_pages <= 32) {
    e = launch_pdl(topk_kernel<1>, dim3(grid), dim3(256), 0, st, p, scores, pitch, idx);
  } else if (p.max_pages <= 64) {
    e = launch_pdl(topk_kernel<2>, dim3(grid), dim3(256), 0, st, p, scores, pitch, idx);
  } else if (p.max_pages <= 128) {
    e = launch_pdl(topk_kernel<4>, dim3(grid), dim3(256), 0, st, p, scores, pitch, idx);
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
    static_assert(kMaxPagesWideK <= 32 * 32, "the widest lane layouts hold 32 x 32 pages");
    e = launch_pdl(topk_filter_kernel<32, 32>, dim3(grid), dim3(256), 0, st, p, scores, pitch, idx);
  }
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace sps
