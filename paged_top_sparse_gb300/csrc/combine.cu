// combine.cu -- streaming LSE merge of split partials into BF16 ("MSA PR 21: Q8KV4 paged
// sparse prefill", Combine: one streaming kernel for every prefill op).
//
// out[r] = sum_s w_s * partial[s][r] / sum_s w_s,  w_s = exp(lse_s - max_s lse_s), with an
// empty slot (lse = -inf) given weight 0 by selection so its partial is never read.
//
// Design (GB300): a persistent grid of 3 CTAs per SM.  A CTA owns tiles of TR consecutive
// rows (TR * D * 4 bytes = 16 KB, one contiguous chunk of every split slab).  A producer warp
// reads the tile's LSEs, computes the weights, and streams each split that has at least one
// finite LSE in the tile through a 4-slot shared-memory ring with one plain bulk copy
// (cp.async.bulk) per slot, completion tracked by one mbarrier per slot.  Eight consumer
// warps accumulate in FP32 registers: each lane owns one float4 column group of 4 rows, so
// shared-memory reads are conflict-free and the BF16 output of a row is one contiguous
// 256-byte (D=128) warp store.
#include <cuda_bf16.h>

#include "ptx.cuh"
#include "sps_internal.h"

namespace sps {
namespace {

constexpr int kSlots = 4;
constexpr int kSlotData = 16384;         // bytes of partial data per slot
constexpr int kConsumers = 256;          // 8 warps
constexpr int kThreads = kConsumers + 32;

struct SlotHeader {
  float w[64];      // weight of each tile row for this slot's split (0 for -inf rows)
  float m[64];      // max LSE of each tile row (valid on the tile's last slot)
  int32_t split;    // -1: the tile has no finite LSE at all (no data in this slot)
  int32_t last;     // 1 on the tile's last slot
  int32_t pad[14];
};

struct __align__(128) CombineSmem {
  float data[kSlots][kSlotData / 4];
  SlotHeader hdr[kSlots];
  uint64_t full[kSlots];
  uint64_t empty[kSlots];
  int abort_flag;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 3)
combine_kernel(int64_t rows, int32_t splits, const float* __restrict__ partial,
               int64_t split_stride, const float* __restrict__ lse, int64_t lse_split_stride,
               __nv_bfloat16* __restrict__ out, int64_t out_row_stride, float* __restrict__ out_lse,
               int32_t* status) {
  constexpr int TR = kSlotData / (D * 4);   // rows per tile: 32 (D=128) or 64 (D=64)
  constexpr int LPR = D / 4;                // lanes per row (one float4 each)
  constexpr int RPI = 32 / LPR;             // rows per warp instruction
  constexpr int RPW = TR / 8;               // rows per consumer warp
  constexpr int IT = RPW / RPI;             // float4 items per lane (always 4)
  static_assert(IT == 4, "layout");
  extern __shared__ uint8_t smem_raw[];
  CombineSmem& sm = *reinterpret_cast<CombineSmem*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int64_t ntiles = (rows + TR - 1) / TR;

  if (tid == 0) {
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(smem_u32(&sm.full[s]), 1);
      mbar_init(smem_u32(&sm.empty[s]), kConsumers / 32);
    }
    sm.abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == 8) {
    // ---------------- producer warp
    uint32_t slot = 0, phase = 0;
    for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
      const int64_t r0 = tile * TR;
      const int nvalid = (int)((rows - r0) < TR ? (rows - r0) : TR);
      constexpr int RPL = TR / 32;  // rows per lane: 1 or 2
      float m[RPL];
      uint64_t act = 0;  // bit s: some row of the tile has a finite lse at split s
#pragma unroll
      for (int j = 0; j < RPL; ++j) m[j] = -INFINITY;
      // 16 splits per batch of independent loads, so their latencies overlap
      for (int s0 = 0; s0 < splits; s0 += 16) {
        float x[16][RPL];
#pragma unroll
        for (int u = 0; u < 16; ++u)
#pragma unroll
          for (int j = 0; j < RPL; ++j) {
            int rr = lane + 32 * j;
            x[u][j] = (s0 + u < splits && rr < nvalid)
                          ? __ldg(lse + (s0 + u) * lse_split_stride + r0 + rr)
                          : -INFINITY;
          }
#pragma unroll
        for (int u = 0; u < 16; ++u)
#pragma unroll
          for (int j = 0; j < RPL; ++j) {
            m[j] = fmaxf(m[j], x[u][j]);
            if (__any_sync(0xffffffffu, x[u][j] != -INFINITY)) act |= 1ull << (s0 + u);
          }
      }
      const int nact = __popcll(act);
      for (int k = 0; k < (nact > 0 ? nact : 1); ++k) {
        int s = -1;
        if (nact > 0) {  // k-th set bit of act
          uint64_t a = act;
          for (int q = 0; q < k; ++q) a &= a - 1;
          s = __ffsll((long long)a) - 1;
        }
        if (!mbar_wait(smem_u32(&sm.empty[slot]), phase ^ 1, &sm.abort_flag, status)) break;
        SlotHeader& h = sm.hdr[slot];
#pragma unroll
        for (int j = 0; j < RPL; ++j) {
          int rr = lane + 32 * j;
          float w = 0.f;
          if (s >= 0 && rr < nvalid) {
            float x = __ldg(lse + s * lse_split_stride + r0 + rr);
            w = (x == -INFINITY) ? 0.f : expf(x - m[j]);  // select, never exp(-inf - -inf)
          }
          h.w[rr] = w;
          h.m[rr] = m[j];
        }
        if (lane == 0) {
          h.split = s;
          h.last = (k == (nact > 0 ? nact : 1) - 1);
        }
        __syncwarp();
        if (lane == 0) {
          uint32_t full = smem_u32(&sm.full[slot]);
          if (s >= 0) {
            uint32_t bytes = (uint32_t)nvalid * D * 4;
            mbar_expect_tx(full, bytes);
            bulk_load(smem_u32(sm.data[slot]), partial + s * split_stride + r0 * D, bytes, full);
          } else {
            mbar_arrive(full);
          }
        }
        __syncwarp();
        if (++slot == kSlots) { slot = 0; phase ^= 1; }
      }
      if (sm.abort_flag) break;
    }
  } else if (warp < 8) {
    // ---------------- consumer warps
    uint32_t slot = 0, phase = 0;
    const int rsub = lane / LPR;        // row within an instruction
    const int c4 = lane % LPR;          // float4 column group
    for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
      const int64_t r0 = tile * TR;
      float4 acc[IT];
      float wsum[IT];
#pragma unroll
      for (int i = 0; i < IT; ++i) { acc[i] = make_float4(0.f, 0.f, 0.f, 0.f); wsum[i] = 0.f; }
      bool done = false, ok = true;
      while (!done) {
        if (!mbar_wait(smem_u32(&sm.full[slot]), phase, &sm.abort_flag, status)) { ok = false; break; }
        const SlotHeader& h = sm.hdr[slot];
        const bool has_data = h.split >= 0;
        done = h.last != 0;
#pragma unroll
        for (int i = 0; i < IT; ++i) {
          int rr = warp * RPW + i * RPI + rsub;
          float w = h.w[rr];
          wsum[i] += w;
          if (has_data) {
            // a row whose lse is -inf at this split has w == 0 and its partial may hold
            // anything (it was never written): select, never multiply it in
            const float4 v = reinterpret_cast<const float4*>(sm.data[slot])[rr * LPR + c4];
            const bool use = w != 0.f;
            acc[i].x = use ? fmaf(w, v.x, acc[i].x) : acc[i].x;
            acc[i].y = use ? fmaf(w, v.y, acc[i].y) : acc[i].y;
            acc[i].z = use ? fmaf(w, v.z, acc[i].z) : acc[i].z;
            acc[i].w = use ? fmaf(w, v.w, acc[i].w) : acc[i].w;
          }
        }
        float mrow[IT];
        if (done) {
#pragma unroll
          for (int i = 0; i < IT; ++i) mrow[i] = h.m[warp * RPW + i * RPI + rsub];
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sm.empty[slot]));
        if (++slot == kSlots) { slot = 0; phase ^= 1; }
        if (done) {
#pragma unroll
          for (int i = 0; i < IT; ++i) {
            int rr = warp * RPW + i * RPI + rsub;
            int64_t r = r0 + rr;
            if (r >= rows) continue;
            float inv = wsum[i] > 0.f ? 1.f / wsum[i] : 0.f;
            __nv_bfloat162 lo = __floats2bfloat162_rn(acc[i].x * inv, acc[i].y * inv);
            __nv_bfloat162 hi = __floats2bfloat162_rn(acc[i].z * inv, acc[i].w * inv);
            uint2 pk;
            pk.x = *reinterpret_cast<uint32_t*>(&lo);
            pk.y = *reinterpret_cast<uint32_t*>(&hi);
            *reinterpret_cast<uint2*>(out + r * out_row_stride + c4 * 4) = pk;
            if (out_lse && c4 == 0)
              out_lse[r] = wsum[i] > 0.f ? mrow[i] + logf(wsum[i]) : -INFINITY;
          }
        }
      }
      if (!ok) break;
    }
  }
}

}  // namespace

cudaError_t launch_combine(int64_t rows, int32_t splits, int32_t D, const float* partial,
                           int64_t split_stride, const float* lse, int64_t lse_split_stride,
                           void* out, int64_t out_row_stride, float* out_lse, int32_t* status,
                           cudaStream_t st) {
  const int smem = (int)sizeof(CombineSmem) + 128;
  const int TR = kSlotData / (D * 4);
  int64_t ntiles = (rows + TR - 1) / TR;
  int64_t grid = std::min<int64_t>(ntiles, 3LL * num_sms());
  if (grid < 1) return cudaSuccess;
  auto* o = static_cast<__nv_bfloat16*>(out);
  if (D == 128) {
    cudaFuncSetAttribute(combine_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    combine_kernel<128><<<(unsigned)grid, kThreads, smem, st>>>(
        rows, splits, partial, split_stride, lse, lse_split_stride, o, out_row_stride, out_lse,
        status);
  } else {
    cudaFuncSetAttribute(combine_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    combine_kernel<64><<<(unsigned)grid, kThreads, smem, st>>>(
        rows, splits, partial, split_stride, lse, lse_split_stride, o, out_row_stride, out_lse,
        status);
  }
  return cudaGetLastError();
}

}  // namespace sps
