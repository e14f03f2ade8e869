// combine.cu -- streaming LSE merge of split partials into BF16 ("MSA PR 21: Q8KV4 paged
// sparse prefill", Combine: one streaming kernel for every prefill op).
//
// out[r] = sum_s w_s * partial[s][r] / sum_s w_s,  w_s = exp(lse_s - max_s lse_s), with an
// empty slot (lse = -inf) given weight 0 by selection so its partial is never read.
//
// Design (GB300): a persistent grid of 3 CTAs per SM.  A CTA owns tiles of TR consecutive
// rows (TR * D * 4 bytes = 16 KB for FP32 partials, one contiguous chunk of every split slab;
// BF16 partials, the pages' own storage, take 64 rows per tile).  A producer warp
// reads the tile's LSEs, computes the weights, and streams each split that has at least one
// finite LSE in the tile through a 4-slot shared-memory ring with one plain bulk copy
// (cp.async.bulk) per slot, completion tracked by one mbarrier per slot.  Eight consumer
// warps accumulate in FP32 registers: each lane owns one 16-byte column group (4 FP32 or 8
// BF16 partial values) of a few rows, so shared-memory reads are conflict-free and the BF16
// output of a row is one contiguous warp store.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

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

// P: partial element type, float, __nv_bfloat16 or __half.
template <int D, typename P>
__global__ void __launch_bounds__(kThreads, 3)
combine_kernel(int64_t rows, int32_t splits, const P* __restrict__ partial,
               int64_t split_stride, const float* __restrict__ lse, int64_t lse_split_stride,
               __nv_bfloat16* __restrict__ out, int64_t out_row_stride, float* __restrict__ out_lse,
               int32_t* status) {
  constexpr int PE = (int)sizeof(P);
  constexpr int TR = kSlotData / (D * PE) < 64 ? kSlotData / (D * PE) : 64;  // rows per tile
  constexpr int EPL = 16 / PE;              // partial values per lane (one 16-byte chunk)
  constexpr int LPR = D / EPL;              // lanes per row
  constexpr int RPI = 32 / LPR;             // rows per warp instruction
  constexpr int RPW = TR / 8;               // rows per consumer warp
  constexpr int IT = RPW / RPI;             // 16-byte items per lane
  static_assert(IT >= 1 && RPW % RPI == 0, "layout");
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
  pdl_wait();  // the prologue may overlap the previous kernel (the forward)

  if (warp == 8) {
    // ---------------- producer warp
    uint32_t slot = 0, phase = 0;
    for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
      // tiles from the last rows down: a page-parallel forward writes the highest pages last,
      // and only late rows select those, so the first tiles read partials still in L2
      const int64_t r0 = (ntiles - 1 - tile) * TR;
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
            uint32_t bytes = (uint32_t)nvalid * D * PE;
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
    const int c4 = lane % LPR;          // 16-byte column group
    for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
      const int64_t r0 = (ntiles - 1 - tile) * TR;  // same order as the producer
      float acc[IT][EPL];
      float wsum[IT];
#pragma unroll
      for (int i = 0; i < IT; ++i) {
        wsum[i] = 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) acc[i][e] = 0.f;
      }
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
            const uint4 raw = reinterpret_cast<const uint4*>(sm.data[slot])[rr * LPR + c4];
            const uint32_t wd[4] = {raw.x, raw.y, raw.z, raw.w};
            float v[EPL];
#pragma unroll
            for (int e = 0; e < EPL; ++e) {
              if (PE == 4) {
                v[e] = __uint_as_float(wd[e]);
              } else if (std::is_same<P, __half>::value) {
                const uint32_t hw = wd[e / 2];
                const __half2 h2 = *reinterpret_cast<const __half2*>(&hw);
                v[e] = e & 1 ? __high2float(h2) : __low2float(h2);
              } else {
                v[e] = __uint_as_float(e & 1 ? wd[e / 2] & 0xffff0000u : wd[e / 2] << 16);
              }
            }
            const bool use = w != 0.f;
#pragma unroll
            for (int e = 0; e < EPL; ++e) acc[i][e] = use ? fmaf(w, v[e], acc[i][e]) : acc[i][e];
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
            uint32_t pk[EPL / 2];
#pragma unroll
            for (int e = 0; e < EPL; e += 2) {
              __nv_bfloat162 b2 = __floats2bfloat162_rn(acc[i][e] * inv, acc[i][e + 1] * inv);
              pk[e / 2] = *reinterpret_cast<uint32_t*>(&b2);
            }
            if (EPL == 4)
              *reinterpret_cast<uint2*>(out + r * out_row_stride + c4 * EPL) = make_uint2(pk[0], pk[1]);
            else
              *reinterpret_cast<uint4*>(out + r * out_row_stride + c4 * EPL) =
                  make_uint4(pk[0], pk[1], pk[EPL / 2 > 2 ? 2 : 0], pk[EPL / 2 > 3 ? 3 : 0]);
            if (out_lse && c4 == 0)
              out_lse[r] = wsum[i] > 0.f ? mrow[i] + logf(wsum[i]) : -INFINITY;
          }
        }
      }
      if (!ok) break;
    }
  }
  // a block exits only when all its threads have: the producer's copies land first
  settle_after_abort(&sm.abort_flag);
}

template <typename P>
cudaError_t launch_combine_t(int64_t rows, int32_t splits, int32_t D, const P* partial,
                             int64_t split_stride, const float* lse, int64_t lse_split_stride,
                             void* out, int64_t out_row_stride, float* out_lse, int32_t* status,
                             cudaStream_t st) {
  const int smem = (int)sizeof(CombineSmem) + 128;
  const int TR = std::min(64, kSlotData / (D * (int)sizeof(P)));
  int64_t ntiles = (rows + TR - 1) / TR;
  int64_t grid = std::min<int64_t>(ntiles, 3LL * num_sms());
  if (grid < 1) return cudaSuccess;
  auto* o = static_cast<__nv_bfloat16*>(out);
  auto kern = D == 128 ? combine_kernel<128, P> : combine_kernel<64, P>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  e = launch_pdl(kern, dim3((unsigned)grid), dim3(kThreads), smem, st, rows, splits, partial,
                 split_stride, lse, lse_split_stride, o, out_row_stride, out_lse, status);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

cudaError_t launch_combine(int64_t rows, int32_t splits, int32_t D, const float* partial,
                           int64_t split_stride, const float* lse, int64_t lse_split_stride,
                           void* out, int64_t out_row_stride, float* out_lse, int32_t* status,
                           cudaStream_t st) {
  return launch_combine_t<float>(rows, splits, D, partial, split_stride, lse, lse_split_stride,
                                 out, out_row_stride, out_lse, status, st);
}

cudaError_t launch_combine_bf16p(int64_t rows, int32_t splits, int32_t D, const void* partial,
                                 int64_t split_stride, const float* lse, int64_t lse_split_stride,
                                 void* out, int64_t out_row_stride, float* out_lse,
                                 int32_t* status, cudaStream_t st) {
  return launch_combine_t<__nv_bfloat16>(rows, splits, D,
                                         static_cast<const __nv_bfloat16*>(partial), split_stride,
                                         lse, lse_split_stride, out, out_row_stride, out_lse,
                                         status, st);
}

cudaError_t launch_combine_f16p(int64_t rows, int32_t splits, int32_t D, const void* partial,
                                int64_t split_stride, const float* lse, int64_t lse_split_stride,
                                void* out, int64_t out_row_stride, float* out_lse,
                                int32_t* status, cudaStream_t st) {
  return launch_combine_t<__half>(rows, splits, D, static_cast<const __half*>(partial),
                                  split_stride, lse, lse_split_stride, out, out_row_stride,
                                  out_lse, status, st);
}

}  // namespace sps
