// indexer.cu -- page indexer: S[r][p] = max over the visible keys j of page p of q_r . k_j
// ("MSA PR 36: Q8KV8 prefill indexer", Changes: per-page max by TMEM load-and-reduce,
// two Q stages, K loader reading the page table; Wrapper API: caller-owned FP32 scores).
//
// Design (GB300, one CTA per SM, persistent over a host-built work list):
//   * work item = query tile (up to 128 consecutive tokens of one request) x 1-2 query heads
//     of one KV group x a chunk of pages;
//   * warp 0 (TMA producer): per item, the Q tile of each head (3-D tensor map over
//     [T][H][D], 128-byte swizzle) into a 2-stage Q ring; per page, the physical K tile
//     (looked up in the page table) into a 3-stage K ring;
//   * warp 1 (MMA issuer, one thread): S_h = Q_h K^T, M = 128 rows, N = 128 keys, FP32
//     accumulators in TMEM, double-buffered per head (4 x 128 columns).  The two heads' K
//     steps are issued interleaved from descriptors built once per tile: a single thread has
//     to issue an MMA every ~64 cycles to keep the tensor core busy, so the loop stays short.
//     Each barrier wait in that thread stalls the MMA stream (~100 cycles), so a page step
//     has one wait and one commit: the K ring's "full" barrier also collects the epilogue's
//     release of the accumulator pair the step writes, and its "empty" barrier (the step's
//     MMAs are done) is what the epilogue waits on;
//   * warps 2-9 (epilogue, one warpgroup per head, a thread per row): the per-page row max
//     comes straight out of TMEM with tcgen05.ld.red.max; only rows whose own page it is take
//     the element-wise masked path (a warp-uniform vote picks the path).
// Operands: BF16/FP16 Q and K use kind::f16; E4M3 Q and K use kind::f8f6f4 (K = 32 per
// instruction).  Either way one 128-byte swizzled row carries 64 or 128 elements.
#include <cuda_bf16.h>

#include "ptx.cuh"
#include "sps_internal.h"

namespace sps {
namespace {

constexpr int kQStages = 2;
constexpr int kKStages = 3;
constexpr int kThreads = 320;  // 10 warps

template <int ROWB>  // bytes per Q/K row: 128 or 256
struct IdxSmem {
  static constexpr int TILE = 128 * ROWB;  // one 128-row tile
  uint8_t q[kQStages][2][TILE];
  uint8_t k[kKStages][TILE];
  uint64_t q_full[kQStages], q_empty[kQStages];
  // k_full[s]: the K tile of the stage's next page step has landed AND the accumulator pair
  // that step writes has been read out (arrivals: the producer's expect_tx + one per epilogue
  // warp); k_empty[s]: the step's MMAs are done (the K tile is free and its accumulators hold
  // the scores)
  uint64_t k_full[kKStages], k_empty[kKStages];
  uint64_t done;
  uint32_t tmem_base;
  int abort_flag;
};

template <int ROWB, bool FP8, bool BF16IN>
__global__ void __launch_bounds__(kThreads, 1)
indexer_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               DevPlan p, const int32_t* __restrict__ page_table, float* __restrict__ scores,
               int64_t pitch, float qk_scale) {
  using Smem = IdxSmem<ROWB>;
  constexpr int DB = ROWB / 128;       // 128-byte column blocks per row
  constexpr int KSTEPS = DB * 4;       // 32-byte K steps per row
  constexpr int TILE = Smem::TILE;
  constexpr uint32_t IDESC = idesc_mma(BF16IN, BF16IN, 128, 128, false, false);
  extern __shared__ uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                      ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  int32_t* status = p.status;

  if (tid == 0) {
    for (int i = 0; i < kQStages; ++i) {
      mbar_init(smem_u32(&sm.q_full[i]), 1);
      mbar_init(smem_u32(&sm.q_empty[i]), 1);
    }
    for (int i = 0; i < kKStages; ++i) {
      mbar_init(smem_u32(&sm.k_full[i]), 1 + 8);
      mbar_init(smem_u32(&sm.k_empty[i]), 1);
    }
    mbar_init(smem_u32(&sm.done), 1);
    sm.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&sm.tmem_base), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  volatile int* abort_flag = &sm.abort_flag;

  if (warp == 0) {
    // ------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      uint32_t q_it = 0, k_it = 0;
      for (int ti = blockIdx.x; ti < p.n_idx_tasks && !*abort_flag; ti += gridDim.x) {
        const IdxTask t = p.idx_tasks[ti];
        const int qs = q_it % kQStages;
        if (!mbar_wait(smem_u32(&sm.q_empty[qs]), ((q_it / kQStages) & 1) ^ 1, abort_flag, status))
          break;
        const uint32_t qf = smem_u32(&sm.q_full[qs]);
        mbar_expect_tx(qf, t.nh * TILE);
        for (int h = 0; h < t.nh; ++h)
          for (int db = 0; db < DB; ++db)
            tma_load_3d(smem_u32(sm.q[qs][h]) + db * 16384, &tmQ, db * (FP8 ? 128 : 64),
                        t.h0 + h, t.tok0, qf);
        ++q_it;
        const int32_t* pt_row = page_table + (int64_t)t.req * p.max_pages;
        for (int pg = t.page_begin; pg < t.page_end; ++pg) {
          const int ks = k_it % kKStages;
          if (!mbar_wait(smem_u32(&sm.k_empty[ks]), ((k_it / kKStages) & 1) ^ 1, abort_flag,
                         status))
            break;
          int phys = __ldg(pt_row + pg);
          if (phys < 0 || phys >= p.num_phys) {
            set_status(status, DEV_BAD_PAGE);
            phys = 0;
          }
          const uint32_t kf = smem_u32(&sm.k_full[ks]);
          mbar_expect_tx(kf, TILE);
          const int krow = (phys * p.Hkv + t.g) * 128;
          for (int db = 0; db < DB; ++db)
            tma_load_2d(smem_u32(sm.k[ks]) + db * 16384, &tmK, db * (FP8 ? 128 : 64), krow, kf);
          ++k_it;
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t q_it = 0, k_it = 0, a_it = 0;
      for (int ti = blockIdx.x; ti < p.n_idx_tasks && !*abort_flag; ti += gridDim.x) {
        const IdxTask t = p.idx_tasks[ti];
        const int qs = q_it % kQStages;
        if (!mbar_wait(smem_u32(&sm.q_full[qs]), (q_it / kQStages) & 1, abort_flag, status)) break;
        bool ok = true;
        const uint64_t ad0 = sdesc_sw128(smem_u32(sm.q[qs][0]), 16, 1024);
        const uint64_t ad1 = sdesc_sw128(smem_u32(sm.q[qs][1]), 16, 1024);
        for (int pg = t.page_begin; pg < t.page_end; ++pg) {
          const int ks = k_it % kKStages;
          const int ab = a_it & 1;
          if (!mbar_wait(smem_u32(&sm.k_full[ks]), (k_it / kKStages) & 1, abort_flag, status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // descriptors built once; a K step only moves the start address (16-byte units)
          const uint64_t bd0 = sdesc_sw128(smem_u32(sm.k[ks]), 16, 1024);
          const uint32_t d0 = tmem + (uint32_t)(ab * 256);
          if (t.nh == 2) {
#pragma unroll
            for (int kk = 0; kk < KSTEPS; ++kk) {
              const uint64_t off = (uint64_t)(((kk / 4) * 16384 + (kk % 4) * 32) >> 4);
              if (FP8) {
                mma_f8_ss(d0, ad0 + off, bd0 + off, IDESC, kk > 0);
                mma_f8_ss(d0 + 128, ad1 + off, bd0 + off, IDESC, kk > 0);
              } else {
                mma_f16_ss(d0, ad0 + off, bd0 + off, IDESC, kk > 0);
                mma_f16_ss(d0 + 128, ad1 + off, bd0 + off, IDESC, kk > 0);
              }
            }
          } else {
#pragma unroll
            for (int kk = 0; kk < KSTEPS; ++kk) {
              const uint64_t off = (uint64_t)(((kk / 4) * 16384 + (kk % 4) * 32) >> 4);
              if (FP8) mma_f8_ss(d0, ad0 + off, bd0 + off, IDESC, kk > 0);
              else mma_f16_ss(d0, ad0 + off, bd0 + off, IDESC, kk > 0);
            }
          }
          mma_commit(smem_u32(&sm.k_empty[ks]));
          ++k_it;
          ++a_it;
        }
        mma_commit(smem_u32(&sm.q_empty[qs]));
        ++q_it;
        if (!ok) break;
      }
      // every commit above has landed before the CTA may exit
      mma_commit(smem_u32(&sm.done));
      mbar_wait(smem_u32(&sm.done), 0, nullptr, status);
    }
  } else {
    // ------------------------------------------------ epilogue: warps 2..9
    const int e = (warp - 2) / 4;          // head of the pair
    const int quarter = warp % 4;          // TMEM lanes 32*quarter ...
    const int row = quarter * 32 + lane;   // tile row = token within the tile
    const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
    uint32_t a_it = 0;
    // both accumulator pairs start free: page steps 0 and 1
    if (lane == 0) {
      mbar_arrive(smem_u32(&sm.k_full[0]));
      mbar_arrive(smem_u32(&sm.k_full[1]));
    }
    for (int ti = blockIdx.x; ti < p.n_idx_tasks; ti += gridDim.x) {
      const IdxTask t = p.idx_tasks[ti];
      const ReqInfo ri = p.reqs[t.req];
      const bool valid = row < t.ntok && e < t.nh;
      const int tpos = ri.ctx + (t.tok0 - ri.tok0) + row;  // absolute position of the row
      const int o = tpos >> 7;
      float* srow = scores + ((int64_t)(t.tok0 + row) * p.H + t.h0 + e) * pitch;
      bool ok = true;
      for (int pg = t.page_begin; pg < t.page_end; ++pg) {
        const int ab = a_it & 1;
        if (!mbar_wait(smem_u32(&sm.k_empty[a_it % kKStages]), (a_it / kKStages) & 1, abort_flag,
                       status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (e < t.nh) {
          const uint32_t base = tmem + lane_addr + (uint32_t)((ab * 2 + e) * 128);
          const bool own = valid && pg == o;
          float mx = -INFINITY;
          if (__any_sync(0xffffffffu, own)) {
            const int nvis = own ? (tpos & 127) + 1 : 128;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              uint32_t v[32];
              tmem_ld32(base + c * 32, v);
              tmem_ld_wait();
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (c * 32 + j < nvis) mx = fmaxf(mx, __uint_as_float(v[j]));
            }
          } else {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              uint32_t v[32];
              const float red = tmem_ld32_max(base + c * 32, v);
              tmem_ld_wait();
              mx = fmaxf(mx, red);
            }
          }
          if (valid && pg <= o) srow[pg] = mx * qk_scale;
        }
        tc_fence_before();
        __syncwarp();
        // this accumulator pair is free for page step a_it + 2
        if (lane == 0) mbar_arrive(smem_u32(&sm.k_full[(a_it + 2) % kKStages]));
        ++a_it;
      }
      if (!ok) break;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int ROWB, bool FP8, bool BF16IN>
cudaError_t run_indexer(const DevPlan& p, int tm_dtype, const void* q, const void* kc,
                        const int32_t* page_table, float* scores, int64_t pitch, float scale,
                        cudaStream_t st) {
  const int EB = FP8 ? 1 : 2;
  alignas(64) CUtensorMap tmQ, tmK;
  const uint32_t box_inner = 128 / EB;
  if (!encode_tmap_3d(&tmQ, tm_dtype, const_cast<void*>(q), (uint64_t)p.D, (uint64_t)p.H,
                      (uint64_t)p.T, (uint64_t)p.D * EB, (uint64_t)p.H * p.D * EB, box_inner, 1,
                      128, true))
    return cudaErrorInvalidValue;
  if (!encode_tmap_2d(&tmK, tm_dtype, const_cast<void*>(kc), (uint64_t)p.D,
                      (uint64_t)p.num_phys * p.Hkv * 128, (uint64_t)p.D * EB, box_inner, 128, true))
    return cudaErrorInvalidValue;
  const int smem = (int)sizeof(IdxSmem<ROWB>) + 1024;
  auto kern = indexer_kernel<ROWB, FP8, BF16IN>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int grid = std::max(1, std::min(p.n_idx_tasks, num_sms()));
  kern<<<grid, kThreads, smem, st>>>(tmQ, tmK, p, page_table, scores, pitch, scale);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_indexer(const DevPlan& p, sps_dtype qt, sps_dtype kt, const void* q,
                           float q_scale, const void* kc, const void* kscales, float k_scale,
                           const int32_t* page_table, float* scores, int64_t pitch,
                           cudaStream_t st) {
  const float scale = q_scale * k_scale;
  if (qt == SPS_BF16 && kt == SPS_BF16) {
    if (p.D == 128) return run_indexer<256, false, true>(p, 0, q, kc, page_table, scores, pitch, scale, st);
    return run_indexer<128, false, true>(p, 0, q, kc, page_table, scores, pitch, scale, st);
  }
  if (qt == SPS_E4M3 && kt == SPS_E4M3 && p.D == 128)
    return run_indexer<128, true, false>(p, 2, q, kc, page_table, scores, pitch, scale, st);
  if (qt == SPS_E4M3 && kt == SPS_NVFP4) {
    // E4M3 codes and NVFP4 products are exact in FP16: convert both, then the FP16 MMA path
    // (the per-tensor scales stay in the FP32 epilogue)
    if (!p.qconv || !p.kconv) return cudaErrorInvalidValue;
    cudaError_t e = launch_dequant(SPS_E4M3, q, nullptr, (int64_t)p.T * p.H * p.D, p.qconv, st);
    if (e != cudaSuccess) return e;
    e = launch_dequant(SPS_NVFP4, kc, kscales, (int64_t)p.num_phys * p.Hkv * 128 * p.D, p.kconv,
                       st);
    if (e != cudaSuccess) return e;
    if (p.D == 128)
      return run_indexer<256, false, false>(p, 1, p.qconv, p.kconv, page_table, scores, pitch, scale, st);
    return run_indexer<128, false, false>(p, 1, p.qconv, p.kconv, page_table, scores, pitch, scale, st);
  }
  return cudaErrorNotSupported;
}

}  // namespace sps
