// indexer.cu -- page indexer: S[r][p] = max over the visible keys j of page p of q_r . k_j
// ("MSA PR 36: Q8KV8 prefill indexer", Changes: per-page max by TMEM load-and-reduce,
// two Q stages, K loader reading the page table; Wrapper API: caller-owned FP32 scores).
//
// Design (GB300, one CTA per SM, persistent over a host-built work list):
//   * work item = query tile (up to 128 consecutive tokens of one request) x 1-2 query heads
//     of one KV group x a chunk of pages, walked two pages at a time;
//   * warp 0 (TMA producer): per item, the Q tile of each head (3-D tensor map over
//     [T][H][D], 128-byte swizzle) into a ring of three one-head slots (the next item's first
//     head loads while the current item runs); per page pair, the two physical K tiles
//     (looked up in the page table) stacked into one 256-row operand, in a ring of 2 stages
//     (4 for 128-byte rows);
//   * warp 1 (MMA issuer, one thread): S_h = Q_h K^T with M = 128 rows and N = 256 keys (two
//     pages per instruction), FP32 accumulators in TMEM, one 256-column buffer per head.  A
//     128 x 128 x 16 MMA with both operands in shared memory reads 8 KB in 64 cycles, all of
//     the SM's shared-memory bandwidth, and the K tiles land in the same memory; at N = 256
//     one read of the Q operand serves two pages, which leaves room for the K loads.  Each
//     barrier wait in this thread stalls the MMA stream, so a head step has one wait and one
//     commit: the K ring's "full" barrier also collects the release of head 0's accumulator,
//     and head 1's step waits only for its own accumulator;
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

constexpr int kQSlots = 3;     // one-head Q tiles: an item's two heads + the next item's first
constexpr int kThreads = 320;  // 10 warps

template <int ROWB>  // bytes per Q/K row: 128 or 256
struct IdxSmem {
  static constexpr int TILE = 128 * ROWB;  // one 128-row tile
  // page-pair stages: the shorter rows' pairs take half the MMA time and half the space, so
  // they get a deeper ring to hide the same load latency
  static constexpr int kKStages = ROWB == 128 ? 4 : 2;
  uint8_t q[kQSlots][TILE];                // [column block][128 rows][128 B]
  uint8_t k[kKStages][2 * TILE];           // [column block][256 rows][128 B], page A then B
  uint64_t q_full[kQSlots], q_empty[kQSlots];
  // k_full[s]: the stage's page pair has landed AND head 0's accumulator has been read out
  // (arrivals: the producer's expect_tx + one per head-0 epilogue warp); a1_free[s]: head 1's
  // accumulator has been read out for the stage's pair; k_empty[s]: both heads' MMAs of the
  // pair are done (the K tiles are free, head 1's scores are in TMEM); a0_full: head 0's MMAs
  // of the current pair are done
  uint64_t k_full[kKStages], a1_free[kKStages], k_empty[kKStages];
  uint64_t a0_full;
  uint64_t done;
  uint32_t tmem_base;
  int abort_flag;
};

template <int ROWB, bool FP8, bool BF16IN>
__global__ void __launch_bounds__(kThreads, 1)
indexer_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               DevPlan p, const int32_t* __restrict__ page_table, float* __restrict__ scores,
               int64_t pitch, float qk_scale, int logical_keys) {
  using Smem = IdxSmem<ROWB>;
  constexpr int DB = ROWB / 128;       // 128-byte column blocks per row
  constexpr int KSTEPS = DB * 4;       // 32-byte K steps per row
  constexpr int TILE = Smem::TILE;
  constexpr int kKStages = Smem::kKStages;
  constexpr int CB = 128 * 128;        // bytes of one column block of a 128-row tile
  constexpr uint32_t IDESC2 = idesc_mma(BF16IN, BF16IN, 128, 256, false, false);
  constexpr uint32_t IDESC1 = idesc_mma(BF16IN, BF16IN, 128, 128, false, false);
  extern __shared__ uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                      ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  int32_t* status = p.status;

  if (tid == 0) {
    for (int i = 0; i < kQSlots; ++i) {
      mbar_init(smem_u32(&sm.q_full[i]), 1);
      mbar_init(smem_u32(&sm.q_empty[i]), 1);
    }
    for (int i = 0; i < kKStages; ++i) {
      mbar_init(smem_u32(&sm.k_full[i]), 1 + 4);
      mbar_init(smem_u32(&sm.a1_free[i]), 4);
      mbar_init(smem_u32(&sm.k_empty[i]), 1);
    }
    mbar_init(smem_u32(&sm.a0_full), 1);
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
  // the prologue above may overlap the previous kernel (the plan upload); from here on the
  // kernel reads what it wrote
  pdl_wait();
  pdl_trigger();
  const uint32_t tmem = sm.tmem_base;  // head h's accumulator: columns 256 h .. 256 h + 255
  volatile int* abort_flag = &sm.abort_flag;

  if (warp == 0) {
    // ------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      uint32_t jp = 0, hs = 0;  // page pairs and Q head slots loaded so far
      bool ok = true;
      for (int ti = blockIdx.x; ti < p.n_idx_tasks && ok && !*abort_flag; ti += gridDim.x) {
        const IdxTask t = p.idx_tasks[ti];
        // Q of head 0 goes before the item's first page pair, Q of head 1 after it: head 1's
        // slot may still hold the previous item's head 0
        const int32_t* pt_row = page_table + (int64_t)t.req * p.max_pages;
        for (int pb = t.page_begin; pb < t.page_end && ok; pb += 2, ++jp) {
          if (pb == t.page_begin) {  // Q of head 0
            const uint32_t s0 = hs % kQSlots;
            if (!mbar_wait(smem_u32(&sm.q_empty[s0]), ((hs / kQSlots) & 1) ^ 1, abort_flag,
                           status)) {
              ok = false;
              break;
            }
            const uint32_t qf = smem_u32(&sm.q_full[s0]);
            mbar_expect_tx(qf, TILE);
            for (int db = 0; db < DB; ++db)
              tma_load_3d(smem_u32(sm.q[s0]) + db * CB, &tmQ, db * (FP8 ? 128 : 64), t.h0,
                          t.tok0, qf);
          }
          const int ks = jp % kKStages;
          if (!mbar_wait(smem_u32(&sm.k_empty[ks]), ((jp / kKStages) & 1) ^ 1, abort_flag,
                         status)) {
            ok = false;
            break;
          }
          const int npg = min(2, t.page_end - pb);
          const uint32_t kf = smem_u32(&sm.k_full[ks]);
          mbar_expect_tx(kf, npg * TILE);
          for (int u = 0; u < npg; ++u) {
            // logical_keys: the key tiles were copied in logical page order (global page slot)
            int phys = logical_keys ? p.reqs[t.req].page_base + pb + u : __ldg(pt_row + pb + u);
            if (!logical_keys && (phys < 0 || phys >= p.num_phys)) {
              set_status(status, DEV_BAD_PAGE);
              phys = 0;
            }
            const int krow = (phys * p.Hkv + t.g) * 128;
            for (int db = 0; db < DB; ++db)
              tma_load_2d(smem_u32(sm.k[ks]) + db * 2 * CB + u * CB, &tmK, db * (FP8 ? 128 : 64),
                          krow, kf);
          }
          if (pb == t.page_begin && t.nh == 2) {  // Q of head 1, after the first pair
            const uint32_t s1 = (hs + 1) % kQSlots;
            if (!mbar_wait(smem_u32(&sm.q_empty[s1]), (((hs + 1) / kQSlots) & 1) ^ 1, abort_flag,
                           status)) {
              ok = false;
              break;
            }
            const uint32_t qf = smem_u32(&sm.q_full[s1]);
            mbar_expect_tx(qf, TILE);
            for (int db = 0; db < DB; ++db)
              tma_load_3d(smem_u32(sm.q[s1]) + db * CB, &tmQ, db * (FP8 ? 128 : 64), t.h0 + 1,
                          t.tok0, qf);
          }
        }
        hs += t.nh;
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t jp = 0, hs = 0;
      bool ok = true;
      for (int ti = blockIdx.x; ti < p.n_idx_tasks && ok && !*abort_flag; ti += gridDim.x) {
        const IdxTask t = p.idx_tasks[ti];
        const uint32_t s0 = hs % kQSlots, s1 = (hs + 1) % kQSlots;
        if (!mbar_wait(smem_u32(&sm.q_full[s0]), (hs / kQSlots) & 1, abort_flag, status)) break;
        // descriptors built once per item; a K step only moves the start address (16-byte units)
        const uint64_t ad0 = sdesc_sw128(smem_u32(sm.q[s0]), 16, 1024);
        const uint64_t ad1 = sdesc_sw128(smem_u32(sm.q[s1]), 16, 1024);
        for (int pb = t.page_begin; pb < t.page_end; pb += 2, ++jp) {
          const int ks = jp % kKStages;
          const uint32_t ph = (jp / kKStages) & 1;
          const uint32_t idesc = pb + 1 < t.page_end ? IDESC2 : IDESC1;
          if (!mbar_wait(smem_u32(&sm.k_full[ks]), ph, abort_flag, status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t bd = sdesc_sw128(smem_u32(sm.k[ks]), 16, 1024);
#pragma unroll
          for (int kk = 0; kk < KSTEPS; ++kk) {
            const uint64_t oa = (uint64_t)(((kk / 4) * CB + (kk % 4) * 32) >> 4);
            const uint64_t ob = (uint64_t)(((kk / 4) * 2 * CB + (kk % 4) * 32) >> 4);
            if (FP8) mma_f8_ss(tmem, ad0 + oa, bd + ob, idesc, kk > 0);
            else mma_f16_ss(tmem, ad0 + oa, bd + ob, idesc, kk > 0);
          }
          mma_commit(smem_u32(&sm.a0_full));
          if (t.nh == 2) {
            if ((pb == t.page_begin &&
                 !mbar_wait(smem_u32(&sm.q_full[s1]), ((hs + 1) / kQSlots) & 1, abort_flag,
                            status)) ||
                !mbar_wait(smem_u32(&sm.a1_free[ks]), ph, abort_flag, status)) {
              ok = false;
              break;
            }
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < KSTEPS; ++kk) {
              const uint64_t oa = (uint64_t)(((kk / 4) * CB + (kk % 4) * 32) >> 4);
              const uint64_t ob = (uint64_t)(((kk / 4) * 2 * CB + (kk % 4) * 32) >> 4);
              if (FP8) mma_f8_ss(tmem + 256, ad1 + oa, bd + ob, idesc, kk > 0);
              else mma_f16_ss(tmem + 256, ad1 + oa, bd + ob, idesc, kk > 0);
            }
          }
          mma_commit(smem_u32(&sm.k_empty[ks]));
        }
        mma_commit(smem_u32(&sm.q_empty[s0]));
        if (t.nh == 2) mma_commit(smem_u32(&sm.q_empty[s1]));
        hs += t.nh;
      }
      // every commit above has landed before the CTA may exit
      mma_commit(smem_u32(&sm.done));
      mbar_wait(smem_u32(&sm.done), 0, nullptr, status);
    }
  } else {
    // ------------------------------------------------ epilogue: warps 2..9
    const int e = (warp - 2) / 4;          // head of the pair = accumulator
    const int quarter = warp % 4;          // TMEM lanes 32*quarter ...
    const int row = quarter * 32 + lane;   // tile row = token within the tile
    const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
    // Every item of a plan has the same head count (two when the group's query-head count is
    // even).  With one head, the second warpgroup has no accumulator to read and nothing waits
    // for its arrivals, so it takes no part: a warpgroup that only waited and arrived could fall
    // a whole ring behind the K barriers and then mistake a later phase for the one it wants.
    const int nh_plan = (p.Hg % 2 == 0) ? 2 : 1;
    const int n_items = e < nh_plan ? p.n_idx_tasks : 0;
    uint32_t jp = 0;
    // both accumulators start free (page pair 0)
    if (lane == 0 && e < nh_plan) mbar_arrive(smem_u32(e == 0 ? &sm.k_full[0] : &sm.a1_free[0]));
    for (int ti = blockIdx.x; ti < n_items; ti += gridDim.x) {
      const IdxTask t = p.idx_tasks[ti];
      const ReqInfo ri = p.reqs[t.req];
      const bool valid = row < t.ntok && e < t.nh;
      const int tpos = ri.ctx + (t.tok0 - ri.tok0) + row;  // absolute position of the row
      const int o = tpos >> 7;
      float* srow = scores + ((int64_t)(t.tok0 + row) * p.H + t.h0 + e) * pitch;
      bool ok = true;
      for (int pb = t.page_begin; pb < t.page_end; pb += 2, ++jp) {
        const int ks = jp % kKStages;
        const bool got = e == 0
            ? mbar_wait(smem_u32(&sm.a0_full), jp & 1, abort_flag, status)
            : mbar_wait(smem_u32(&sm.k_empty[ks]), (jp / kKStages) & 1, abort_flag, status);
        if (!got) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (e < t.nh) {
          const int npg = min(2, t.page_end - pb);
          for (int u = 0; u < npg; ++u) {
            const int pg = pb + u;
            const uint32_t base = tmem + lane_addr + (uint32_t)(e * 256 + u * 128);
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
        }
        tc_fence_before();
        __syncwarp();
        // this accumulator is free for page pair jp + 1
        if (lane == 0)
          mbar_arrive(smem_u32(e == 0 ? &sm.k_full[(jp + 1) % kKStages]
                                      : &sm.a1_free[(jp + 1) % kKStages]));
      }
      if (!ok) break;
    }
  }
  settle_after_abort(abort_flag);
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
                        cudaStream_t st, bool logical_keys = false) {
  const int EB = FP8 ? 1 : 2;
  alignas(64) CUtensorMap tmQ, tmK;
  const uint32_t box_inner = 128 / EB;
  if (!encode_tmap_3d(&tmQ, tm_dtype, const_cast<void*>(q), (uint64_t)p.D, (uint64_t)p.H,
                      (uint64_t)p.T, (uint64_t)p.D * EB, (uint64_t)p.H * p.D * EB, box_inner, 1,
                      128, true))
    return cudaErrorInvalidValue;
  const uint64_t key_tiles = (uint64_t)(logical_keys ? p.total_pages : p.num_phys) * p.Hkv;
  if (!encode_tmap_2d(&tmK, tm_dtype, const_cast<void*>(kc), (uint64_t)p.D, key_tiles * 128,
                      (uint64_t)p.D * EB, box_inner, 128, true))
    return cudaErrorInvalidValue;
  const int smem = (int)sizeof(IdxSmem<ROWB>) + 1024;
  auto kern = indexer_kernel<ROWB, FP8, BF16IN>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int grid = std::max(1, std::min(p.n_idx_tasks, num_sms()));
  e = launch_pdl(kern, dim3(grid), dim3(kThreads), smem, st, tmQ, tmK, p, page_table, scores,
                 pitch, scale, logical_keys ? 1 : 0);
  return e != cudaSuccess ? e : cudaGetLastError();
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
    // E4M3 codes and NVFP4 products are exact in FP16: convert Q, and the key tiles of the
    // pages the batch sees (through the page table, into logical order: every one of them is
    // read, by many query tiles, so each is converted once rather than in every loader), then
    // the FP16 MMA path (the per-tensor scales stay in the FP32 epilogue)
    if (!p.qconv || !p.kconv) return cudaErrorInvalidValue;
    cudaError_t e = launch_dequant(SPS_E4M3, q, nullptr, (int64_t)p.T * p.H * p.D, p.qconv, st);
    if (e != cudaSuccess) return e;
    e = launch_dequant_pages(p, kc, kscales, page_table, p.kconv, st);
    if (e != cudaSuccess) return e;
    if (p.D == 128)
      return run_indexer<256, false, false>(p, 1, p.qconv, p.kconv, page_table, scores, pitch,
                                            scale, st, true);
    return run_indexer<128, false, false>(p, 1, p.qconv, p.kconv, page_table, scores, pitch,
                                          scale, st, true);
  }
  return cudaErrorNotSupported;
}

}  // namespace sps
