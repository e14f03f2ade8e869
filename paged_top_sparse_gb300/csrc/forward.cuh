// forward.cuh -- page-parallel sparse forward ("MSA PR 21: Q8KV4 paged sparse prefill", K1):
// one work item per (page, KV head, query split), the rows that selected the page streamed
// through in groups of 128; every (row, page) pair yields a partial output normalised by its
// row sum plus the LSE, written into the split-strided partial buffer at the row's slot.
// Only the row's own page is causally masked; K/V come through the page table.
//
// Design (GB300, one CTA per SM, persistent over the device-built work list):
//   (warps 0-3 form the producer/MMA warpgroup, 4-7 the softmax, 8-11 the epilogue, 12-15 the
//   Q gather; setmaxnreg moves registers to the softmax)
//   warp 0     the item's K and V: BF16 tiles by TMA (128-byte swizzle, separate barriers: the
//              next item's K loads as soon as the last S of the current item has read the old
//              tile, its V after the last P.V); NVFP4 codes and scales by plain bulk copies
//              into a raw staging area one item ahead of their conversion;
//   warps 2-3  the loaders' conversions: BF16 V -> FP16 in place; NVFP4 K and V -> FP16 (or K
//              -> E4M3 on the FP8 route) straight from the raw staging into the swizzled
//              operand tiles, exactly (code x scale), once per item;
//   warps 12-15 per group the 128 query rows by TMA tile::gather4 into the same swizzled
//              layout, in a ring of Q stages (as many as the shared memory holds, up to four).
//              A warp issues its gathers one lane after another, so the group's gathers are
//              spread over four warps (one per SM sub-partition); the row indices of the next
//              group (across item boundaries) are loaded while the current one is issued;
//   warp 1     MMA issuer (one thread): S = Q K^T (shared x shared, N = 128 keys) into a
//              double-buffered TMEM accumulator, and O = P V with P read from TMEM (the
//              softmax overwrites S with P in place) and V as an MN-major FP16 operand; it
//              polls both streams and issues whichever is ready, so S of group g+1 overlaps
//              the softmax of group g without a late Q tile delaying P.V of group g;
//   warps 4-7  softmax, a thread per row: per group, one TMEM read of the row
//              (tcgen05.ld.red.max gives the max unless some lane of the warp owns the page,
//              then the masked element-wise path), p = 2^(s c - m c) rounded to FP16 back into
//              TMEM over S, l = sum p, LSE = m * scale + ln l straight to global;
//   warps 8-11 epilogue, a thread per row: O / l from TMEM into a padded staging row, then one
//              bulk copy of the whole row into partial[slot][row].  On this GPU a bulk store
//              costs the SM's TMA engine roughly the same whatever its size, and whole 512-byte
//              rows reach the HBM write bandwidth; the load/store unit's stores do not.
#pragma once
#include <cuda_bf16.h>
#include <cstring>
#include <cuda_fp16.h>

#include "ptx.cuh"
#include "sps_internal.h"

namespace sps {
namespace fwd {

constexpr int kThreads = 512;  // 4 warpgroups

// Operand modes: kModeBF16 (Q, K, V BF16), kModeF16 (Q FP16 -- the exact copy of E4M3 codes --
// and NVFP4 K/V converted in the loader), kModeFP8QK (Q E4M3 bytes, NVFP4 K rounded to E4M3,
// S on the FP8 tensor core; V FP16).
constexpr int kModeBF16 = 0, kModeF16 = 1, kModeFP8QK = 2;
// Partial storage: FP32, BF16 or FP16 (nearest even).
constexpr int kPF32 = 0, kPBF16 = 1, kPF16 = 2;

template <int D, int MODE, int PT>
struct FwdSmem {
  static constexpr bool RAW = MODE != kModeBF16;  // K/V arrive as NVFP4 codes + scales
  static constexpr int QE = MODE == kModeFP8QK ? 1 : 2;  // bytes per Q / K element
  static constexpr int PE = PT == kPF32 ? 4 : 2;         // bytes per partial element
  static constexpr int TQK = 128 * D * QE;  // 128-row Q or K tile
  static constexpr int TV = 128 * D * 2;    // 128-row V tile (16-bit)
  static constexpr int RC = 128 * D / 2;    // NVFP4 codes of one tile
  static constexpr int RSC = 128 * D / 16;  // its E4M3 scales
  static constexpr int RAWB = RAW ? RC + RSC : 16;
  static constexpr int EPR = D * PE + 16;  // staging row pitch (pad: conflict-free writes)
  static constexpr int EPB = 32 * EPR;     // one epilogue warp's 32 rows
  static constexpr int kBudget = 227 * 1024 - 1024;  // dynamic smem minus the alignment slack
  static constexpr int FIXED = TQK + TV + 2 * RAWB + 4 * EPB + 4096;
  static constexpr int QS0 = (kBudget - FIXED) / TQK;
  static constexpr int QS = QS0 > 4 ? 4 : QS0;  // Q ring stages
  static_assert(QS >= 2, "shared memory");
  uint8_t k[TQK];
  uint8_t v[TV];
  uint8_t q[QS][TQK];
  alignas(16) uint8_t kraw[RAWB];
  alignas(16) uint8_t vraw[RAWB];
  alignas(16) uint8_t ep[4][EPB];
  float inv_l[2][128];
  int2 rs[2][128];
  uint64_t k_full, k_empty, v_full, v_empty, v_ready;
  uint64_t kraw_full, kraw_empty, vraw_full, vraw_empty;
  uint64_t q_full[QS], q_empty[QS];
  uint64_t s_full[2], p_full[2], s_free[2], o_full[2], o_empty[2], st_full[2], st_empty[2];
  uint64_t done;
  uint32_t tmem_base;
  int abort_flag;
};

// Physical tile (page, KV head) of a work item, or tile 0 with DEV_BAD_PAGE raised.
__device__ __forceinline__ int item_tile(const DevPlan& p, const int32_t* page_table,
                                         const FwdTask& t) {
  const int gp = t.bucket / p.Hkv, g = t.bucket % p.Hkv;
  const int req = p.page_req[gp];
  const int pg = gp - p.reqs[req].page_base;
  int phys = __ldg(page_table + (int64_t)req * p.max_pages + pg);
  if (phys < 0 || phys >= p.num_phys) {
    set_status(p.status, DEV_BAD_PAGE);
    phys = 0;
  }
  return phys * p.Hkv + g;
}

// One NVFP4 tile (codes [128][D/2], then scales [128][D/16], in `raw`) into the operand tile
// `dst`: 128 rows of D elements in the 128-byte-swizzled layout TMA writes, as FP16 products
// code x scale (exact) in column blocks of 64 elements (16 KB each), or, with E4M3OUT, as those
// products rounded to E4M3 (one 128-byte block per row; D = 128).  Thread t of nt converts the
// 16-byte code chunks t, t + nt, ... (32 elements each).
template <int D, bool E4M3OUT>
__device__ __forceinline__ void nvfp4_tile_convert(const uint8_t* raw, uint8_t* dst, int t, int nt) {
  constexpr int CPR = D / 32;  // code chunks per row
  const uint8_t* scl = raw + 128 * D / 2;
  for (int c = t; c < 128 * CPR; c += nt) {
    const int row = c / CPR, i = c % CPR;
    const uint4 cw = reinterpret_cast<const uint4*>(raw)[c];
    const uint32_t sb = *reinterpret_cast<const uint16_t*>(scl + row * (D / 16) + 2 * i);
    const uint32_t s0 = cvt_e4m3x2((uint16_t)((sb & 0xffu) * 0x0101u));  // elements 0..15
    const uint32_t s1 = cvt_e4m3x2((uint16_t)((sb >> 8) * 0x0101u));     // elements 16..31
    const uint32_t w[4] = {cw.x, cw.y, cw.z, cw.w};
    uint32_t h[16];  // h[4 j + b]: elements 8 j + 2 b, +1 of the chunk
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int b = 0; b < 4; ++b)
        h[4 * j + b] = hmul2_u32(cvt_e2m1x2((uint16_t)((w[j] >> (8 * b)) & 0xffu)), j < 2 ? s0 : s1);
    if (E4M3OUT) {
      uint32_t e[8];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        e[u] = (uint32_t)cvt_f16x2_e4m3x2(h[2 * u]) | ((uint32_t)cvt_f16x2_e4m3x2(h[2 * u + 1]) << 16);
#pragma unroll
      for (int u = 0; u < 2; ++u)
        *reinterpret_cast<uint4*>(dst + sw128_offset(row, 2 * i + u)) =
            make_uint4(e[4 * u], e[4 * u + 1], e[4 * u + 2], e[4 * u + 3]);
    } else {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int col = 32 * i + 8 * u;
        *reinterpret_cast<uint4*>(dst + (col / 64) * 16384 + sw128_offset(row, (col % 64) / 8)) =
            make_uint4(h[4 * u], h[4 * u + 1], h[4 * u + 2], h[4 * u + 3]);
      }
    }
  }
}

template <int PT>
__device__ __forceinline__ uint32_t pack_partial2(float a, float b) {
  if (PT == kPBF16) {
    __nv_bfloat162 x = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&x);
  } else {
    __half2 x = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&x);
  }
}

// MODE, PT: see above.  For the NVFP4 modes kc/ks/vc/vs are the caches' codes and scales
// (tmK/tmV unused); for BF16 they are unused.
template <int D, int MODE, int PT>
__global__ void __launch_bounds__(kThreads, 1)
forward_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, DevPlan p, const uint8_t* __restrict__ kc, const uint8_t* __restrict__ ks,
               const uint8_t* __restrict__ vc, const uint8_t* __restrict__ vs,
               const int32_t* __restrict__ page_table, void* __restrict__ partial,
               int64_t split_stride, float* __restrict__ lse, int64_t lse_split_stride,
               float q_scale) {
  using Smem = FwdSmem<D, MODE, PT>;
  constexpr bool RAW = Smem::RAW;
  constexpr bool FP8QK = MODE == kModeFP8QK;
  constexpr int kQS = Smem::QS;
  constexpr int DB = D / 64;               // 128-byte column blocks of a 16-bit (V) row
  constexpr int DBQ = D * Smem::QE / 128;  // 128-byte column blocks of a Q / K row
  constexpr int TQK = Smem::TQK, TILE = Smem::TV;
  constexpr int QK_STEPS = D * Smem::QE / 32;  // one MMA per 32 bytes of K depth
  constexpr int PE = Smem::PE;
  constexpr uint32_t IDESC_QK = idesc_mma(MODE == kModeBF16, MODE == kModeBF16, 128, 128, false,
                                          false);
  constexpr uint32_t IDESC_PV = idesc_mma(false, false, 128, D, false, true);
  extern __shared__ uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                      ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  int32_t* status = p.status;
  const int64_t R = (int64_t)p.T * p.H;

  if (tid == 0) {
    mbar_init(smem_u32(&sm.k_full), RAW ? 2 : 1);  // the converter warps, or the TMA bytes
    mbar_init(smem_u32(&sm.k_empty), 1);
    mbar_init(smem_u32(&sm.v_full), 1);
    mbar_init(smem_u32(&sm.v_empty), 1);
    mbar_init(smem_u32(&sm.v_ready), 2);  // the two converter warps
    mbar_init(smem_u32(&sm.kraw_full), 1);
    mbar_init(smem_u32(&sm.kraw_empty), 2);
    mbar_init(smem_u32(&sm.vraw_full), 1);
    mbar_init(smem_u32(&sm.vraw_empty), 2);
    for (int i = 0; i < kQS; ++i) {
      mbar_init(smem_u32(&sm.q_full[i]), 4);  // one arrival per gather warp
      mbar_init(smem_u32(&sm.q_empty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&sm.s_full[i]), 1);
      mbar_init(smem_u32(&sm.p_full[i]), 4);
      mbar_init(smem_u32(&sm.s_free[i]), 1);
      mbar_init(smem_u32(&sm.o_full[i]), 1);
      mbar_init(smem_u32(&sm.o_empty[i]), 4);
      mbar_init(smem_u32(&sm.st_full[i]), 4);
      mbar_init(smem_u32(&sm.st_empty[i]), 4);
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
  // the prologue above may overlap the previous kernel (the inversion); from here on the
  // kernel reads what it wrote
  pdl_wait();
  pdl_trigger();
  const int ntasks = *(volatile int32_t*)(p.counters + 2);
  const uint32_t tmem = sm.tmem_base;  // S[b] at column 128 b, O[b] at 256 + 128 b
  volatile int* abort_flag = &sm.abort_flag;

  // Registers: the block launches with 128 per thread (512 x 128 = 65536); the producer/MMA
  // and gather warpgroups give part of their share to the softmax warpgroup, which holds a
  // whole S row ((96 + 232 + 128 + 56) x 128 = 65536).  Each role's code sits under its own
  // setmaxnreg so the compiler allocates it within that budget.
  if (warp < 4) {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 96;");
  if (warp == 0) {
    // ------------------------------------------------ K/V producer (one lane)
    uint32_t kv_it = 0;
    for (int ti = blockIdx.x; ti < ntasks && lane == 0; ti += gridDim.x) {
      if (*abort_flag) break;
      const int tile = item_tile(p, page_table, p.fwd_tasks[ti]);
      if (!RAW) {
        const int krow = tile * 128;
        // K as soon as the previous item's last S has read the old tile, V after its last P.V
        if (!mbar_wait(smem_u32(&sm.k_empty), (kv_it & 1) ^ 1, abort_flag, status)) break;
        const uint32_t kf = smem_u32(&sm.k_full);
        mbar_expect_tx(kf, TQK);
        for (int db = 0; db < DBQ; ++db)
          tma_load_2d(smem_u32(sm.k) + db * 16384, &tmK, db * (128 / Smem::QE), krow, kf);
        if (!mbar_wait(smem_u32(&sm.v_empty), (kv_it & 1) ^ 1, abort_flag, status)) break;
        const uint32_t vf = smem_u32(&sm.v_full);
        mbar_expect_tx(vf, TILE);
        for (int db = 0; db < DB; ++db)
          tma_load_2d(smem_u32(sm.v) + db * 16384, &tmV, db * 64, krow, vf);
        // items of a group or less (the plan's fwd_prefetch): the next item's tiles into L2
        // while this one runs
        const int tn = ti + p.fwd_prefetch * (int)gridDim.x;
        if (p.fwd_prefetch > 0 && tn < ntasks) {
          const int tile_n = item_tile(p, page_table, p.fwd_tasks[tn]);
          bulk_prefetch_l2(kc + (int64_t)tile_n * TQK, TQK);
          bulk_prefetch_l2(vc + (int64_t)tile_n * TILE, TILE);
        }
      } else {
        // codes and scales of K, then of V, one item ahead of the conversion
        if (!mbar_wait(smem_u32(&sm.kraw_empty), (kv_it & 1) ^ 1, abort_flag, status)) break;
        uint32_t f = smem_u32(&sm.kraw_full);
        mbar_expect_tx(f, Smem::RC + Smem::RSC);
        bulk_load(smem_u32(sm.kraw), kc + (int64_t)tile * Smem::RC, Smem::RC, f);
        bulk_load(smem_u32(sm.kraw) + Smem::RC, ks + (int64_t)tile * Smem::RSC, Smem::RSC, f);
        if (!mbar_wait(smem_u32(&sm.vraw_empty), (kv_it & 1) ^ 1, abort_flag, status)) break;
        f = smem_u32(&sm.vraw_full);
        mbar_expect_tx(f, Smem::RC + Smem::RSC);
        bulk_load(smem_u32(sm.vraw), vc + (int64_t)tile * Smem::RC, Smem::RC, f);
        bulk_load(smem_u32(sm.vraw) + Smem::RC, vs + (int64_t)tile * Smem::RSC, Smem::RSC, f);
      }
      ++kv_it;
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer (one thread)
    // Two streams: S(g) = Q K^T into S[g & 1] once Q(g) has landed, and P.V(g) into O[g & 1]
    // once the softmax has written P(g).  The thread polls both and issues whichever is ready
    // (P.V first), so a late Q tile never holds back the P.V and epilogue of earlier groups.
    if (lane == 0) {
      // S cursor (task ti_s, group grp_s) and P.V cursor (ti_p, grp_p); gs / gp count groups
      int ti_s = blockIdx.x, grp_s = 0, ti_p = blockIdx.x, grp_p = 0;
      auto ngroups_of = [&](int ti) { return ti < ntasks ? (p.fwd_tasks[ti].count + 127) / 128 : 0; };
      int ng_s = ngroups_of(ti_s);
      int ng_p = ng_s;
      // group counts of the following items, loaded ahead of the item switch
      int ng_s_next = ngroups_of(ti_s + gridDim.x), ng_p_next = ng_s_next;
      uint32_t gs = 0, gp = 0, q_it = 0, kv_s = 0, kv_p = 0;
      uint64_t t_last = globaltimer_ns();
      uint32_t spins = 0;
      while (ti_p < ntasks) {
        bool progressed = false;
        if (gp < gs) {  // P.V(gp)
          const int b = gp & 1;
          const uint32_t ph = (gp >> 1) & 1;
          if (mbar_try_wait(smem_u32(&sm.p_full[b]), ph) &&
              mbar_try_wait(smem_u32(&sm.o_empty[b]), ph ^ 1) &&
              (grp_p != 0 || mbar_try_wait(smem_u32(&sm.v_ready), kv_p & 1))) {
            tc_fence_after();
            const uint32_t vb = smem_u32(sm.v);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)  // 128 keys, K = 16 per step
              mma_f16_ts(tmem + 256 + b * 128, tmem + b * 128 + kk * 8,
                         sdesc_sw128(vb + kk * 2048, 16384, 1024), IDESC_PV, kk > 0);
            mma_commit(smem_u32(&sm.s_free[b]));
            mma_commit(smem_u32(&sm.o_full[b]));
            ++gp;
            if (++grp_p == ng_p) {  // the item's last P.V: its V tile may be replaced
              mma_commit(smem_u32(&sm.v_empty));
              ++kv_p;
              grp_p = 0;
              ti_p += gridDim.x;
              ng_p = ng_p_next;
              ng_p_next = ngroups_of(ti_p + gridDim.x);
            }
            progressed = true;
          }
        }
        if (ti_s < ntasks && gs < gp + 2) {  // S(gs)
          const int qs = q_it % kQS;
          const int b = gs & 1;
          if ((grp_s != 0 || mbar_try_wait(smem_u32(&sm.k_full), kv_s & 1)) &&
              mbar_try_wait(smem_u32(&sm.q_full[qs]), (q_it / kQS) & 1) &&
              mbar_try_wait(smem_u32(&sm.s_free[b]), ((gs >> 1) & 1) ^ 1)) {
            tc_fence_after();
            const uint32_t qb = smem_u32(sm.q[qs]), kb = smem_u32(sm.k);
#pragma unroll
            for (int kk = 0; kk < QK_STEPS; ++kk) {
              const uint32_t off = (kk / 4) * 16384 + (kk % 4) * 32;
              if (FP8QK)
                mma_f8_ss(tmem + b * 128, sdesc_sw128(qb + off, 16, 1024),
                          sdesc_sw128(kb + off, 16, 1024), IDESC_QK, kk > 0);
              else
                mma_f16_ss(tmem + b * 128, sdesc_sw128(qb + off, 16, 1024),
                           sdesc_sw128(kb + off, 16, 1024), IDESC_QK, kk > 0);
            }
            mma_commit(smem_u32(&sm.s_full[b]));
            mma_commit(smem_u32(&sm.q_empty[qs]));
            ++q_it;
            ++gs;
            if (++grp_s == ng_s) {  // the item's last S: its K tile may be replaced
              mma_commit(smem_u32(&sm.k_empty));
              ++kv_s;
              grp_s = 0;
              ti_s += gridDim.x;
              ng_s = ng_s_next;
              ng_s_next = ngroups_of(ti_s + gridDim.x);
            }
            progressed = true;
          }
        }
        if (progressed) {
          spins = 0;
          t_last = globaltimer_ns();
        } else if ((++spins & 63u) == 0) {
          if (*abort_flag) break;
          if (globaltimer_ns() - t_last > kWaitLimitNs) {
            set_status(status, DEV_TIMEOUT);
            *abort_flag = 1;
            break;
          }
        }
      }
      mma_commit(smem_u32(&sm.done));
      mbar_wait(smem_u32(&sm.done), 0, nullptr, status);
    }
  } else {
    // ------------------------------------------------ loader conversions: warps 2, 3
    const int ct = (warp - 2) * 32 + lane;
    uint32_t kv_it = 0;
    for (int ti = blockIdx.x; ti < ntasks; ti += gridDim.x) {
      const uint32_t ph = kv_it & 1;
      if (!RAW) {
        // BF16 V -> FP16 in place
        if (!mbar_wait(smem_u32(&sm.v_full), ph, abort_flag, status)) break;
        uint4* v4 = reinterpret_cast<uint4*>(sm.v);
        for (int i = ct; i < TILE / 16; i += 64) {
          uint4 x = v4[i];
          uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float lo = __uint_as_float(w[j] << 16);
            const float hi = __uint_as_float(w[j] & 0xffff0000u);
            __half2 h2 = __floats2half2_rn(lo, hi);
            w[j] = *reinterpret_cast<uint32_t*>(&h2);
          }
          v4[i] = make_uint4(w[0], w[1], w[2], w[3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sm.v_ready));
      } else {
        // NVFP4 K once the previous item's last S is done, then V after its last P.V
        if (!mbar_wait(smem_u32(&sm.kraw_full), ph, abort_flag, status) ||
            !mbar_wait(smem_u32(&sm.k_empty), ph ^ 1, abort_flag, status))
          break;
        nvfp4_tile_convert<D, FP8QK>(sm.kraw, sm.k, ct, 64);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(smem_u32(&sm.k_full));
          mbar_arrive(smem_u32(&sm.kraw_empty));
        }
        if (!mbar_wait(smem_u32(&sm.vraw_full), ph, abort_flag, status) ||
            !mbar_wait(smem_u32(&sm.v_empty), ph ^ 1, abort_flag, status))
          break;
        nvfp4_tile_convert<D, false>(sm.vraw, sm.v, ct, 64);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(smem_u32(&sm.v_ready));
          mbar_arrive(smem_u32(&sm.vraw_empty));
        }
      }
      ++kv_it;
    }
  }
  } else if (warp < 8) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 232;");
    // ------------------------------------------------ softmax: warps 4..7
    const int quarter = warp % 4;
    const int row = quarter * 32 + lane;
    const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
    const float c = p.sm_scale * q_scale * 1.4426950408889634f;  // scale * log2(e)
    uint32_t g_it = 0;
    for (int ti = blockIdx.x; ti < ntasks; ti += gridDim.x) {
      const FwdTask t = p.fwd_tasks[ti];
      const int gp = t.bucket / p.Hkv;
      const int pg = gp - p.reqs[p.page_req[gp]].page_base;
      const int ngroups = (t.count + 127) / 128;
      bool ok = true;
      // this thread's entry of group g+1 is loaded while group g is processed
      int2 nxt = row < t.count ? __ldg(&p.entries[t.entry_begin + row]) : make_int2(-1, 0);
      for (int grp = 0; grp < ngroups; ++grp) {
        const int b = g_it & 1;
        const uint32_t ph = (g_it >> 1) & 1;
        int2 rs = nxt;
        {
          const int ei = (grp + 1) * 128 + row;
          if (grp + 1 < ngroups) nxt = ei < t.count ? __ldg(&p.entries[t.entry_begin + ei]) : make_int2(-1, 0);
        }
        int tpos = rs.y >> 6;
        rs.y &= 63;
        if (rs.x < 0 || rs.x >= R || rs.y >= p.K) rs = make_int2(-1, -1);
        const bool live = rs.x >= 0;
        const bool own = live && (tpos >> 7) == pg;
        const int nvis = own ? (tpos & 127) + 1 : 128;
        if (!mbar_wait(smem_u32(&sm.s_full[b]), ph, abort_flag, status)) { ok = false; break; }
        tc_fence_after();
        const uint32_t sbase = tmem + lane_addr + b * 128;
        const bool masked = __any_sync(0xffffffffu, own);
        // the whole S row in one pass: four loads in flight, one wait
        uint32_t v[4][32];
        float red[4];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) red[cc] = tmem_ld32_max(sbase + cc * 32, v[cc]);
        tmem_ld_wait();
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          reg_fence(v[cc]);
          reg_fence1(red[cc]);
        }
        float m;
        if (masked) {
          m = -INFINITY;
#pragma unroll
          for (int cc = 0; cc < 4; ++cc)
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (cc * 32 + j < nvis) m = fmaxf(m, __uint_as_float(v[cc][j]));
        } else {
          m = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
        }
        if (!live) m = 0.f;
        const float mc = m * c;
        // p = 2^(s c - m c) as FP16 pairs written over the S columns, l = sum p (four
        // independent partial sums)
        float lsum[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t pk[16];
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            float p0 = fast_exp2(fmaf(__uint_as_float(v[cc][j]), c, -mc));
            float p1 = fast_exp2(fmaf(__uint_as_float(v[cc][j + 1]), c, -mc));
            if (masked) {
              if (cc * 32 + j >= nvis) p0 = 0.f;
              if (cc * 32 + j + 1 >= nvis) p1 = 0.f;
            }
            lsum[(j >> 1) & 3] += p0 + p1;
            __half2 h2 = __floats2half2_rn(p0, p1);
            pk[j / 2] = *reinterpret_cast<uint32_t*>(&h2);
          }
          tmem_st16(sbase + cc * 16, pk);
        }
        const float l = (lsum[0] + lsum[1]) + (lsum[2] + lsum[3]);
        tmem_st_wait();
        // row statistics for the epilogue; LSE straight to global
        if (!mbar_wait(smem_u32(&sm.st_empty[b]), ph ^ 1, abort_flag, status)) { ok = false; break; }
        sm.inv_l[b][row] = 1.f / l;
        sm.rs[b][row] = rs;
        if (live) lse[rs.y * lse_split_stride + rs.x] = (mc + log2f(l)) * 0.6931471805599453f;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(smem_u32(&sm.p_full[b]));
          mbar_arrive(smem_u32(&sm.st_full[b]));
        }
        ++g_it;
      }
      if (!ok) break;
    }
  } else if (warp < 12) {
    // ------------------------------------------------ epilogue: warps 8..11
    const int quarter = warp % 4;
    const int row = quarter * 32 + lane;
    const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
    const uint64_t pol_out = l2_policy_evict_first();  // partials are read once, by the combine
    uint32_t g_it = 0;
    bool ok = true;
    // A thread per row: O / l from TMEM into its padded staging row (FP32, or 16-bit rounded
    // to nearest even), then one bulk copy of the whole row (D x 4 or D x 2 bytes) into
    // partial[slot][row].  The stores run on the TMA engine and leave the load/store unit to
    // the Q gather.
    uint8_t* srow = sm.ep[0] + row * Smem::EPR;
    for (int ti = blockIdx.x; ti < ntasks && ok; ti += gridDim.x) {
      const FwdTask t = p.fwd_tasks[ti];
      const int ngroups = (t.count + 127) / 128;
      for (int grp = 0; grp < ngroups; ++grp, ++g_it) {
        const int b = g_it & 1;
        const uint32_t ph = (g_it >> 1) & 1;
        if (!mbar_wait(smem_u32(&sm.o_full[b]), ph, abort_flag, status) ||
            !mbar_wait(smem_u32(&sm.st_full[b]), ph, abort_flag, status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float inv = sm.inv_l[b][row];
        const int2 rs = sm.rs[b][row];
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sm.st_empty[b]));
        const uint32_t obase = tmem + lane_addr + 256 + b * 128;
        bulk_wait_read<0>();  // this row's previous store has finished reading the staging row
#pragma unroll
        for (int hh = 0; hh < D / 64; ++hh) {
          uint32_t v[2][32];
          tmem_ld32(obase + hh * 64, v[0]);
          tmem_ld32(obase + hh * 64 + 32, v[1]);
          tmem_ld_wait();
          reg_fence(v[0]);
          reg_fence(v[1]);
          if (hh == D / 64 - 1) {  // O[b] fully read: hand the accumulator back to the MMA
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&sm.o_empty[b]));
          }
          if (PT != kPF32) {
#pragma unroll
            for (int cc = 0; cc < 2; ++cc)
#pragma unroll
              for (int j = 0; j < 32; j += 8) {
                uint32_t w[4];
#pragma unroll
                for (int u = 0; u < 4; ++u)
                  w[u] = pack_partial2<PT>(__uint_as_float(v[cc][j + 2 * u]) * inv,
                                           __uint_as_float(v[cc][j + 2 * u + 1]) * inv);
                *reinterpret_cast<uint4*>(srow + (hh * 64 + cc * 32 + j) * 2) =
                    make_uint4(w[0], w[1], w[2], w[3]);
              }
          } else {
#pragma unroll
            for (int cc = 0; cc < 2; ++cc)
#pragma unroll
              for (int j = 0; j < 32; j += 4)
                *reinterpret_cast<float4*>(srow + (hh * 64 + cc * 32 + j) * 4) = make_float4(
                    __uint_as_float(v[cc][j]) * inv, __uint_as_float(v[cc][j + 1]) * inv,
                    __uint_as_float(v[cc][j + 2]) * inv, __uint_as_float(v[cc][j + 3]) * inv);
          }
        }
        fence_proxy_async_smem();
        if (rs.x >= 0)
          bulk_store_hint(static_cast<uint8_t*>(partial) +
                              ((int64_t)rs.y * split_stride + (int64_t)rs.x * D) * PE,
                          smem_u32(srow), D * PE, pol_out);
        bulk_commit();
      }
    }
    bulk_wait_all<0>();
  } else {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 56;");
    // ------------------------------------------------ Q gather (TMA tile::gather4): warps 12..15
    // A group's 32 DBQ gather4 operations (4 rows x one 128-byte column block each) are spread
    // over the four warps, one per SM sub-partition: lane l < 8 DBQ of warp w issues operation
    // op = 8 DBQ w + l, column block op / 32, group rows 4 (op % 32) .. +3 (rows past the end of
    // the group repeat its first row).  The indices of group g+1 are fetched while g is issued.
    // (The SM's TMA engine carries these gathers and the epilogue's bulk stores; cp.async
    // copies of the load/store unit were measured slower here, alone or sharing the rows.)
    const int nops = 8 * DBQ;
    const int op = (warp - 12) * nops + lane;
    const int db = op / 32, quad = op % 32;
    const bool active = lane < nops;
    const uint64_t pol_q = l2_policy_evict_last();  // Q rows are re-read once per page
    uint32_t q_it = 0;
    bool ok = true;
    auto fetch_rows = [&](const FwdTask& tk, int grp, int (&rows)[4]) {
      const int base = tk.entry_begin + grp * 128;
      const int n_in = min(128, tk.count - grp * 128);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int i = 4 * quad + j;
        rows[j] = active ? __ldg(&p.entries[base + (i < n_in ? i : 0)].x) : 0;
      }
    };
    // groups of this CTA's items in order; the row indices (and, across an item boundary, the
    // next item's descriptor) of group n+1 are loaded while group n is issued
    int ti = blockIdx.x, grp = 0;
    FwdTask t;
    int nxt[4];
    if (ti < ntasks) {
      t = p.fwd_tasks[ti];
      fetch_rows(t, 0, nxt);
    }
    while (ti < ntasks && ok) {
      int rows[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        rows[j] = nxt[j];
        if (rows[j] < 0 || rows[j] >= R) {
          set_status(status, DEV_OVERFLOW);
          rows[j] = 0;
        }
      }
      int ti2 = ti, grp2 = grp + 1;
      FwdTask t2 = t;
      if (grp2 * 128 >= t.count) {
        ti2 = ti + gridDim.x;
        grp2 = 0;
        if (ti2 < ntasks) t2 = p.fwd_tasks[ti2];
      }
      if (ti2 < ntasks) fetch_rows(t2, grp2, nxt);
      const int qs = q_it % kQS;
      const uint32_t qf = smem_u32(&sm.q_full[qs]);
      if (lane == 0) {
        ok = mbar_wait(smem_u32(&sm.q_empty[qs]), ((q_it / kQS) & 1) ^ 1, abort_flag, status);
        if (ok) mbar_expect_tx(qf, TQK / 4);
      }
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      if (active)
        tma_gather4_hint(smem_u32(sm.q[qs]) + db * 16384 + quad * 512, &tmQ,
                         db * (128 / Smem::QE), rows[0], rows[1], rows[2], rows[3], qf, pol_q);
      ++q_it;
      ti = ti2;
      grp = grp2;
      t = t2;
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

// Launch of one instantiation.  q: the Q the tensor cores read (BF16, FP16 or E4M3 bytes);
// kc/vc: BF16 caches, or NVFP4 codes with their scales ks/vs.
template <int D, int MODE, int PT>
cudaError_t run_forward(const DevPlan& p, const void* q, const void* kc, const void* vc,
                        const void* ks, const void* vs, const int32_t* page_table, void* partial,
                        int64_t split_stride, float* lse, int64_t lse_split_stride, float q_scale,
                        cudaStream_t st) {
  alignas(64) CUtensorMap tmQ, tmK, tmV;
  memset(&tmK, 0, sizeof tmK);
  memset(&tmV, 0, sizeof tmV);
  const uint64_t R = (uint64_t)p.T * p.H;
  const uint64_t kv_rows = (uint64_t)p.num_phys * p.Hkv * 128;
  // tensor-map element types: BF16 (0), FP16 (1) or bytes (2); Q and K rows of 128 bytes
  const int dq = MODE == kModeBF16 ? 0 : (MODE == kModeF16 ? 1 : 2);
  const uint64_t qe = MODE == kModeFP8QK ? 1 : 2;
  const uint32_t box_q = (uint32_t)(128 / qe);
  if (!encode_tmap_2d(&tmQ, dq, const_cast<void*>(q), D, R, (uint64_t)D * qe, box_q, 1, true))
    return cudaErrorInvalidValue;
  if (MODE == kModeBF16 &&
      (!encode_tmap_2d(&tmK, 0, const_cast<void*>(kc), D, kv_rows, (uint64_t)D * 2, 64, 128, true) ||
       !encode_tmap_2d(&tmV, 0, const_cast<void*>(vc), D, kv_rows, (uint64_t)D * 2, 64, 128, true)))
    return cudaErrorInvalidValue;
  const int smem = (int)sizeof(FwdSmem<D, MODE, PT>) + 1024;
  auto kern = forward_kernel<D, MODE, PT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  e = launch_pdl(kern, dim3(num_sms()), dim3(kThreads), smem, st, tmQ, tmK, tmV, p,
                 static_cast<const uint8_t*>(kc), static_cast<const uint8_t*>(ks),
                 static_cast<const uint8_t*>(vc), static_cast<const uint8_t*>(vs), page_table,
                 partial, split_stride, lse, lse_split_stride, q_scale);
  return e != cudaSuccess ? e : cudaGetLastError();
}

// The forward for a plan's dtypes: BF16 Q/K/V, or E4M3 Q (an exact FP16 copy in the
// workspace, the per-tensor scale kept in the softmax exponent) with NVFP4 K/V dequantised in
// the loader; fp8qk: the pages' Q8KV4 route (E4M3 Q as given, K rounded to E4M3).
template <int PT>
cudaError_t launch_forward_pt(const DevPlan& p, sps_dtype qt, sps_dtype kvt, const void* q,
                              float q_scale, const void* kc, const void* vc, const void* ks,
                              const void* vs, const int32_t* page_table, void* partial,
                              int64_t split_stride, float* lse, int64_t lse_split_stride,
                              bool fp8qk, cudaStream_t st) {
  if (fp8qk) {
    if (qt != SPS_E4M3 || kvt != SPS_NVFP4 || p.D != 128) return cudaErrorNotSupported;
    return run_forward<128, kModeFP8QK, PT>(p, q, kc, vc, ks, vs, page_table, partial,
                                            split_stride, lse, lse_split_stride, q_scale, st);
  }
  if (qt == SPS_BF16 && kvt == SPS_BF16) {
    if (p.D == 128)
      return run_forward<128, kModeBF16, PT>(p, q, kc, vc, nullptr, nullptr, page_table, partial,
                                             split_stride, lse, lse_split_stride, q_scale, st);
    return run_forward<64, kModeBF16, PT>(p, q, kc, vc, nullptr, nullptr, page_table, partial,
                                          split_stride, lse, lse_split_stride, q_scale, st);
  }
  if (qt == SPS_E4M3 && kvt == SPS_NVFP4) {
    if (!p.qconv) return cudaErrorInvalidValue;
    cudaError_t e = launch_dequant(SPS_E4M3, q, nullptr, (int64_t)p.T * p.H * p.D, p.qconv, st);
    if (e != cudaSuccess) return e;
    if (p.D == 128)
      return run_forward<128, kModeF16, PT>(p, p.qconv, kc, vc, ks, vs, page_table, partial,
                                            split_stride, lse, lse_split_stride, q_scale, st);
    return run_forward<64, kModeF16, PT>(p, p.qconv, kc, vc, ks, vs, page_table, partial,
                                         split_stride, lse, lse_split_stride, q_scale, st);
  }
  return cudaErrorNotSupported;
}

}  // namespace fwd
}  // namespace sps
