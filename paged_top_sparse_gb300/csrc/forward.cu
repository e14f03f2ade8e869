// forward.cu -- page-parallel sparse forward ("MSA PR 21: Q8KV4 paged sparse prefill", K1):
// one work item per (page, KV head, query split), the rows that selected the page streamed
// through in groups of 128; every (row, page) pair yields a partial output normalised by its
// row sum plus the LSE, written into the split-strided FP32 partial buffer at the row's slot.
// Only the row's own page is causally masked; K/V come through the page table.
//
// Design (GB300, one CTA per SM, persistent over the device-built work list):
//   warp 0     TMA producer: the K and V tiles of the item's physical page (128-byte swizzle),
//              then per group the 128 query rows, gathered four at a time (tile::gather4)
//              into a 2-stage Q ring;
//   warp 1     MMA issuer (one thread): S = Q K^T (shared x shared, N = 128 keys) into a
//              double-buffered TMEM accumulator, and O = P V with P read from TMEM (the
//              softmax overwrites S with P in place) and V as an MN-major FP16 operand;
//              S of group g+1 is issued before P.V of group g so softmax and MMA overlap;
//   warps 2-5  softmax, a thread per row: converts the V tile BF16 -> FP16 in place once per
//              item; per group, the row max (tcgen05.ld.red.max unless some lane of the warp
//              owns the page, then the masked element-wise path), p = 2^(s c - m c) rounded
//              to FP16 into TMEM, l = sum p, LSE = m * scale + ln l straight to global;
//   warps 6-9  epilogue, a thread per row: O / l from TMEM in 64-column halves into a padded
//              staging buffer, then one 256-byte bulk store per row and half into
//              partial[slot][row] (double-buffered staging, stores drain asynchronously).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx.cuh"
#include "sps_internal.h"

namespace sps {
namespace {

constexpr int kQS = 2;          // Q ring stages
constexpr int kThreads = 320;   // 10 warps
constexpr int kStagePitch = 68; // floats per staging row (64 + 4 pad: conflict-free writes)

template <int D>
struct FwdSmem {
  static constexpr int TILE = 128 * D * 2;  // 128 rows of D 16-bit elements
  uint8_t k[TILE];
  uint8_t v[TILE];
  uint8_t q[kQS][TILE];
  float stage[2][128 * kStagePitch];
  float inv_l[2][128];
  int2 rs[2][128];
  uint64_t kv_full, kv_empty, v_ready;
  uint64_t q_full[kQS], q_empty[kQS];
  uint64_t s_full[2], p_full[2], s_free[2], o_full[2], o_empty[2], st_full[2], st_empty[2];
  uint64_t done;
  uint32_t tmem_base;
  int abort_flag;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
forward_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, DevPlan p,
               const int32_t* __restrict__ page_table, float* __restrict__ partial,
               int64_t split_stride, float* __restrict__ lse, int64_t lse_split_stride,
               float q_scale) {
  using Smem = FwdSmem<D>;
  constexpr int DB = D / 64;          // 128-byte column blocks of a 16-bit row
  constexpr int TILE = Smem::TILE;
  constexpr int QK_STEPS = D / 16;
  constexpr uint32_t IDESC_QK = idesc_mma(true, true, 128, 128, false, false);
  constexpr uint32_t IDESC_PV = idesc_mma(false, false, 128, D, false, true);
  extern __shared__ uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                      ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  int32_t* status = p.status;
  const int ntasks = *(volatile int32_t*)(p.counters + 2);
  const int64_t R = (int64_t)p.T * p.H;

  if (tid == 0) {
    mbar_init(smem_u32(&sm.kv_full), 1);
    mbar_init(smem_u32(&sm.kv_empty), 1);
    mbar_init(smem_u32(&sm.v_ready), 4);
    for (int i = 0; i < kQS; ++i) {
      mbar_init(smem_u32(&sm.q_full[i]), 1);
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
  const uint32_t tmem = sm.tmem_base;  // S[b] at column 128 b, O[b] at 256 + 128 b
  volatile int* abort_flag = &sm.abort_flag;

  if (warp == 0) {
    // ------------------------------------------------ TMA producer (whole warp)
    uint32_t kv_it = 0, q_it = 0;
    for (int ti = blockIdx.x; ti < ntasks; ti += gridDim.x) {
      if (*abort_flag) break;
      const FwdTask t = p.fwd_tasks[ti];
      const int gp = t.bucket / p.Hkv, g = t.bucket % p.Hkv;
      const int req = p.page_req[gp];
      const int pg = gp - p.reqs[req].page_base;
      bool ok = true;
      if (lane == 0) {
        ok = mbar_wait(smem_u32(&sm.kv_empty), (kv_it & 1) ^ 1, abort_flag, status);
        if (ok) {
          int phys = __ldg(page_table + (int64_t)req * p.max_pages + pg);
          if (phys < 0 || phys >= p.num_phys) {
            set_status(status, DEV_BAD_PAGE);
            phys = 0;
          }
          const uint32_t f = smem_u32(&sm.kv_full);
          mbar_expect_tx(f, 2 * TILE);
          const int krow = (phys * p.Hkv + g) * 128;
          for (int db = 0; db < DB; ++db) {
            tma_load_2d(smem_u32(sm.k) + db * 16384, &tmK, db * 64, krow, f);
            tma_load_2d(smem_u32(sm.v) + db * 16384, &tmV, db * 64, krow, f);
          }
        }
      }
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      ++kv_it;
      const int ngroups = (t.count + 127) / 128;
      for (int grp = 0; grp < ngroups; ++grp) {
        const int qs = q_it % kQS;
        if (lane == 0) {
          ok = mbar_wait(smem_u32(&sm.q_empty[qs]), ((q_it / kQS) & 1) ^ 1, abort_flag, status);
          if (ok) mbar_expect_tx(smem_u32(&sm.q_full[qs]), TILE);
        }
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
        // lane l gathers group rows 4l .. 4l+3; rows past the end repeat the first row
        const int base = t.entry_begin + grp * 128;
        const int n_in = min(128, t.count - grp * 128);
        int rows[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int i = 4 * lane + j;
          int r = p.entries[base + (i < n_in ? i : 0)].x;
          if (r < 0 || r >= R) {
            set_status(status, DEV_OVERFLOW);
            r = 0;
          }
          rows[j] = r;
        }
        const uint32_t qf = smem_u32(&sm.q_full[qs]);
        for (int db = 0; db < DB; ++db)
          tma_gather4(smem_u32(sm.q[qs]) + db * 16384 + lane * 512, &tmQ, db * 64, rows[0],
                      rows[1], rows[2], rows[3], qf);
        ++q_it;
      }
      if (!ok) break;
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t kv_it = 0, q_it = 0, g_issue = 0, g_pv = 0;
      bool ok = true;
      // S = Q K^T for global group index gi into S[gi & 1]
      auto issue_s = [&](uint32_t gi) -> bool {
        const int qs = q_it % kQS;
        const int b = gi & 1;
        if (!mbar_wait(smem_u32(&sm.q_full[qs]), (q_it / kQS) & 1, abort_flag, status)) return false;
        if (!mbar_wait(smem_u32(&sm.s_free[b]), ((gi >> 1) & 1) ^ 1, abort_flag, status)) return false;
        tc_fence_after();
        const uint32_t qb = smem_u32(sm.q[qs]), kb = smem_u32(sm.k);
#pragma unroll
        for (int kk = 0; kk < QK_STEPS; ++kk) {
          const uint32_t off = (kk / 4) * 16384 + (kk % 4) * 32;
          mma_f16_ss(tmem + b * 128, sdesc_sw128(qb + off, 16, 1024),
                     sdesc_sw128(kb + off, 16, 1024), IDESC_QK, kk > 0);
        }
        mma_commit(smem_u32(&sm.s_full[b]));
        mma_commit(smem_u32(&sm.q_empty[qs]));
        ++q_it;
        return true;
      };
      for (int ti = blockIdx.x; ti < ntasks && ok; ti += gridDim.x) {
        const FwdTask t = p.fwd_tasks[ti];
        const int ngroups = (t.count + 127) / 128;
        if (!mbar_wait(smem_u32(&sm.kv_full), kv_it & 1, abort_flag, status)) break;
        ok = issue_s(g_issue++);
        for (int grp = 0; grp < ngroups && ok; ++grp) {
          if (grp + 1 < ngroups) ok = issue_s(g_issue++);
          if (!ok) break;
          const int b = g_pv & 1;
          const uint32_t ph = (g_pv >> 1) & 1;
          if (!mbar_wait(smem_u32(&sm.p_full[b]), ph, abort_flag, status) ||
              (grp == 0 && !mbar_wait(smem_u32(&sm.v_ready), kv_it & 1, abort_flag, status)) ||
              !mbar_wait(smem_u32(&sm.o_empty[b]), ph ^ 1, abort_flag, status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t vb = smem_u32(sm.v);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)  // 128 keys, K = 16 per step
            mma_f16_ts(tmem + 256 + b * 128, tmem + b * 128 + kk * 8,
                       sdesc_sw128(vb + kk * 2048, 16384, 1024), IDESC_PV, kk > 0);
          mma_commit(smem_u32(&sm.s_free[b]));
          mma_commit(smem_u32(&sm.o_full[b]));
          ++g_pv;
        }
        mma_commit(smem_u32(&sm.kv_empty));
        ++kv_it;
      }
      mma_commit(smem_u32(&sm.done));
      mbar_wait(smem_u32(&sm.done), 0, nullptr, status);
    }
  } else if (warp < 6) {
    // ------------------------------------------------ softmax: warps 2..5
    const int quarter = warp % 4;
    const int row = quarter * 32 + lane;
    const int sm_tid = (warp - 2) * 32 + lane;
    const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
    const float c = p.sm_scale * q_scale * 1.4426950408889634f;  // scale * log2(e)
    uint32_t kv_it = 0, g_it = 0;
    for (int ti = blockIdx.x; ti < ntasks; ti += gridDim.x) {
      const FwdTask t = p.fwd_tasks[ti];
      const int gp = t.bucket / p.Hkv;
      const int pg = gp - p.reqs[p.page_req[gp]].page_base;
      // V tile: BF16 -> FP16 in place (same swizzled positions)
      if (!mbar_wait(smem_u32(&sm.kv_full), kv_it & 1, abort_flag, status)) break;
      {
        uint4* v4 = reinterpret_cast<uint4*>(sm.v);
        for (int i = sm_tid; i < TILE / 16; i += 128) {
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
      }
      ++kv_it;
      const int ngroups = (t.count + 127) / 128;
      bool ok = true;
      for (int grp = 0; grp < ngroups; ++grp) {
        const int b = g_it & 1;
        const uint32_t ph = (g_it >> 1) & 1;
        const int ei = grp * 128 + row;
        const bool valid = ei < t.count;
        int2 rs = make_int2(-1, -1);
        int tpos = 0;
        if (valid) {
          rs = p.entries[t.entry_begin + ei];
          if (rs.x < 0 || rs.x >= R || rs.y < 0 || rs.y >= p.K) rs = make_int2(-1, -1);
          else tpos = __ldg(p.tok_pos + rs.x / p.H);
        }
        const bool live = rs.x >= 0;
        const bool own = live && (tpos >> 7) == pg;
        const int nvis = own ? (tpos & 127) + 1 : 128;
        if (!mbar_wait(smem_u32(&sm.s_full[b]), ph, abort_flag, status)) { ok = false; break; }
        tc_fence_after();
        const uint32_t sbase = tmem + lane_addr + b * 128;
        const bool masked = __any_sync(0xffffffffu, own);
        // pass 1: raw row max
        float m = -INFINITY;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t v[32];
          if (masked) {
            tmem_ld32(sbase + cc * 32, v);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (cc * 32 + j < nvis) m = fmaxf(m, __uint_as_float(v[j]));
          } else {
            const float red = tmem_ld32_max(sbase + cc * 32, v);
            tmem_ld_wait();
            m = fmaxf(m, red);
          }
        }
        if (!live) m = 0.f;
        const float mc = m * c;
        // pass 2: p = 2^(s c - m c) as FP16 pairs over the S columns, l = sum p
        float l = 0.f;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t v[32], pk[16];
          tmem_ld32(sbase + cc * 32, v);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            float p0 = fast_exp2(fmaf(__uint_as_float(v[j]), c, -mc));
            float p1 = fast_exp2(fmaf(__uint_as_float(v[j + 1]), c, -mc));
            if (masked) {
              if (cc * 32 + j >= nvis) p0 = 0.f;
              if (cc * 32 + j + 1 >= nvis) p1 = 0.f;
            }
            l += p0 + p1;
            __half2 h2 = __floats2half2_rn(p0, p1);
            pk[j / 2] = *reinterpret_cast<uint32_t*>(&h2);
          }
          tmem_st16(sbase + cc * 16, pk);
        }
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
  } else {
    // ------------------------------------------------ epilogue: warps 6..9
    const int quarter = warp % 4;
    const int row = quarter * 32 + lane;
    const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
    uint32_t g_it = 0, st_it = 0;
    bool ok = true;
    for (int ti = blockIdx.x; ti < ntasks && ok; ti += gridDim.x) {
      const FwdTask t = p.fwd_tasks[ti];
      const int ngroups = (t.count + 127) / 128;
      for (int grp = 0; grp < ngroups; ++grp) {
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
        const uint32_t obase = tmem + lane_addr + 256 + b * 128;
#pragma unroll
        for (int hh = 0; hh < DB; ++hh) {
          const int sb = st_it & 1;
          bulk_wait_read<1>();  // this thread's store from staging[sb] two halves ago is done
          float* srow = sm.stage[sb] + row * kStagePitch;
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            uint32_t v[32];
            tmem_ld32(obase + hh * 64 + cc * 32, v);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; j += 4)
              *reinterpret_cast<float4*>(srow + cc * 32 + j) =
                  make_float4(__uint_as_float(v[j]) * inv, __uint_as_float(v[j + 1]) * inv,
                              __uint_as_float(v[j + 2]) * inv, __uint_as_float(v[j + 3]) * inv);
          }
          fence_proxy_async_smem();
          if (rs.x >= 0)
            bulk_store(partial + (int64_t)rs.y * split_stride + (int64_t)rs.x * D + hh * 64,
                       smem_u32(srow), 256);
          bulk_commit();
          ++st_it;
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(smem_u32(&sm.o_empty[b]));
          mbar_arrive(smem_u32(&sm.st_empty[b]));
        }
        ++g_it;
      }
    }
    bulk_wait_all<0>();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D>
cudaError_t run_forward(const DevPlan& p, const void* q, const void* kc, const void* vc,
                        const int32_t* page_table, float* partial, int64_t split_stride,
                        float* lse, int64_t lse_split_stride, float q_scale, cudaStream_t st) {
  alignas(64) CUtensorMap tmQ, tmK, tmV;
  const uint64_t R = (uint64_t)p.T * p.H;
  const uint64_t kv_rows = (uint64_t)p.num_phys * p.Hkv * 128;
  if (!encode_tmap_2d(&tmQ, 0, const_cast<void*>(q), D, R, (uint64_t)D * 2, 64, 1, true) ||
      !encode_tmap_2d(&tmK, 0, const_cast<void*>(kc), D, kv_rows, (uint64_t)D * 2, 64, 128, true) ||
      !encode_tmap_2d(&tmV, 0, const_cast<void*>(vc), D, kv_rows, (uint64_t)D * 2, 64, 128, true))
    return cudaErrorInvalidValue;
  const int smem = (int)sizeof(FwdSmem<D>) + 1024;
  auto kern = forward_kernel<D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<num_sms(), kThreads, smem, st>>>(tmQ, tmK, tmV, p, page_table, partial, split_stride,
                                          lse, lse_split_stride, q_scale);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_forward(const DevPlan& p, sps_dtype qt, sps_dtype kvt, const void* q,
                           float q_scale, const void* kc, const void* vc, const void* ks,
                           const void* vs, const int32_t* page_table, float* partial,
                           int64_t split_stride, float* lse, int64_t lse_split_stride,
                           cudaStream_t st) {
  (void)ks;
  (void)vs;
  if (qt == SPS_BF16 && kvt == SPS_BF16) {
    if (p.D == 128)
      return run_forward<128>(p, q, kc, vc, page_table, partial, split_stride, lse,
                              lse_split_stride, q_scale, st);
    return run_forward<64>(p, q, kc, vc, page_table, partial, split_stride, lse,
                           lse_split_stride, q_scale, st);
  }
  return cudaErrorNotSupported;
}

}  // namespace sps
