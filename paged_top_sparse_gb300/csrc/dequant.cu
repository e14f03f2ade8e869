// dequant.cu -- exact dequantisation of E4M3 and NVFP4 data to FP16 ("MSA PR 21: Q8KV4 paged
// sparse prefill", Build the prefill for SM107: an E2M1 code times its E4M3 scale is exact in
// FP16, so the product needs no rounding).
//
//   E4M3  -> FP16: every E4M3 value is an FP16 value (3 mantissa bits, exponents 2^-9..2^8).
//   NVFP4 -> FP16: E2M1 code (hardware cvt to FP16) times the E4M3 scale of its 16-element
//                  block (cvt to FP16), one FP16 multiply that is exact: the product has at
//                  most 6 significant bits and lies within [2^-10, 2688].
//
// Streaming kernels (grid-stride, 16 elements per thread per step): the E4M3 query copy that
// the FP16 tensor-core paths read, the public sps_dequantize, and, for an indexer over NVFP4
// keys, the batch's visible key pages gathered through the page table into logical order (the
// forward dequantises its K/V tiles inside its own loader instead).
#include <cuda_fp16.h>

#include "ptx.cuh"
#include "sps_internal.h"

namespace sps {

namespace {

__global__ void __launch_bounds__(256)
e4m3_to_f16_kernel(const uint4* __restrict__ in, uint4* __restrict__ out, int64_t n16) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n16;
       i += (int64_t)gridDim.x * blockDim.x) {
    const uint4 v = __ldg(in + i);  // 16 codes
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t h[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      h[2 * j] = cvt_e4m3x2((uint16_t)(w[j] & 0xffff));
      h[2 * j + 1] = cvt_e4m3x2((uint16_t)(w[j] >> 16));
    }
    out[2 * i] = make_uint4(h[0], h[1], h[2], h[3]);
    out[2 * i + 1] = make_uint4(h[4], h[5], h[6], h[7]);
  }
}

__global__ void __launch_bounds__(256)
nvfp4_to_f16_kernel(const uint2* __restrict__ codes, const uint8_t* __restrict__ scales,
                    uint4* __restrict__ out, int64_t nblocks) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < nblocks;
       i += (int64_t)gridDim.x * blockDim.x) {
    const uint2 c = __ldg(codes + i);  // 16 codes of one 16-element block
    const uint8_t sb = __ldg(scales + i);
    const uint32_t s2 = cvt_e4m3x2((uint16_t)(sb | (sb << 8)));  // (scale, scale)
    const uint32_t w[2] = {c.x, c.y};
    uint32_t h[8];
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int b = 0; b < 4; ++b)
        h[4 * j + b] = hmul2_u32(cvt_e2m1x2((uint16_t)((w[j] >> (8 * b)) & 0xff)), s2);
    out[2 * i] = make_uint4(h[0], h[1], h[2], h[3]);
    out[2 * i + 1] = make_uint4(h[4], h[5], h[6], h[7]);
  }
}

// One NVFP4 block -> 16 E4M3 codes: the exact FP16 product, then cvt.rn.satfinite to E4M3.
__global__ void __launch_bounds__(256)
nvfp4_to_e4m3_kernel(const uint2* __restrict__ codes, const uint8_t* __restrict__ scales,
                     uint4* __restrict__ out, int64_t nblocks) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < nblocks;
       i += (int64_t)gridDim.x * blockDim.x) {
    const uint2 c = __ldg(codes + i);
    const uint8_t sb = __ldg(scales + i);
    const uint32_t s2 = cvt_e4m3x2((uint16_t)(sb | (sb << 8)));
    const uint32_t w[2] = {c.x, c.y};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int b = 0; b < 4; b += 2) {
        const uint32_t h0 = hmul2_u32(cvt_e2m1x2((uint16_t)((w[j] >> (8 * b)) & 0xff)), s2);
        const uint32_t h1 = hmul2_u32(cvt_e2m1x2((uint16_t)((w[j] >> (8 * b + 8)) & 0xff)), s2);
        uint16_t e0, e1;
        asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(e0) : "r"(h0));
        asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(e1) : "r"(h1));
        o[2 * j + b / 2] = (uint32_t)e0 | ((uint32_t)e1 << 16);
      }
    out[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// The batch's visible key pages, in logical order: block (global page slot gp, KV head g)
// converts the NVFP4 tile of physical page page_table[req][pg] into tile gp * H_kv + g of `out`
// (FP16 [total_pages][H_kv][128][D]).  A page-table entry outside [0, num_phys_pages) raises
// DEV_BAD_PAGE and converts page 0 instead.
__global__ void __launch_bounds__(256)
nvfp4_pages_to_f16_kernel(DevPlan p, const uint2* __restrict__ codes,
                          const uint8_t* __restrict__ scales, const int32_t* __restrict__ pt,
                          uint4* __restrict__ out) {
  const int gp = blockIdx.x / p.Hkv, g = blockIdx.x % p.Hkv;
  const int req = p.page_req[gp];
  const int pg = gp - p.reqs[req].page_base;
  int phys = __ldg(pt + (int64_t)req * p.max_pages + pg);
  if (phys < 0 || phys >= p.num_phys) {
    if (threadIdx.x == 0) set_status(p.status, DEV_BAD_PAGE);
    phys = 0;
  }
  const int nb = 128 * p.D / 16;  // 16-element blocks of one tile
  const int64_t src = (int64_t)(phys * p.Hkv + g) * nb;
  const int64_t dst = (int64_t)blockIdx.x * nb;
  for (int i = threadIdx.x; i < nb; i += blockDim.x) {
    const uint2 c = __ldg(codes + src + i);
    const uint8_t sb = __ldg(scales + src + i);
    const uint32_t s2 = cvt_e4m3x2((uint16_t)(sb | (sb << 8)));
    const uint32_t w[2] = {c.x, c.y};
    uint32_t h[8];
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int b = 0; b < 4; ++b)
        h[4 * j + b] = hmul2_u32(cvt_e2m1x2((uint16_t)((w[j] >> (8 * b)) & 0xff)), s2);
    out[2 * (dst + i)] = make_uint4(h[0], h[1], h[2], h[3]);
    out[2 * (dst + i) + 1] = make_uint4(h[4], h[5], h[6], h[7]);
  }
}

}  // namespace

cudaError_t launch_dequant_pages(const DevPlan& p, const void* codes, const void* scales,
                                 const int32_t* page_table, void* out, cudaStream_t st) {
  const int64_t tiles = (int64_t)p.total_pages * p.Hkv;
  if (tiles <= 0) return cudaSuccess;
  nvfp4_pages_to_f16_kernel<<<(unsigned)tiles, 256, 0, st>>>(
      p, static_cast<const uint2*>(codes), static_cast<const uint8_t*>(scales), page_table,
      static_cast<uint4*>(out));
  return cudaGetLastError();
}

cudaError_t launch_dequant_e4m3(const void* in, const void* scales, int64_t n, void* out,
                                cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  const int64_t blocks = n / 16;
  const unsigned grid = (unsigned)std::min<int64_t>((blocks + 255) / 256, 8LL * num_sms());
  nvfp4_to_e4m3_kernel<<<grid, 256, 0, st>>>(static_cast<const uint2*>(in),
                                              static_cast<const uint8_t*>(scales),
                                              static_cast<uint4*>(out), blocks);
  return cudaGetLastError();
}

cudaError_t launch_dequant(sps_dtype dt, const void* in, const void* scales, int64_t n,
                           void* out, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  const int64_t units = n / 16;
  const unsigned grid = (unsigned)std::min<int64_t>((units + 255) / 256, 8LL * num_sms());
  if (dt == SPS_E4M3)
    e4m3_to_f16_kernel<<<grid, 256, 0, st>>>(static_cast<const uint4*>(in),
                                              static_cast<uint4*>(out), units);
  else if (dt == SPS_NVFP4)
    nvfp4_to_f16_kernel<<<grid, 256, 0, st>>>(static_cast<const uint2*>(in),
                                               static_cast<const uint8_t*>(scales),
                                               static_cast<uint4*>(out), units);
  else
    return cudaErrorNotSupported;
  return cudaGetLastError();
}

}  // namespace sps
