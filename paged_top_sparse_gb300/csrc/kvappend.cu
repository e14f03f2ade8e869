// kvappend.cu -- the chunked-prefill step before the indexer: the new tokens' K/V go into the
// paged cache through the page table, quantised to NVFP4 where the cache is NVFP4, and the
// query is quantised to E4M3 with a per-tensor scale.  (The pages fix the formats -- "MSA PR
// 21: Q8KV4 paged sparse prefill", E4M3 query and NVFP4 KV with an E4M3 scale per 16
// elements -- but not this step's rounding; every division here is binary32 and every
// conversion rounds to nearest even and saturates, the cvt.rn.satfinite forms.)
//
//   kv append   a warp per (token, KV head) row; BF16: a plain copy of the row into slot
//               t % 128 of physical page page_table[req][t / 128]; NVFP4: each 16-element
//               block gets scale = E4M3(absmax / 6) and codes E2M1(x / scale), zero codes
//               when the scale rounds to zero; the lanes of a block combine their maxima with
//               shuffles and each lane writes its own packed codes.
//   quantise    E4M3(x / scale) for BF16 x, 16 elements per thread.
//   absmax      max |x| over BF16 values into one FP32 word (bit-ordered atomicMax).
#include <cuda_fp16.h>

#include "ptx.cuh"
#include "sps_internal.h"

namespace sps {
namespace {

__device__ __forceinline__ float bf16_to_f32(uint32_t bits16) { return __uint_as_float(bits16 << 16); }

// E4M3 code of x (round to nearest even, saturating).
__device__ __forceinline__ uint32_t f32_to_e4m3(float x) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(x));
  return r & 0xffu;
}
// Two E2M1 codes packed in a byte: lo in the low nibble (round to nearest even, saturating).
__device__ __forceinline__ uint32_t f32x2_to_e2m1x2(float lo, float hi) {
  uint16_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tmov.b16 %0, {t, t};\n\t}"
      : "=h"(r)
      : "f"(hi), "f"(lo));
  return r & 0xffu;
}
// Value of an E4M3 code (exact).
__device__ __forceinline__ float e4m3_to_f32(uint32_t code) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((uint16_t)code));
  return __half2float(__ushort_as_half((unsigned short)(h2 & 0xffffu)));
}

template <int D, bool NVFP4>
__global__ void __launch_bounds__(256)
kv_append_kernel(DevPlan p, const uint16_t* __restrict__ knew, const uint16_t* __restrict__ vnew,
                 const int32_t* __restrict__ page_table, uint8_t* __restrict__ kc,
                 uint8_t* __restrict__ vc, uint8_t* __restrict__ ks, uint8_t* __restrict__ vs) {
  constexpr int EPL = D / 32;  // elements per lane: 4 (D=128) or 2 (D=64)
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);  // (token, kv head)
  if (row >= (int64_t)p.T * p.Hkv) return;
  const int tok = (int)(row / p.Hkv), g = (int)(row % p.Hkv);
  const int t = __ldg(p.tok_pos + tok), req = __ldg(p.tok_req + tok);
  const int phys = __ldg(page_table + (int64_t)req * p.max_pages + (t >> 7));
  if (phys < 0 || phys >= p.num_phys) {
    if (lane == 0) set_status(p.status, DEV_BAD_PAGE);
    return;
  }
  const int64_t slot = ((int64_t)phys * p.Hkv + g) * 128 + (t & 127);
#pragma unroll
  for (int kv = 0; kv < 2; ++kv) {
    const uint16_t* src = (kv ? vnew : knew) + row * D + lane * EPL;
    uint8_t* cache = kv ? vc : kc;
    uint32_t w[EPL / 2];
    if (EPL == 4) {
      const uint2 x = __ldg(reinterpret_cast<const uint2*>(src));
      w[0] = x.x;
      w[EPL / 2 - 1] = x.y;
    } else {
      w[0] = __ldg(reinterpret_cast<const uint32_t*>(src));
    }
    if (!NVFP4) {
      uint8_t* dst = cache + (slot * D + lane * EPL) * 2;
      if (EPL == 4) *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[EPL / 2 - 1]);
      else *reinterpret_cast<uint32_t*>(dst) = w[0];
      continue;
    }
    float x[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) x[e] = bf16_to_f32((w[e / 2] >> (16 * (e & 1))) & 0xffffu);
    float amax = 0.f;
#pragma unroll
    for (int e = 0; e < EPL; ++e) amax = fmaxf(amax, fabsf(x[e]));
    constexpr int LPB = 16 / EPL;  // lanes per 16-element block
#pragma unroll
    for (int o = 1; o < LPB; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const uint32_t scode = f32_to_e4m3(__fdiv_rn(amax, 6.0f));
    const float sv = e4m3_to_f32(scode);
    uint32_t packed = 0;  // EPL / 2 bytes of codes
#pragma unroll
    for (int e = 0; e < EPL; e += 2) {
      const uint32_t b = sv == 0.f ? 0u
                                   : f32x2_to_e2m1x2(__fdiv_rn(x[e], sv), __fdiv_rn(x[e + 1], sv));
      packed |= b << (8 * (e / 2));
    }
    uint8_t* dst = cache + slot * (D / 2) + lane * (EPL / 2);
    if (EPL == 4) *reinterpret_cast<uint16_t*>(dst) = (uint16_t)packed;
    else *dst = (uint8_t)packed;
    if (lane % LPB == 0) (kv ? vs : ks)[slot * (D / 16) + lane / LPB] = (uint8_t)scode;
  }
}

__global__ void __launch_bounds__(256)
quantize_e4m3_kernel(const uint4* __restrict__ in, float scale, uint4* __restrict__ out,
                     int64_t n16) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n16;
       i += (int64_t)gridDim.x * blockDim.x) {
    const uint4 a = __ldg(in + 2 * i), b = __ldg(in + 2 * i + 1);  // 16 BF16 values
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t v = 0;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint32_t h = (w[2 * j + u / 2] >> (16 * (u & 1))) & 0xffffu;
        v |= f32_to_e4m3(__fdiv_rn(bf16_to_f32(h), scale)) << (8 * u);
      }
      o[j] = v;
    }
    out[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

__global__ void __launch_bounds__(256)
absmax_bf16_kernel(const uint4* __restrict__ in, int64_t n8, uint32_t* __restrict__ out) {
  uint32_t m = 0;  // bits of a non-negative float order like the float
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n8;
       i += (int64_t)gridDim.x * blockDim.x) {
    const uint4 a = __ldg(in + i);
    const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      m = max(m, (w[j] & 0x7fffu) << 16);
      m = max(m, w[j] & 0x7fff0000u);
    }
  }
  m = __reduce_max_sync(0xffffffffu, m);
  if ((threadIdx.x & 31) == 0 && m) atomicMax(out, m);
}

}  // namespace

cudaError_t launch_kv_append(const DevPlan& p, bool nvfp4, const void* knew, const void* vnew,
                             const int32_t* page_table, void* kc, void* vc, void* ks, void* vs,
                             cudaStream_t st) {
  const int64_t rows = (int64_t)p.T * p.Hkv;
  if (rows == 0) return cudaSuccess;
  const unsigned grid = (unsigned)((rows + 7) / 8);
  auto k16 = static_cast<const uint16_t*>(knew), v16 = static_cast<const uint16_t*>(vnew);
  auto kc8 = static_cast<uint8_t*>(kc), vc8 = static_cast<uint8_t*>(vc);
  auto ks8 = static_cast<uint8_t*>(ks), vs8 = static_cast<uint8_t*>(vs);
  if (p.D == 128) {
    if (nvfp4) kv_append_kernel<128, true><<<grid, 256, 0, st>>>(p, k16, v16, page_table, kc8, vc8, ks8, vs8);
    else kv_append_kernel<128, false><<<grid, 256, 0, st>>>(p, k16, v16, page_table, kc8, vc8, ks8, vs8);
  } else {
    if (nvfp4) kv_append_kernel<64, true><<<grid, 256, 0, st>>>(p, k16, v16, page_table, kc8, vc8, ks8, vs8);
    else kv_append_kernel<64, false><<<grid, 256, 0, st>>>(p, k16, v16, page_table, kc8, vc8, ks8, vs8);
  }
  return cudaGetLastError();
}

cudaError_t launch_quantize_e4m3(const void* in, int64_t n, float scale, void* out,
                                 cudaStream_t st) {
  const int64_t n16 = n / 16;
  if (n16 == 0) return cudaSuccess;
  const unsigned grid = (unsigned)std::min<int64_t>((n16 + 255) / 256, 8LL * num_sms());
  quantize_e4m3_kernel<<<grid, 256, 0, st>>>(static_cast<const uint4*>(in), scale,
                                              static_cast<uint4*>(out), n16);
  return cudaGetLastError();
}

cudaError_t launch_absmax_bf16(const void* in, int64_t n, float* out, cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(out, 0, sizeof(float), st);
  if (e != cudaSuccess) return e;
  const int64_t n8 = n / 8;
  if (n8 == 0) return cudaSuccess;
  const unsigned grid = (unsigned)std::min<int64_t>((n8 + 255) / 256, 4LL * num_sms());
  absmax_bf16_kernel<<<grid, 256, 0, st>>>(static_cast<const uint4*>(in), n8,
                                            reinterpret_cast<uint32_t*>(out));
  return cudaGetLastError();
}

}  // namespace sps
