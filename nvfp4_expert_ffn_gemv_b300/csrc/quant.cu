// NVFP4 quantiser for weights (fp32 -> E2M1 codes, E4M3 block scales, fp32 tensor scale).
//
// The pages name NVFP4 as the shipped format ("Recursive Flint 40B-A2.5B：まず速さを
// 第一に考えて作られたコーディングモデル", section "量子化のレシピは最も転用しやすい部分
// です") without a definition.  Reading used, all in IEEE fp32 with
// round-to-nearest-even, one operation at a time (no contraction):
//   ts = amax / 2688;  s = E4M3_satfinite(amax_16 / (6 * ts));
//   d = e4m3(s) * ts;  q = E2M1_satfinite(v / d), canonical zero (never -0).
// Three launches: per-tensor amax (atomicMax on the fp32 bit pattern, which
// orders non-negative floats), the block step, and ts = amax / 2688.
#include "internal.h"

namespace nvmoe {

namespace {

__device__ __forceinline__ uint32_t f32_to_e4m3(float v) {
  uint16_t out;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(out) : "f"(0.0f), "f"(v));
  return out & 0xFF;
}

// (even, odd) -> one byte, even element in the low nibble; -0 canonicalised to 0
__device__ __forceinline__ uint32_t f32x2_to_e2m1x2(float even, float odd) {
  uint16_t out;
  asm("{\n\t.reg .b8 b;\n\tcvt.rn.satfinite.e2m1x2.f32 b, %1, %2;\n\tcvt.u16.u8 %0, b;\n\t}"
      : "=h"(out) : "f"(odd), "f"(even));
  uint32_t v = out & 0xFF;
  if ((v & 0x07) == 0) v &= 0xF0;
  if ((v & 0x70) == 0) v &= 0x0F;
  return v;
}

__global__ void amax_kernel(const float* __restrict__ w, size_t per_tensor, uint32_t* amax_bits) {
  const int n = blockIdx.y;
  const float4* p = reinterpret_cast<const float4*>(w + (size_t)n * per_tensor);
  const size_t n4 = per_tensor / 4;
  float m = 0.f;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4;
       i += (size_t)gridDim.x * blockDim.x) {
    const float4 v = __ldg(p + i);
    m = fmaxf(m, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) atomicMax(amax_bits + n, __float_as_uint(m));
}

// one thread per 16-element block
__global__ void block_quant_kernel(const float* __restrict__ w, size_t per_tensor,
                                   const uint32_t* __restrict__ amax_bits, uint8_t* __restrict__ codes,
                                   uint8_t* __restrict__ scales) {
  const int n = blockIdx.y;
  const size_t nblk = per_tensor / 16;
  const size_t b = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= nblk) return;
  const float amax = __uint_as_float(amax_bits[n]);
  const float ts = __fdiv_rn(amax, 2688.0f);
  const float4* p = reinterpret_cast<const float4*>(w + (size_t)n * per_tensor + b * 16);
  float v[16];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float4 t = __ldg(p + q);
    v[4 * q] = t.x; v[4 * q + 1] = t.y; v[4 * q + 2] = t.z; v[4 * q + 3] = t.w;
  }
  uint32_t s_code = 0;
  float dq = 0.f;
  if (ts > 0.f) {
    float ab = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) ab = fmaxf(ab, fabsf(v[i]));
    const float six_ts = __fmul_rn(6.0f, ts);
    s_code = f32_to_e4m3(__fdiv_rn(ab, six_ts));
    dq = __fmul_rn(e4m3_to_f32(s_code), ts);
  }
  uint32_t lo = 0, hi = 0;
  if (dq > 0.f) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      lo |= f32x2_to_e2m1x2(__fdiv_rn(v[2 * i], dq), __fdiv_rn(v[2 * i + 1], dq)) << (8 * i);
      hi |= f32x2_to_e2m1x2(__fdiv_rn(v[8 + 2 * i], dq), __fdiv_rn(v[8 + 2 * i + 1], dq)) << (8 * i);
    }
  }
  reinterpret_cast<uint2*>(codes + (size_t)n * (per_tensor / 2))[b] = make_uint2(lo, hi);
  scales[(size_t)n * nblk + b] = static_cast<uint8_t>(s_code);
}

__global__ void finish_ts_kernel(float* ts, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) ts[i] = __fdiv_rn(__uint_as_float(reinterpret_cast<uint32_t*>(ts)[i]), 2688.0f);
}

}  // namespace

cudaError_t launch_quantize_nvfp4(const float* w, int n, int rows, int K, uint8_t* codes,
                                  uint8_t* scales, float* ts, cudaStream_t s) {
  const size_t per = (size_t)rows * K;
  cudaError_t err = cudaMemsetAsync(ts, 0, sizeof(float) * n, s);
  if (err != cudaSuccess) return err;
  uint32_t* bits = reinterpret_cast<uint32_t*>(ts);
  int gx = (int)((per / 4 + 255) / 256);
  if (gx > 256) gx = 256;
  amax_kernel<<<dim3(gx, n), 256, 0, s>>>(w, per, bits);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  const size_t nblk = per / 16;
  block_quant_kernel<<<dim3((unsigned)((nblk + 255) / 256), n), 256, 0, s>>>(w, per, bits, codes, scales);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  finish_ts_kernel<<<(n + 255) / 256, 256, 0, s>>>(ts, n);
  return cudaGetLastError();
}

}  // namespace nvmoe
