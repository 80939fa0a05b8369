// Device helpers and internal data structures of the NVFP4 MoE library (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/nvfp4_moe.h"

namespace nvmoe {

// ---------------------------------------------------------------------------
// device status word: the first non-zero code wins, later ones are dropped
// ---------------------------------------------------------------------------
__device__ __forceinline__ void latch_status(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

// ---------------------------------------------------------------------------
// NVFP4 decode
// ---------------------------------------------------------------------------
// Two E2M1 codes (one byte, even element in the low nibble) -> f16x2, exact.
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte) {
  uint32_t out;
  asm("{\n\t.reg .b8 b;\n\tcvt.u8.u32 b, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b;\n\t}"
      : "=r"(out) : "r"(byte));
  return out;
}

// One E4M3 byte -> fp32, exact.
__device__ __forceinline__ float e4m3_to_f32(uint32_t byte) {
  uint32_t h2;
  uint16_t in = static_cast<uint16_t>(byte & 0xFF);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
  return __half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xFFFF)));
}

// Two E4M3 bytes (lo = first) -> two fp32, exact.
__device__ __forceinline__ float2 e4m3x2_to_f32x2(uint32_t two) {
  uint32_t h2;
  uint16_t in = static_cast<uint16_t>(two & 0xFFFF);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
  __half2 h = *reinterpret_cast<__half2*>(&h2);
  return __half22float2(h);
}

__device__ __forceinline__ float2 f16x2_to_f32x2(uint32_t v) {
  __half2 h = *reinterpret_cast<__half2*>(&v);
  return __half22float2(h);
}

// Sum over 16 E2M1 codes (8 bytes: lo, hi words) times 16 fp32 x values.
// Each product e2m1 * x is exact in fp32 (2 + 8 significant bits).
__device__ __forceinline__ float dot16_e2m1(uint32_t lo, uint32_t hi, const float* x) {
  float acc = 0.f;
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    float2 v = f16x2_to_f32x2(e2m1x2_to_f16x2((lo >> (8 * b)) & 0xFF));
    acc = fmaf(v.x, x[2 * b], acc);
    acc = fmaf(v.y, x[2 * b + 1], acc);
  }
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    float2 v = f16x2_to_f32x2(e2m1x2_to_f16x2((hi >> (8 * b)) & 0xFF));
    acc = fmaf(v.x, x[8 + 2 * b], acc);
    acc = fmaf(v.y, x[8 + 2 * b + 1], acc);
  }
  return acc;
}

// Decode 32 E2M1 codes (a uint4) into 32 fp32 values (unscaled).
__device__ __forceinline__ void decode32_e2m1(const uint4& c, float* out) {
  const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      float2 v = f16x2_to_f32x2(e2m1x2_to_f16x2((w[q] >> (8 * b)) & 0xFF));
      out[q * 8 + 2 * b] = v.x;
      out[q * 8 + 2 * b + 1] = v.y;
    }
  }
}

__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + __expf(-z)); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Sum over aligned segments of `seg` lanes (seg a power of two <= 32).
__device__ __forceinline__ float segment_sum(float v, int seg) {
  for (int o = seg >> 1; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// ---------------------------------------------------------------------------
// Library-owned device layouts (set up by moe_init).
//
//   gu_codes  [n_all][2f][d/2]   rows of W_gate and W_up interleaved in tiles of
//                                64: tile t holds gate rows 64t..64t+63, then up
//                                rows 64t..64t+63 (so one 128-row tile feeds a
//                                SwiGLU of 64 outputs)
//   gu_scales [n_all][2f][d/16]  same row order, E4M3 bytes
//   dn_codes  [n_all][d][f/2]    W_down, canonical
//   dn_scales [n_all][d][f/16]
//   tsc       [n_all][3]         fp32 tensor scales (gate, up, down)
//   BF16 format: gu_bf16 [n_all][2f][d], dn_bf16 [n_all][d][f] instead.
// Experts 0..E-1 are routed, E..E+S-1 shared.
// ---------------------------------------------------------------------------
__host__ __device__ __forceinline__ int gu_row_of_gate(int j) { return (j >> 6) * 128 + (j & 63); }
__host__ __device__ __forceinline__ int gu_row_of_up(int j) { return (j >> 6) * 128 + 64 + (j & 63); }

// Per-forward bookkeeping written by the bucketing kernel.
//   positions p order the (token, expert) pairs: routed pairs grouped by expert
//   (token-major inside a group), then shared expert s at T*k + s*T + t.
struct Routing {
  int32_t* idx;        // [T][k]
  float* w;            // [T][k]
  int32_t* counts;     // [E]
  int32_t* offsets;    // [E+1]
  int32_t* slot_pos;   // [T*k] slot -> position
  int32_t* pos_tok;    // [T*k + S*T] position -> token
  float* pos_w;        // [T*k + S*T] position -> combine weight (1 for shared experts)
  int32_t* act_e;      // [E+S] active experts (count > 0), shared last
  int32_t* act_pos;    // [E+S] first position of each active expert
  int32_t* act_n;      // [E+S] tokens of each active expert
  int32_t* n_active;   // [1]
  int32_t* act_ppos;   // [E+S+1] prefill: padded first row (multiple of 128), total last
  int32_t* blk_a;      // [padded rows / 128] prefill: active expert of each 128-row block
  int32_t* chunk_cnt;  // [ceil(T/32)][E] scratch
  int32_t* group_cnt;  // [ceil(T/256)][E] scratch (bucketing of large batches)
  int32_t* rank;       // [T*k] scratch
};

struct Shape {
  int d, f, E, k, S, T;
};

}  // namespace nvmoe
