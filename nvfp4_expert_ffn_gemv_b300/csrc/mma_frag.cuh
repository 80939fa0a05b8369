// NVFP4 operands for mma.sync m16n8k16 (f16 inputs, fp32 accumulation):
// expansion of E2M1 codes and E4M3 block scales into exact f16 A fragments,
// the k permutation that lets every thread read contiguous code bytes, and
// the f16 hi + lo split of an fp32 operand.
//
// Exactness: an E2M1 code times its E4M3 block scale has at most 6 significant
// bits and lies in [2^-10, 2688], so it is exact in f16; the product is formed
// with the hardware cvt (e2m1x2 -> f16x2) and an f16x2 multiply that cannot
// round.  An fp32 operand v enters as hi = f16(v * 2^s), lo = f16(v * 2^s - hi)
// after a power-of-two prescale 2^s, about 22 significant bits; the products
// of the two with an exact f16 weight are exact in fp32.
//
// K permutation.  A sum over k does not depend on the order of k, so the MMA's
// k slots are assigned to actual k such that every thread reads contiguous
// bytes: in a 128-wide k chunk, thread quad position c (lane % 4) owns k =
// 32c .. 32c+31 (16 code bytes of a row), and MMA step kk (0..7) takes its k
// slots {2c, 2c+1} <- k = 32c+4kk+{0,1} and {2c+8, 2c+9} <- 32c+4kk+{2,3}.
// The B operand is stored in that order: 8-byte groups (kk, c), see perm_off.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

namespace nvmoe {
namespace frag {

__device__ __forceinline__ uint32_t cvt_e4m3x2_f16x2(uint32_t two) {
  uint32_t out;
  const uint16_t in = static_cast<uint16_t>(two & 0xFFFF);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(out) : "h"(in));
  return out;
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t out;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(out) : "r"(a), "r"(b));
  return out;
}

// {lo, lo} and {hi, hi} of an f16x2
__device__ __forceinline__ uint32_t bcast_lo(uint32_t v) { return __byte_perm(v, v, 0x1010); }
__device__ __forceinline__ uint32_t bcast_hi(uint32_t v) { return __byte_perm(v, v, 0x3232); }

__device__ __forceinline__ void mma_f16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint2 lds64(const uint8_t* p) { return *reinterpret_cast<const uint2*>(p); }

// 2^k as a float for -126 <= k <= 127
__device__ __forceinline__ float pow2i(int k) { return __uint_as_float((uint32_t)(k + 127) << 23); }

// exponent shift that maps max|v| (as fp32 bits, non-negative) into [2^14, 2^15)
__device__ __forceinline__ int prescale_shift(uint32_t amax_bits) {
  if (amax_bits == 0u) return 0;
  const int ex = (int)((amax_bits >> 23) & 0xFF) - 127;
  return max(-126, min(126, 14 - ex));
}

// byte offset, inside one 128-wide k chunk of f16 values, of the 4 values
// k = 32c + 4kk + 0..3
__device__ __forceinline__ int perm_off(int c, int kk) { return (kk * 4 + c) * 8; }

// Eight E2M1 codes (one word, element 2j in the low nibble of byte j) -> four
// exact f16x2, one mov splitting the word into bytes and four hardware cvts.
__device__ __forceinline__ void cvt_e2m1x8(uint32_t w, uint32_t (&o)[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3]) : "r"(w));
}

// A fragments of the two MMA steps 2w and 2w+1 from word w of the quad's code
// slice of rows g (wg) and g+8 (wg8): bytes 0, 1 feed step 2w, bytes 2, 3 step
// 2w+1; every f16x2 is multiplied by its row's block scale (exact).
__device__ __forceinline__ void a_frag_pair(uint32_t (&a0)[4], uint32_t (&a1)[4], uint32_t wg, uint32_t wg8,
                                            uint32_t sg, uint32_t sg8) {
  uint32_t g[4], h[4];
  cvt_e2m1x8(wg, g);
  cvt_e2m1x8(wg8, h);
  a0[0] = hmul2(g[0], sg);
  a0[2] = hmul2(g[1], sg);
  a0[1] = hmul2(h[0], sg8);
  a0[3] = hmul2(h[1], sg8);
  a1[0] = hmul2(g[2], sg);
  a1[2] = hmul2(g[3], sg);
  a1[1] = hmul2(h[2], sg8);
  a1[3] = hmul2(h[3], sg8);
}

__device__ __forceinline__ uint32_t word_of(const uint4& v, int i) {
  return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

// hi + lo f16 split of four prescaled fp32 values (packed as two f16x2 each)
__device__ __forceinline__ void split_hi_lo(float s0, float s1, float s2, float s3, uint2& hi, uint2& lo) {
  const __half2 h01 = __floats2half2_rn(s0, s1), h23 = __floats2half2_rn(s2, s3);
  const float2 r01 = __half22float2(h01), r23 = __half22float2(h23);
  const __half2 l01 = __floats2half2_rn(s0 - r01.x, s1 - r01.y);
  const __half2 l23 = __floats2half2_rn(s2 - r23.x, s3 - r23.y);
  hi = make_uint2(*reinterpret_cast<const uint32_t*>(&h01), *reinterpret_cast<const uint32_t*>(&h23));
  lo = make_uint2(*reinterpret_cast<const uint32_t*>(&l01), *reinterpret_cast<const uint32_t*>(&l23));
}

}  // namespace frag
}  // namespace nvmoe
