// Batched decode (T >= 2 tokens, NVFP4 weights): the expert products as small
// tensor-core GEMMs, one (expert, 128 weight rows, up to 16 tokens) tile per
// CTA iteration.
//
// The Flint pages frame decode as streaming the chosen experts' weights
// ("Recursive Flint 40B-A2.5B：まず速さを第一に考えて作られたコーディングモデル",
// section "このアーキテクチャはメモリ帯域幅に関する主張である").  Once a batch
// sends several tokens to one expert, every weight byte feeds several tokens,
// and on CUDA cores the per-token FMAs (about 1.2e9 for 64 tokens) would cost
// as much time as streaming the bytes.  Here each weight is expanded once and
// multiplied on the tensor cores (mma.sync m16n8k16, f16 inputs, fp32
// accumulation), so the kernels stay bound by the weight stream.
//
// Exactness of the operands:
//   - weights: an E2M1 code times its E4M3 block scale has at most 6
//     significant bits and lies in [2^-13, 2688], so it is exact in f16; the
//     product is formed with the hardware cvt (e2m1x2 -> f16x2) and an f16x2
//     multiply that cannot round.  The FP32 tensor scale is applied to the
//     fp32 result.
//   - x: bf16 values, times a per-token power of two that maps max|x| into
//     [2^14, 2^15), are exact in f16 down to 2^-29 of the token's largest
//     entry (below that f16 keeps fewer bits).
//   - h (fp32) enters the down projection as hi + lo, two f16 numbers after a
//     per-position power-of-two prescale (about 22 significant bits), i.e. two
//     MMAs per tile.
// Every product is exact; only the fp32 accumulation rounds.
//
// K permutation.  A sum over k does not depend on the order of k, so the MMA's
// k slots are assigned to actual k such that every thread reads contiguous
// bytes: in a 128-wide k chunk, thread quad position c (lane % 4) owns k =
// 32c .. 32c+31 (16 code bytes of a row), and MMA step kk (0..7) takes its k
// slots {2c, 2c+1} <- k = 32c+4kk+{0,1} and {2c+8, 2c+9} <- 32c+4kk+{2,3}.
// Activations are stored in shared memory in that order (8-byte groups
// (kk, c)), with a row stride of 32 bytes mod 128, so the B fragment loads
// are free of bank conflicts.
#include <cuda_fp16.h>

#include "internal.h"
#include "mma_frag.cuh"

namespace nvmoe {

namespace {

using namespace frag;

constexpr int kThreads = 256;   // 8 warps x 16 weight rows = 128 rows per tile
constexpr int kTok = 8;         // tokens (positions) per tile: one MMA column group
constexpr int kChunk = 128;     // k per chunk

// ---------------------------------------------------------------------------
// small helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" :: "r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

// Weight bytes are read once per call: a read-only load that does not allocate
// in L1 (the L1 / shared-memory pipe is busy with the activation fragments).
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 v;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

struct MmaArgs {
  Routing r;
  const __nv_bfloat16* x;   // [T][d]
  const uint8_t* gu_codes;  // [n_all][2f][d/2], gate/up tiles of 64 rows
  const uint8_t* gu_scales; // [n_all][2f][d/16]
  const uint8_t* dn_codes;  // [n_all][d][f/2]
  const uint8_t* dn_scales; // [n_all][d][f/16]
  const float* tsc;         // [n_all][3]
  uint8_t* x16;             // [T][d] f16, prescaled, k-permuted per 128 chunk
  float* xunshift;          // [T]
  float* h;                 // [P][f]
  float* yexp;              // [P][d]
  int d, f, T;
};

// Per-CTA table of 16-position groups: gpre[a] = first group of active expert a,
// gpre[na] = total.  One warp builds it (na <= 258).
__device__ __forceinline__ int build_groups(const Routing& r, int* gpre) {
  const int na = *r.n_active;
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int base = 0;
    for (int a0 = 0; a0 < na; a0 += 32) {
      const int a = a0 + lane;
      const int g = a < na ? (r.act_n[a] + kTok - 1) / kTok : 0;
      int inc = g;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int up = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += up;
      }
      if (a < na) gpre[a] = base + inc - g;
      base += __shfl_sync(0xffffffffu, inc, 31);
    }
    if (lane == 0) gpre[na] = base;
  }
  __syncthreads();
  return na;
}

__device__ __forceinline__ int find_group(const int* gpre, int na, int gidx) {
  int lo = 0, hi = na - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (gpre[mid] <= gidx) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// ---------------------------------------------------------------------------
// x -> prescaled f16 in the permuted chunk order (one warp per token)
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) xprep_kernel(MmaArgs g) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  if (t >= g.T) return;
  const int d = g.d;
  const uint4* src = reinterpret_cast<const uint4*>(g.x + (size_t)t * d);
  float m = 0.f;
  for (int i = lane; i < d / 8; i += 32) {
    const uint4 v = __ldg(src + i);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q)
      m = fmaxf(m, fmaxf(fabsf(__uint_as_float(w[q] << 16)), fabsf(__uint_as_float(w[q] & 0xFFFF0000u))));
  }
  const uint32_t mb = __reduce_max_sync(0xffffffffu, __float_as_uint(m));
  const int shift = prescale_shift(mb);
  const float sc = pow2i(shift);
  uint8_t* dst = g.x16 + (size_t)t * d * 2;
  for (int i = lane; i < d / 8; i += 32) {
    const uint4 v = __ldg(src + i);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t hv[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const __half2 hh = __floats2half2_rn(__uint_as_float(w[q] << 16) * sc,
                                           __uint_as_float(w[q] & 0xFFFF0000u) * sc);
      hv[q] = *reinterpret_cast<const uint32_t*>(&hh);
    }
    // elements k0 .. k0+7 of the row, k0 = 8i: chunk k0/128, k' = k0 % 128 = 32c + 4kk (kk even)
    const int k0 = 8 * i, ch = k0 / kChunk, kp = k0 % kChunk;
    const int c = kp / 32, kk = (kp % 32) / 4;
    uint8_t* base = dst + (size_t)ch * kChunk * 2;
    *reinterpret_cast<uint2*>(base + perm_off(c, kk)) = make_uint2(hv[0], hv[1]);
    *reinterpret_cast<uint2*>(base + perm_off(c, kk + 1)) = make_uint2(hv[2], hv[3]);
  }
  if (lane == 0) g.xunshift[t] = pow2i(-shift);
}

// ---------------------------------------------------------------------------
// gate/up + SwiGLU.  Tile = (active expert, 128 gate/up rows = 64 hidden
// units, up to 16 of its positions).  Warps 0-3 hold the gate rows, 4-7 the up
// rows of the same hidden units.
// ---------------------------------------------------------------------------
template <int D>
struct GuSmem {
  static constexpr int kXRow = D * 2 + 32;                 // bytes per staged token row
  static constexpr int kX = 0;
  static constexpr int kG = kX + kTok * kXRow;             // float [64][kTok + 1]
  static constexpr int kU = kG + 64 * (kTok + 1) * 4;
  static constexpr int kTokInfo = kU + 64 * (kTok + 1) * 4;  // int tok[kTok], float unshift[kTok]
  static constexpr int kGroups = kTokInfo + kTok * 8;      // int gpre[E + S + 1]
  static constexpr int bytes(int na_max) { return kGroups + (na_max + 1) * 4; }
};

template <int D>
__global__ void __launch_bounds__(kThreads, 4) gateup_mma_kernel(MmaArgs g) {
  using L = GuSmem<D>;
  constexpr int NCH = D / kChunk;        // 128-wide k chunks
  constexpr int B = 2;                   // chunks per register batch
  constexpr int NB = NCH / B;
  extern __shared__ __align__(16) uint8_t sm[];
  float* sG = reinterpret_cast<float*>(sm + L::kG);
  float* sU = reinterpret_cast<float*>(sm + L::kU);
  int* sTok = reinterpret_cast<int*>(sm + L::kTokInfo);
  float* sUn = reinterpret_cast<float*>(sm + L::kTokInfo + kTok * 4);
  int* gpre = reinterpret_cast<int*>(sm + L::kGroups);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = lane >> 2, c = lane & 3;
  const int f = g.f;
  const int rtiles = 2 * f / 128;
  const int na = build_groups(g.r, gpre);
  const int units = gpre[na] * rtiles;

  for (int u = blockIdx.x; u < units; u += gridDim.x) {
    const int gi = u / rtiles, rt = u % rtiles;
    const int a = find_group(gpre, na, gi);
    const int e = g.r.act_e[a];
    const int p0 = g.r.act_pos[a] + (gi - gpre[a]) * kTok;
    const int nt = min(kTok, g.r.act_n[a] - (gi - gpre[a]) * kTok);

    // weight rows of this thread: tile row 16*warp + gq and + 8
    const size_t row = (size_t)e * 2 * f + rt * 128 + warp * 16 + gq;
    const uint8_t* cg = g.gu_codes + row * (D / 2) + c * 16;
    const uint8_t* cg8 = cg + (size_t)8 * (D / 2);
    const uint8_t* sgp = g.gu_scales + row * (D / 16) + c * 2;
    const uint8_t* sg8p = sgp + (size_t)8 * (D / 16);

    uint4 wc[B], wc8[B];
    uint32_t ws[B], ws8[B];
#pragma unroll
    for (int i = 0; i < B; ++i) {
      wc[i] = ld_stream16(cg + i * 64);
      wc8[i] = ld_stream16(cg8 + i * 64);
      ws[i] = __ldg(reinterpret_cast<const uint16_t*>(sgp + i * 8));
      ws8[i] = __ldg(reinterpret_cast<const uint16_t*>(sg8p + i * 8));
    }

    __syncthreads();  // previous tile's smem readers are done
    if (threadIdx.x < kTok) {
      const int t = threadIdx.x < nt ? g.r.pos_tok[p0 + threadIdx.x] : 0;
      sTok[threadIdx.x] = t;
      sUn[threadIdx.x] = g.xunshift[t];
    }
    __syncthreads();
    // stage the tile's tokens (prescaled f16 rows) with async copies
    for (int i = threadIdx.x; i < nt * (D * 2 / 16); i += kThreads) {
      const int rr = i / (D * 2 / 16), q = i % (D * 2 / 16);
      cp_async16(sm + L::kX + rr * L::kXRow + q * 16, g.x16 + (size_t)sTok[rr] * D * 2 + q * 16);
    }
    cp_async_wait_all();
    __syncthreads();

    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    const bool two = nt > 8;
    const uint8_t* xrow0 = sm + L::kX + gq * L::kXRow;
    const uint8_t* xrow1 = xrow0 + 8 * L::kXRow;

#pragma unroll
    for (int b = 0; b < NB; ++b) {
      uint4 nc[B], nc8[B];
      uint32_t ns[B], ns8[B];
      if (b + 1 < NB) {
#pragma unroll
        for (int i = 0; i < B; ++i) {
          const int ch = (b + 1) * B + i;
          nc[i] = ld_stream16(cg + ch * 64);
          nc8[i] = ld_stream16(cg8 + ch * 64);
          ns[i] = __ldg(reinterpret_cast<const uint16_t*>(sgp + ch * 8));
          ns8[i] = __ldg(reinterpret_cast<const uint16_t*>(sg8p + ch * 8));
        }
      }
#pragma unroll
      for (int i = 0; i < B; ++i) {
        const int ch = b * B + i;
        const uint32_t s2 = cvt_e4m3x2_f16x2(ws[i]), s28 = cvt_e4m3x2_f16x2(ws8[i]);
#pragma unroll
        for (int wd = 0; wd < 4; ++wd) {
          const uint32_t sg = wd < 2 ? bcast_lo(s2) : bcast_hi(s2);
          const uint32_t sg8 = wd < 2 ? bcast_lo(s28) : bcast_hi(s28);
          uint32_t afp[2][4];
          a_frag_pair(afp[0], afp[1], word_of(wc[i], wd), word_of(wc8[i], wd), sg, sg8);
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            const int kk = 2 * wd + h2;
            const int off = ch * kChunk * 2 + perm_off(c, kk);
            const uint2 b0 = lds64(xrow0 + off);
            mma_f16(acc[0], afp[h2], b0.x, b0.y);
            if (two) {
              const uint2 b1 = lds64(xrow1 + off);
              mma_f16(acc[1], afp[h2], b1.x, b1.y);
            }
          }
        }
      }
      if (b + 1 < NB) {
#pragma unroll
        for (int i = 0; i < B; ++i) {
          wc[i] = nc[i];
          wc8[i] = nc8[i];
          ws[i] = ns[i];
          ws8[i] = ns8[i];
        }
      }
    }

    // epilogue: scale, hand gate / up values to shared memory, SwiGLU, store h
    const float ts = g.tsc[e * 3 + (warp < 4 ? 0 : 1)];
    float* dst = warp < 4 ? sG : sU;
    const int j0 = (warp & 3) * 16 + gq;
#pragma unroll
    for (int q = 0; q < kTok / 8; ++q) {
      const int col = q * 8 + 2 * c;
      dst[j0 * (kTok + 1) + col] = acc[q][0] * ts * sUn[col];
      dst[j0 * (kTok + 1) + col + 1] = acc[q][1] * ts * sUn[col + 1];
      dst[(j0 + 8) * (kTok + 1) + col] = acc[q][2] * ts * sUn[col];
      dst[(j0 + 8) * (kTok + 1) + col + 1] = acc[q][3] * ts * sUn[col + 1];
    }
    __syncthreads();
    for (int i = threadIdx.x; i < 64 * nt; i += kThreads) {
      const int j = i & 63, col = i >> 6;
      const float gv = sG[j * (kTok + 1) + col], uv = sU[j * (kTok + 1) + col];
      g.h[(size_t)(p0 + col) * f + rt * 64 + j] = silu_f(gv) * uv;
    }
  }
}

// ---------------------------------------------------------------------------
// down projection.  Tile = (active expert, 128 output rows, up to 16 positions).
// ---------------------------------------------------------------------------
template <int F>
struct DnSmem {
  static constexpr int kHRow = F * 2 + 32;
  static constexpr int kHi = 0;
  static constexpr int kLo = kHi + kTok * kHRow;
  static constexpr int kY = kLo + kTok * kHRow;         // float [kTok][128 + 4]
  static constexpr int kUn = kY + kTok * 132 * 4;       // float [kTok]
  static constexpr int kGroups = kUn + kTok * 4;
  static constexpr int bytes(int na_max) { return kGroups + (na_max + 1) * 4; }
};

template <int F>
__global__ void __launch_bounds__(kThreads, 4) down_mma_kernel(MmaArgs g) {
  using L = DnSmem<F>;
  constexpr int NCH = F / kChunk;
  constexpr int B = NCH < 2 ? NCH : 2;
  constexpr int NB = NCH / B;
  extern __shared__ __align__(16) uint8_t sm[];
  float* sY = reinterpret_cast<float*>(sm + L::kY);
  float* sUn = reinterpret_cast<float*>(sm + L::kUn);
  int* gpre = reinterpret_cast<int*>(sm + L::kGroups);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = lane >> 2, c = lane & 3;
  const int d = g.d;
  const int rtiles = d / 128;
  const int na = build_groups(g.r, gpre);
  const int units = gpre[na] * rtiles;

  for (int u = blockIdx.x; u < units; u += gridDim.x) {
    const int gi = u / rtiles, rt = u % rtiles;
    const int a = find_group(gpre, na, gi);
    const int e = g.r.act_e[a];
    const int p0 = g.r.act_pos[a] + (gi - gpre[a]) * kTok;
    const int nt = min(kTok, g.r.act_n[a] - (gi - gpre[a]) * kTok);

    const size_t row = (size_t)e * d + rt * 128 + warp * 16 + gq;
    const uint8_t* cg = g.dn_codes + row * (F / 2) + c * 16;
    const uint8_t* cg8 = cg + (size_t)8 * (F / 2);
    const uint8_t* sgp = g.dn_scales + row * (F / 16) + c * 2;
    const uint8_t* sg8p = sgp + (size_t)8 * (F / 16);
    uint4 wc[B], wc8[B];
    uint32_t ws[B], ws8[B];
#pragma unroll
    for (int i = 0; i < B; ++i) {
      wc[i] = ld_stream16(cg + i * 64);
      wc8[i] = ld_stream16(cg8 + i * 64);
      ws[i] = __ldg(reinterpret_cast<const uint16_t*>(sgp + i * 8));
      ws8[i] = __ldg(reinterpret_cast<const uint16_t*>(sg8p + i * 8));
    }

    __syncthreads();
    // stage h of the tile's positions as prescaled f16 hi + lo (two warps per position pair)
    for (int rr = warp; rr < nt; rr += kThreads / 32) {
      const float4* src = reinterpret_cast<const float4*>(g.h + (size_t)(p0 + rr) * F);
      float4 v[F / 128];
      float m = 0.f;
#pragma unroll
      for (int i = 0; i < F / 128; ++i) {
        v[i] = src[lane + 32 * i];
        m = fmaxf(m, fmaxf(fmaxf(fabsf(v[i].x), fabsf(v[i].y)), fmaxf(fabsf(v[i].z), fabsf(v[i].w))));
      }
      const int shift = prescale_shift(__reduce_max_sync(0xffffffffu, __float_as_uint(m)));
      const float sc = pow2i(shift);
#pragma unroll
      for (int i = 0; i < F / 128; ++i) {
        const int k0 = 4 * (lane + 32 * i), ch = k0 / kChunk, kp = k0 % kChunk;
        const int off = ch * kChunk * 2 + perm_off(kp / 32, (kp % 32) / 4);
        const float s0 = v[i].x * sc, s1 = v[i].y * sc, s2 = v[i].z * sc, s3 = v[i].w * sc;
        const __half2 h01 = __floats2half2_rn(s0, s1), h23 = __floats2half2_rn(s2, s3);
        const float2 r01 = __half22float2(h01), r23 = __half22float2(h23);
        const __half2 l01 = __floats2half2_rn(s0 - r01.x, s1 - r01.y);
        const __half2 l23 = __floats2half2_rn(s2 - r23.x, s3 - r23.y);
        *reinterpret_cast<uint2*>(sm + L::kHi + rr * L::kHRow + off) =
            make_uint2(*reinterpret_cast<const uint32_t*>(&h01), *reinterpret_cast<const uint32_t*>(&h23));
        *reinterpret_cast<uint2*>(sm + L::kLo + rr * L::kHRow + off) =
            make_uint2(*reinterpret_cast<const uint32_t*>(&l01), *reinterpret_cast<const uint32_t*>(&l23));
      }
      if (lane == 0) sUn[rr] = pow2i(-shift);
    }
    __syncthreads();

    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    const bool two = nt > 8;
    const uint8_t* hi0 = sm + L::kHi + gq * L::kHRow;
    const uint8_t* lo0 = sm + L::kLo + gq * L::kHRow;
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      uint4 nc[B], nc8[B];
      uint32_t ns[B], ns8[B];
      if (b + 1 < NB) {
#pragma unroll
        for (int i = 0; i < B; ++i) {
          const int ch = (b + 1) * B + i;
          nc[i] = ld_stream16(cg + ch * 64);
          nc8[i] = ld_stream16(cg8 + ch * 64);
          ns[i] = __ldg(reinterpret_cast<const uint16_t*>(sgp + ch * 8));
          ns8[i] = __ldg(reinterpret_cast<const uint16_t*>(sg8p + ch * 8));
        }
      }
#pragma unroll
      for (int i = 0; i < B; ++i) {
        const int ch = b * B + i;
        const uint32_t s2 = cvt_e4m3x2_f16x2(ws[i]), s28 = cvt_e4m3x2_f16x2(ws8[i]);
#pragma unroll
        for (int wd = 0; wd < 4; ++wd) {
          const uint32_t sg = wd < 2 ? bcast_lo(s2) : bcast_hi(s2);
          const uint32_t sg8 = wd < 2 ? bcast_lo(s28) : bcast_hi(s28);
          uint32_t afp[2][4];
          a_frag_pair(afp[0], afp[1], word_of(wc[i], wd), word_of(wc8[i], wd), sg, sg8);
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            const int kk = 2 * wd + h2;
            const int off = ch * kChunk * 2 + perm_off(c, kk);
            const uint2 bh = lds64(hi0 + off), bl = lds64(lo0 + off);
            mma_f16(acc[0], afp[h2], bh.x, bh.y);
            mma_f16(acc[0], afp[h2], bl.x, bl.y);
            if (two) {
              const uint2 bh1 = lds64(hi0 + 8 * L::kHRow + off), bl1 = lds64(lo0 + 8 * L::kHRow + off);
              mma_f16(acc[1], afp[h2], bh1.x, bh1.y);
              mma_f16(acc[1], afp[h2], bl1.x, bl1.y);
            }
          }
        }
      }
      if (b + 1 < NB) {
#pragma unroll
        for (int i = 0; i < B; ++i) {
          wc[i] = nc[i];
          wc8[i] = nc8[i];
          ws[i] = ns[i];
          ws8[i] = ns8[i];
        }
      }
    }

    const float ts = g.tsc[e * 3 + 2];
    const int r0 = warp * 16 + gq;
#pragma unroll
    for (int q = 0; q < kTok / 8; ++q) {
      const int col = q * 8 + 2 * c;
      sY[col * 132 + r0] = acc[q][0] * ts * sUn[col];
      sY[(col + 1) * 132 + r0] = acc[q][1] * ts * sUn[col + 1];
      sY[col * 132 + r0 + 8] = acc[q][2] * ts * sUn[col];
      sY[(col + 1) * 132 + r0 + 8] = acc[q][3] * ts * sUn[col + 1];
    }
    __syncthreads();
    for (int i = threadIdx.x; i < 32 * nt; i += kThreads) {
      const int q4 = i & 31, col = i >> 5;
      reinterpret_cast<float4*>(g.yexp + (size_t)(p0 + col) * d + rt * 128)[q4] =
          reinterpret_cast<const float4*>(sY + col * 132)[q4];
    }
  }
}

MmaArgs make_mma_args(const moe_ctx* c, const __nv_bfloat16* x, int T) {
  MmaArgs a;
  a.r = c->r;
  a.x = x;
  a.gu_codes = c->gu_codes;
  a.gu_scales = c->gu_scales;
  a.dn_codes = c->dn_codes;
  a.dn_scales = c->dn_scales;
  a.tsc = c->tsc;
  a.x16 = c->x16;
  a.xunshift = c->xunshift;
  a.h = c->h;
  a.yexp = c->yexp;
  a.d = c->cfg.d_model;
  a.f = c->cfg.d_ff;
  a.T = T;
  return a;
}

template <typename K>
cudaError_t set_smem(K kern, size_t bytes) {
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

size_t gu_smem(const moe_ctx* c) {
  const int na = c->cfg.n_experts + c->cfg.n_shared;
  switch (c->cfg.d_model) {
    case 256: return GuSmem<256>::bytes(na);
    case 512: return GuSmem<512>::bytes(na);
    case 1024: return GuSmem<1024>::bytes(na);
    case 2048: return GuSmem<2048>::bytes(na);
    default: return GuSmem<4096>::bytes(na);
  }
}

size_t dn_smem(const moe_ctx* c) {
  const int na = c->cfg.n_experts + c->cfg.n_shared;
  switch (c->cfg.d_ff) {
    case 128: return DnSmem<128>::bytes(na);
    case 256: return DnSmem<256>::bytes(na);
    case 512: return DnSmem<512>::bytes(na);
    default: return DnSmem<1024>::bytes(na);
  }
}

}  // namespace

bool mma_decode_supported(const moe_config& c) { return c.weight_format == MOE_W_NVFP4; }

cudaError_t prepare_mma_decode(const moe_ctx* c) {
  cudaError_t e = cudaSuccess;
  const size_t gs = gu_smem(c), ds = dn_smem(c);
  switch (c->cfg.d_model) {
    case 256: e = set_smem(gateup_mma_kernel<256>, gs); break;
    case 512: e = set_smem(gateup_mma_kernel<512>, gs); break;
    case 1024: e = set_smem(gateup_mma_kernel<1024>, gs); break;
    case 2048: e = set_smem(gateup_mma_kernel<2048>, gs); break;
    case 4096: e = set_smem(gateup_mma_kernel<4096>, gs); break;
    default: return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) return e;
  switch (c->cfg.d_ff) {
    case 128: return set_smem(down_mma_kernel<128>, ds);
    case 256: return set_smem(down_mma_kernel<256>, ds);
    case 512: return set_smem(down_mma_kernel<512>, ds);
    case 1024: return set_smem(down_mma_kernel<1024>, ds);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_mma_decode(const moe_ctx* c, const __nv_bfloat16* x, int T, cudaStream_t s) {
  const MmaArgs a = make_mma_args(c, x, T);
  xprep_kernel<<<(T + 7) / 8, 256, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int grid = 4 * c->sm_count;
  const size_t gs = gu_smem(c), ds = dn_smem(c);
  switch (a.d) {
    case 256: gateup_mma_kernel<256><<<grid, kThreads, gs, s>>>(a); break;
    case 512: gateup_mma_kernel<512><<<grid, kThreads, gs, s>>>(a); break;
    case 1024: gateup_mma_kernel<1024><<<grid, kThreads, gs, s>>>(a); break;
    case 2048: gateup_mma_kernel<2048><<<grid, kThreads, gs, s>>>(a); break;
    case 4096: gateup_mma_kernel<4096><<<grid, kThreads, gs, s>>>(a); break;
    default: return cudaErrorInvalidValue;
  }
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  switch (a.f) {
    case 128: down_mma_kernel<128><<<grid, kThreads, ds, s>>>(a); break;
    case 256: down_mma_kernel<256><<<grid, kThreads, ds, s>>>(a); break;
    case 512: down_mma_kernel<512><<<grid, kThreads, ds, s>>>(a); break;
    case 1024: down_mma_kernel<1024><<<grid, kThreads, ds, s>>>(a); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace nvmoe
