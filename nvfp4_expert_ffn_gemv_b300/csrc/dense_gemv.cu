// Streaming NVFP4 GEMV for the weights every token reads in full: the 4-bit
// output layer (lm_head) and the two dense SwiGLU FFN layers.
//
// The pages say the vendor quantised the output layer to 4 bits because, with
// only ~2.5B active parameters, it is a large share of the weights a token
// reads ("Recursive Flint 40B-A2.5B：まず速さを第一に考えて作られたコーディング
// モデル", section "量子化のレシピは最も転用しやすい部分です"), and that 2 of
// the 49 layers are dense (section "このアーキテクチャはメモリ帯域幅に関する主張
// である").  At decode both are one pass over a large NVFP4 matrix per token
// batch, so the kernel is built to keep HBM busy:
//
//   * persistent CTAs, one per SM; the matrix is cut into units of 16 rows x
//     one K slice, unit u going to CTA u % grid;
//   * warp 0 streams units with TMA bulk copies (the codes and the E4M3 scales
//     of a unit are contiguous, stored swizzled so that the consumers' reads
//     are free of bank conflicts) into a ring of up to 8 shared-memory stages;
//     consumer warp w owns stage w, so a stage is refilled as soon as its
//     warp is done with it and ~150 KB per SM stay in flight;
//   * the consumer multiplies on the tensor cores (mma.sync m16n8k16, f16 in,
//     fp32 accumulate) with exact operands: A = E2M1 code x E4M3 block scale
//     (at most 6 significant bits, exact in f16), B = the activations, bf16
//     after a per-token power-of-two prescale (exact in f16), or for the down
//     projection the fp32 hidden vector split into f16 hi + lo; every product
//     is exact, only the fp32 sums round.  Up to 32 tokens share one pass over
//     the weights (4 MMA column groups); larger batches take several passes.
//
// Epilogues: lm_head writes fp32 logits; the dense gate/up pass (tiles of 8
// gate rows + the matching 8 up rows) applies SwiGLU in registers and writes
// h (fp32); the dense down pass writes fp32 partial sums per K slice, which a
// small kernel adds in a fixed order (plus the residual) into bf16 y.
//
// Every kernel of a forward is launched with programmatic dependent launch
// (PDL): it may start while its predecessor in the stream is still running,
// and waits for it (griddepcontrol.wait) before it touches anything the
// predecessor writes.  It reads such data with plain loads, never through the
// non-coherent path (__ldg, const __restrict__): that path assumes the data is
// fixed for the kernel's whole life, and this kernel was alive while it was
// written.  The GEMV's weight stream does not depend on earlier
// kernels, so its producer warp starts filling the stage ring at once, while
// the small kernel before it (the activation prescale) still runs.
#include "internal.h"
#include "mma_frag.cuh"
#include "sm100.cuh"

namespace nvmoe {

namespace {

using namespace sm100;
using namespace frag;

constexpr int kMaxStages = 10;
constexpr int kTokPass = 32;          // tokens per pass over the weights (4 column groups of 8)
// shared-memory bytes for the stage ring: what the 227 KB of a CTA leave after
// the pair exchange buffers (kMaxStages x 4 KB) and the barriers
constexpr int kStageBudget = 190464;
// Stages (= consumer warp pairs).  The output layer runs 10 (8 -> 10: 42.7 ->
// 39.8 us at one token; its 21 warps get 80 registers a thread), and one
// kernel holds both of its consumers (a one-token kernel of its own compiled
// worse and ran 0.8 us slower).  The dense passes at one token (FMA
// consumers) run 9 (19 warps keep 96 registers; at 10 gate/up spilled and ran
// slower); the dense MMA consumers keep 8 (17 warps, 96 registers).
constexpr int kHeadStages = 10, kDenseT1Stages = 9, kMmaStages = 8;
__host__ __device__ constexpr int max_stages(int mode, bool t1) {
  return mode == 0 ? kHeadStages : (t1 ? kDenseT1Stages : kMmaStages);   // mode 0: the output layer
}
static_assert(kHeadStages <= kMaxStages && kDenseT1Stages <= kMaxStages && kMmaStages <= kMaxStages,
              "stage counts above the shared-memory plan");
static_assert(kMaxStages * 2 * 16 * 32 * 4 + 2 * kMaxStages * 8 + kStageBudget <= 227 * 1024,
              "exchange buffers, barriers and the stage ring must fit one CTA's shared memory");

enum GemvMode { kModeHead = 0, kModeGateUp = 1, kModeDown = 2 };

struct GemvArgs {
  const uint8_t* codes;    // unit (slice s, tile t): codes + s * slice_codes + t * 16 * KS / 2
  const uint8_t* scales;   //                          scales + s * slice_scales + t * 16 * KS / 16
  size_t slice_codes, slice_scales;
  int ntiles, nslices, KS;
  const uint8_t* b_hi;     // B operand [kTokPass][K] f16, prescaled, k-permuted per 128 chunk
  const uint8_t* b_lo;     // down: low halves of h (same layout); otherwise null
  int K;                   // full row length of the B operand
  const float* unshift;    // [kTokPass] 2^-prescale of each token
  int T;                   // tokens of this pass (<= kTokPass)
  float ts0, ts1;          // tensor scales (head: ts0; gate/up: ts0 gate, ts1 up; down: ts0)
  float* out;              // head [T][out_ld] logits; gate/up [T][out_ld] h; down [S][T][out_ld] partials
  uint32_t* hmax;          // gate/up: max |h| of each token (fp32 bits), folded in with atomicMax
  int out_ld;
  int nstages;             // stages = consumer warps
  int* status;
  int dbg;
  const __nv_bfloat16* x1; // head / gate/up at one token: the token's bf16 row (x in registers, FMA dot products)
  const float* h1;         // down at one token: the token's fp32 h row (FMA dot products, no hi/lo split)
};

// B operand (written by the kernel before, which may still run while this one
// starts): plain loads, never the non-coherent read-only path
__device__ __forceinline__ uint2 ldg64(const uint8_t* p) { return *reinterpret_cast<const uint2*>(p); }

__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename Kern, typename... Args>
cudaError_t launch_pdl(Kern kern, dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Stage layout of one unit: the 16 code rows (KS/2 bytes each, a multiple of
// 128) and then the 16 scale rows (KS/16 bytes each), as one bulk copy each.
// The weights are stored swizzled (see swizzle_rows_kernel): inside every
// 128-byte segment of row r, 16-byte granule i sits at granule i ^ m(r % 8),
// m(r) = 4 (r & 1) + (r >> 1).  A quarter-warp's 16-byte code loads cover
// granules {0..3} (or {4..7}) of the two rows 2i and 2i + 1, whose masks
// differ in bit 2, so they land on disjoint banks; the 8 rows of the 2-byte
// scale loads land on 8 different granules.  Scale rows are swizzled the same
// way when their length is a multiple of 128 bytes.
__host__ __device__ __forceinline__ uint32_t stage_bytes_of(int KS) { return 16u * ((uint32_t)KS / 2 + (uint32_t)KS / 16); }

__host__ __device__ __forceinline__ int swz_mask(int r8) { return ((r8 & 1) << 2) | (r8 >> 1); }

__device__ __forceinline__ int swz(int byte, int row8) {
  return (byte & ~0x7F) | ((((byte >> 4) & 7) ^ swz_mask(row8)) << 4) | (byte & 15);
}

// One unit (16 rows x one K slice) by a pair of warps: warp `half` multiplies
// the chunks of its half of the K slice.  The MMAs are spread over CH
// independent accumulator chains (by k step), so the latency of one chain does
// not serialise the unit; the down projection sends the hi and lo halves of h
// to separate chains as well.  The second warp of the pair hands its sums to
// the first through `xch` (the caller's named barrier in between); the first
// adds them and runs the epilogue.
template <int MODE, int NG>
__device__ __forceinline__ void consume_unit(const GemvArgs& g, const uint8_t* sc, const uint8_t* ss, int slice,
                                             int tile, int half, float* xch, int bar_id) {
  constexpr int CH = NG >= 4 ? 1 : (NG == 2 ? 2 : 4);
  const int lane = threadIdx.x & 31, gq = lane >> 2, c = lane & 3;
  const int KS = g.KS;
  const int CB = KS / 2, SB = KS / 16;
  const bool sswz = (SB & 127) == 0;     // scale rows swizzled too
  float acc[CH][NG][4];
  float accl[MODE == kModeDown ? CH : 1][MODE == kModeDown ? NG : 1][4];
#pragma unroll
  for (int h = 0; h < CH; ++h)
#pragma unroll
    for (int q = 0; q < NG; ++q) {
      acc[h][q][0] = acc[h][q][1] = acc[h][q][2] = acc[h][q][3] = 0.f;
      if (MODE == kModeDown) accl[h][q][0] = accl[h][q][1] = accl[h][q][2] = accl[h][q][3] = 0.f;
    }
  const uint8_t* row0 = sc + gq * CB;
  const uint8_t* row8 = row0 + 8 * CB;
  const uint8_t* srow0 = ss + gq * SB;
  const uint8_t* srow8 = srow0 + 8 * SB;
  const size_t brow = (size_t)g.K * 2;
  const int k0 = slice * KS;     // first k of this unit in the B operand
  const int nch = KS / 128, ch0 = half ? nch / 2 : 0, ch1 = half ? nch : nch / 2;
  // the next chunk's code words and scales are loaded one chunk ahead
  auto load_a = [&](int ch, uint4& w, uint4& w8, uint32_t& sr, uint32_t& sr8) {
    const int cb = swz(ch * 64 + c * 16, gq);                       // rows gq and gq + 8: same r % 8
    const int sb = sswz ? swz(ch * 8 + c * 2, gq) : ch * 8 + c * 2;
    w = *reinterpret_cast<const uint4*>(row0 + cb);
    w8 = *reinterpret_cast<const uint4*>(row8 + cb);
    sr = *reinterpret_cast<const uint16_t*>(srow0 + sb);
    sr8 = *reinterpret_cast<const uint16_t*>(srow8 + sb);
  };
  uint4 nwc, nwc8;
  uint32_t nsr, nsr8;
  load_a(ch0, nwc, nwc8, nsr, nsr8);
  for (int ch = ch0; ch < ch1; ++ch) {
    const uint4 wc = nwc, wc8 = nwc8;
    const uint32_t s2 = cvt_e4m3x2_f16x2(nsr), s28 = cvt_e4m3x2_f16x2(nsr8);
    if (ch + 1 < ch1) load_a(ch + 1, nwc, nwc8, nsr, nsr8);
    const size_t boff = (size_t)(k0 + ch * 128) * 2;
#pragma unroll
    for (int wd = 0; wd < 4; ++wd) {
      const uint32_t sg = wd < 2 ? bcast_lo(s2) : bcast_hi(s2);
      const uint32_t sg8 = wd < 2 ? bcast_lo(s28) : bcast_hi(s28);
      uint32_t afp[2][4];
      a_frag_pair(afp[0], afp[1], word_of(wc, wd), word_of(wc8, wd), sg, sg8);
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        const int kk = 2 * wd + h2;
        const int chn = kk % CH;
#pragma unroll
        for (int q = 0; q < NG; ++q) {
          // B column gq of group q is token 8q + gq: lanes past the batch feed zeros without a load
          const bool live = 8 * q + gq < g.T;
          const size_t off = (size_t)(8 * q + gq) * brow + boff + perm_off(c, kk);
          const uint2 b = live ? ldg64(g.b_hi + off) : make_uint2(0u, 0u);
          mma_f16(acc[chn][q], afp[h2], b.x, b.y);
          if (MODE == kModeDown) {
            const uint2 bl = live ? ldg64(g.b_lo + off) : make_uint2(0u, 0u);
            mma_f16(accl[chn % (MODE == kModeDown ? CH : 1)][q % (MODE == kModeDown ? NG : 1)], afp[h2], bl.x, bl.y);
          }
        }
      }
    }
  }
#pragma unroll
  for (int h = 1; h < CH; ++h)
#pragma unroll
    for (int q = 0; q < NG; ++q)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[0][q][i] += acc[h][q][i];
  if (MODE == kModeDown) {
#pragma unroll
    for (int h = 0; h < CH; ++h)
#pragma unroll
      for (int q = 0; q < NG; ++q)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[0][q][i] += accl[h % (MODE == kModeDown ? CH : 1)][q % (MODE == kModeDown ? NG : 1)][i];
  }
  // the pair's sums meet: the second warp writes, the first adds (fixed order: first + second)
  if (half) {
#pragma unroll
    for (int q = 0; q < NG; ++q)
#pragma unroll
      for (int i = 0; i < 4; ++i) xch[(q * 4 + i) * 32 + lane] = acc[0][q][i];
  }
  asm volatile("bar.sync %0, 64;" :: "r"(bar_id) : "memory");
  if (half) return;
#pragma unroll
  for (int q = 0; q < NG; ++q)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[0][q][i] += xch[(q * 4 + i) * 32 + lane];
  // lanes hold rows gq (acc 0, 1) and gq + 8 (acc 2, 3) of the tile, tokens 8q + 2c, 8q + 2c + 1
#pragma unroll
  for (int q = 0; q < NG; ++q) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int t = 8 * q + 2 * c + j;
      if (t >= g.T) continue;
      const float un = g.unshift[t];
      if (MODE == kModeHead) {
        const int r = tile * 16 + gq;
        g.out[(size_t)t * g.out_ld + r] = acc[0][q][j] * g.ts0 * un;
        g.out[(size_t)t * g.out_ld + r + 8] = acc[0][q][2 + j] * g.ts0 * un;
      } else if (MODE == kModeGateUp) {
        const float gv = acc[0][q][j] * g.ts0 * un, uv = acc[0][q][2 + j] * g.ts1 * un;
        g.out[(size_t)t * g.out_ld + tile * 8 + gq] = silu_f(gv) * uv;
      } else {
        float* dst = g.out + ((size_t)slice * g.T + t) * g.out_ld + tile * 16 + gq;
        dst[0] = acc[0][q][j] * g.ts0 * un;
        dst[8] = acc[0][q][2 + j] * g.ts0 * un;
      }
    }
  }
  if (MODE == kModeGateUp) {
    // max |h| per token over this unit's 8 hidden units (the 8 lanes gq of each
    // c hold them), folded into the token's word; NaN is left out, as fmaxf does
#pragma unroll
    for (int q = 0; q < NG; ++q)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int t = 8 * q + 2 * c + j;
        float a = 0.f;
        if (t < g.T) {
          const float hv = silu_f(acc[0][q][j] * g.ts0 * g.unshift[t]) * (acc[0][q][2 + j] * g.ts1 * g.unshift[t]);
          a = fabsf(hv) == fabsf(hv) ? fabsf(hv) : 0.f;
        }
        uint32_t m = __float_as_uint(a);
        m = max(m, __shfl_xor_sync(0xffffffffu, m, 4));
        m = max(m, __shfl_xor_sync(0xffffffffu, m, 8));
        m = max(m, __shfl_xor_sync(0xffffffffu, m, 16));
        if (gq == 0 && t < g.T && m != 0u) atomicMax(g.hmax + t, m);
      }
  }
}

// One token through the output layer.  The MMA path would use one of the
// eight B columns of every m16n8k16, so here each warp of the stage's pair
// takes 8 of the unit's 16 rows whole: lane l holds the token's x for the
// 32-column chunks j = l + 32q (exact f16 after its power-of-two prescale, as
// the MMA path's B operand) and forms each row's partial dot with the
// mixed-precision FMA (E2M1 code as exact f16 x f16 x + fp32; the block scale
// applied once per 16 products).  The 8 row partials are summed over the
// warp with a transposing reduction (9 shuffles), then lane 4r writes row r.
__device__ __forceinline__ void fma2_mixed(uint32_t a, uint32_t b, float& acc, float& acc2) {
  asm("{\n\t.reg .f16 al, ah, bl, bh;\n\tmov.b32 {al, ah}, %2;\n\tmov.b32 {bl, bh}, %3;\n\t"
      "fma.rn.f32.f16 %0, al, bl, %0;\n\tfma.rn.f32.f16 %1, ah, bh, %1;\n\t}"
      : "+f"(acc), "+f"(acc2) : "r"(a), "r"(b));
}

template <int CPL>
__device__ __forceinline__ void load_x1(const GemvArgs& g, uint32_t (&xh)[CPL][16]) {
  const int lane = threadIdx.x & 31;
  const float sc = 1.f / g.unshift[0];   // a power of two
#pragma unroll
  for (int q = 0; q < CPL; ++q) {
    const uint4* src = reinterpret_cast<const uint4*>(g.x1 + (size_t)(lane + 32 * q) * 32);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 v = src[i];
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        const __half2 hh = __floats2half2_rn(__uint_as_float(w[p] << 16) * sc, __uint_as_float(w[p] & 0xFFFF0000u) * sc);
        xh[q][4 * i + p] = *reinterpret_cast<const uint32_t*>(&hh);
      }
    }
  }
}

template <int CPL>
__device__ __forceinline__ void consume_unit_t1_head(const GemvArgs& g, const uint8_t* sc, const uint8_t* ss, int tile,
                                                int half, const uint32_t (&xh)[CPL][16], int bar_id) {
  const int lane = threadIdx.x & 31;
  const int CB = g.KS / 2, SB = g.KS / 16;
  const bool sswz = (SB & 127) == 0;
  float v[8];
#pragma unroll
  for (int rr = 0; rr < 8; ++rr) {
    const int r = half * 8 + rr;
    const uint8_t* crow = sc + r * CB;
    const uint8_t* srow = ss + r * SB;
    float dot = 0.f;
#pragma unroll
    for (int q = 0; q < CPL; ++q) {
      const int j = lane + 32 * q;
      const uint4 cw = *reinterpret_cast<const uint4*>(crow + swz(j * 16, r & 7));
      const uint32_t ws[4] = {cw.x, cw.y, cw.z, cw.w};
      float b[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        uint32_t o[4];
        cvt_e2m1x8(ws[w], o);
#pragma unroll
        for (int p = 0; p < 4; ++p) fma2_mixed(o[p], xh[q][4 * w + p], b[w >> 1][0], b[w >> 1][1]);
      }
      const int sb = sswz ? swz(2 * j, r & 7) : 2 * j;
      const float2 s01 = e4m3x2_to_f32x2(*reinterpret_cast<const uint16_t*>(srow + sb));
      dot = fmaf(b[0][0] + b[0][1], s01.x, dot);
      dot = fmaf(b[1][0] + b[1][1], s01.y, dot);
    }
    v[rr] = dot;
  }
  // transposing sum over the warp: after the xor-16, -8 and -4 steps lane l
  // holds a partial of row (l >> 2) & 7, completed by the xor-2 and -1 steps
  const int b4 = (lane >> 4) & 1, b3 = (lane >> 3) & 1, b2 = (lane >> 2) & 1;
  float w4[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float keep = b4 ? v[i + 4] : v[i], send = b4 ? v[i] : v[i + 4];
    w4[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
  }
  float w2[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float keep = b3 ? w4[i + 2] : w4[i], send = b3 ? w4[i] : w4[i + 2];
    w2[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
  }
  float t = (b2 ? w2[1] : w2[0]) + __shfl_xor_sync(0xffffffffu, b2 ? w2[0] : w2[1], 4);
  t += __shfl_xor_sync(0xffffffffu, t, 2);
  t += __shfl_xor_sync(0xffffffffu, t, 1);
  if ((lane & 3) == 0) g.out[tile * 16 + half * 8 + (lane >> 2)] = t * g.ts0 * g.unshift[0];
  // both warps of the pair are done with the stage before the first one releases it
  asm volatile("bar.sync %0, 64;" :: "r"(bar_id) : "memory");
}

template <int MODE, int CPL>
__device__ __forceinline__ void consume_unit_t1(const GemvArgs& g, const uint8_t* sc, const uint8_t* ss, int tile,
                                                int half, const uint32_t (&xh)[CPL][16], float* xch, int bar_id) {
  const int lane = threadIdx.x & 31;
  const int CB = g.KS / 2, SB = g.KS / 16;
  const bool sswz = (SB & 127) == 0;
  float v[8];
#pragma unroll
  for (int rr = 0; rr < 8; ++rr) {
    const int r = half * 8 + rr;
    const uint8_t* crow = sc + r * CB;
    const uint8_t* srow = ss + r * SB;
    float dot = 0.f;
#pragma unroll
    for (int q = 0; q < CPL; ++q) {
      const int j = lane + 32 * q;
      const uint4 cw = *reinterpret_cast<const uint4*>(crow + swz(j * 16, r & 7));
      const uint32_t ws[4] = {cw.x, cw.y, cw.z, cw.w};
      float b[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        uint32_t o[4];
        cvt_e2m1x8(ws[w], o);
#pragma unroll
        for (int p = 0; p < 4; ++p) fma2_mixed(o[p], xh[q][4 * w + p], b[w >> 1][0], b[w >> 1][1]);
      }
      const int sb = sswz ? swz(2 * j, r & 7) : 2 * j;
      const float2 s01 = e4m3x2_to_f32x2(*reinterpret_cast<const uint16_t*>(srow + sb));
      dot = fmaf(b[0][0] + b[0][1], s01.x, dot);
      dot = fmaf(b[1][0] + b[1][1], s01.y, dot);
    }
    v[rr] = dot;
  }
  // transposing sum over the warp: after the xor-16, -8 and -4 steps lane l
  // holds a partial of row (l >> 2) & 7, completed by the xor-2 and -1 steps
  const int b4 = (lane >> 4) & 1, b3 = (lane >> 3) & 1, b2 = (lane >> 2) & 1;
  float w4[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float keep = b4 ? v[i + 4] : v[i], send = b4 ? v[i] : v[i + 4];
    w4[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
  }
  float w2[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float keep = b3 ? w4[i + 2] : w4[i], send = b3 ? w4[i] : w4[i + 2];
    w2[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
  }
  float t = (b2 ? w2[1] : w2[0]) + __shfl_xor_sync(0xffffffffu, b2 ? w2[0] : w2[1], 4);
  t += __shfl_xor_sync(0xffffffffu, t, 2);
  t += __shfl_xor_sync(0xffffffffu, t, 1);
  // dense gate/up: warp 0 of the pair has the gate rows, warp 1 the up rows of
  // hidden units tile * 8 + r; they meet in shared memory for SwiGLU
  if (half && (lane & 3) == 0) xch[lane >> 2] = t;
  asm volatile("bar.sync %0, 64;" :: "r"(bar_id) : "memory");
  if (half) return;
  const float un = g.unshift[0];
  float a = 0.f;
  if ((lane & 3) == 0) {
    const float hv = silu_f(t * g.ts0 * un) * (xch[lane >> 2] * g.ts1 * un);
    g.out[tile * 8 + (lane >> 2)] = hv;
    a = fabsf(hv) == fabsf(hv) ? fabsf(hv) : 0.f;   // NaN left out of max |h|, as fmaxf does
  }
  uint32_t m = __float_as_uint(a);
  m = max(m, __shfl_xor_sync(0xffffffffu, m, 4));
  m = max(m, __shfl_xor_sync(0xffffffffu, m, 8));
  m = max(m, __shfl_xor_sync(0xffffffffu, m, 16));
  if (lane == 0 && m != 0u) atomicMax(g.hmax, m);
}

// The consumer loops of stage s (warps 2s + 1 and 2s + 2, one per half).  Both
// warps of the pair take the same path (the wait outcome is shared through the
// barrier count only when both run): a failed wait skips nothing but is reported.
template <int MODE>
__device__ __forceinline__ bool consume_loop(const GemvArgs& g, const uint8_t* gsm, uint32_t stage_bytes,
                                          uint32_t scale_off, uint64_t* full_bar, uint64_t* empty_bar,
                                          float (*xch_all)[2][16 * 32], int s, int half, int units) {
  const int lane = threadIdx.x & 31, NS = g.nstages;
  bool ok = true;
  int j = s;
  for (int u = blockIdx.x + s * gridDim.x; u < units; u += NS * gridDim.x, j += NS) {
    if (!wait_parity(&full_bar[s], (j / NS) & 1)) ok = false;
    const uint8_t* sc = gsm + (size_t)s * stage_bytes;
    const int slice = u / g.ntiles, tile = u % g.ntiles;
    const int ngroups = (g.T + 7) / 8;
    float* xch = xch_all[s][(j / NS) & 1];
    if (ngroups <= 1) consume_unit<MODE, 1>(g, sc, sc + scale_off, slice, tile, half, xch, s + 1);
    else if (ngroups == 2) consume_unit<MODE, 2>(g, sc, sc + scale_off, slice, tile, half, xch, s + 1);
    else consume_unit<MODE, 4>(g, sc, sc + scale_off, slice, tile, half, xch, s + 1);
    __syncwarp();
    if (lane == 0 && half == 0) mbar_arrive(&empty_bar[s]);
  }
  return ok;
}

template <int CPL>
__device__ __noinline__ bool consume_loop_t1_head(const GemvArgs& g, const uint8_t* gsm, uint32_t stage_bytes,
                                                  uint32_t scale_off, uint64_t* full_bar, uint64_t* empty_bar, int s,
                                                  int half, int units) {
  const int lane = threadIdx.x & 31, NS = g.nstages;
  uint32_t xh[CPL][16];
  load_x1<CPL>(g, xh);
  bool ok = true;
  int j = s;
  for (int u = blockIdx.x + s * gridDim.x; u < units; u += NS * gridDim.x, j += NS) {
    if (!wait_parity(&full_bar[s], (j / NS) & 1)) ok = false;
    const uint8_t* sc = gsm + (size_t)s * stage_bytes;
    consume_unit_t1_head<CPL>(g, sc, sc + scale_off, u % g.ntiles, half, xh, s + 1);
    __syncwarp();
    if (lane == 0 && half == 0) mbar_arrive(&empty_bar[s]);
  }
  return ok;
}

template <int MODE, int CPL>
__device__ __noinline__ bool consume_loop_t1(const GemvArgs& g, const uint8_t* gsm, uint32_t stage_bytes,
                                             uint32_t scale_off, uint64_t* full_bar, uint64_t* empty_bar,
                                             float (*xch_all)[2][16 * 32], int s, int half, int units) {
  const int lane = threadIdx.x & 31, NS = g.nstages;
  uint32_t xh[CPL][16];
  load_x1<CPL>(g, xh);
  bool ok = true;
  int j = s;
  for (int u = blockIdx.x + s * gridDim.x; u < units; u += NS * gridDim.x, j += NS) {
    if (!wait_parity(&full_bar[s], (j / NS) & 1)) ok = false;
    const uint8_t* sc = gsm + (size_t)s * stage_bytes;
    float* xch = nullptr;
    if constexpr (MODE == kModeGateUp) xch = xch_all[s][(j / NS) & 1];
    consume_unit_t1<MODE, CPL>(g, sc, sc + scale_off, u % g.ntiles, half, xh, xch, s + 1);
    __syncwarp();
    if (lane == 0 && half == 0) mbar_arrive(&empty_bar[s]);
  }
  return ok;
}

// One token through the dense down projection (K slices of 2048): each warp
// of the pair takes one half of the unit's slice for all 16 rows, with that
// half of h (fp32, 32 values a lane) in registers, requested before the
// stage wait.  A code is expanded to exact f16 by the hardware cvt and then
// to fp32, so each product is one fp32 FMA with h (the MMA path splits h into
// f16 hi + lo instead); the block scale multiplies each 16-term partial.  The
// rows are summed over the warp in two groups of 8 (9 shuffles each), the pair
// adds its halves through shared memory (first + second), and warp 0 writes
// the slice's partial outputs.
__device__ __forceinline__ void consume_unit_t1_down(const GemvArgs& g, const uint8_t* sc, const uint8_t* ss,
                                                     int slice, int tile, int half, const float (&hv)[32],
                                                     float* xch, int bar_id) {
  const int lane = threadIdx.x & 31;
  constexpr int CB = 1024, SB = 128;   // code / scale bytes of a 2048-wide row
  const int b4 = (lane >> 4) & 1, b3 = (lane >> 3) & 1, b2 = (lane >> 2) & 1;
  float t2[2];
#pragma unroll
  for (int grp = 0; grp < 2; ++grp) {
    float v[8];
#pragma unroll
    for (int rr = 0; rr < 8; ++rr) {
      const int r = grp * 8 + rr;
      const uint4 cw = *reinterpret_cast<const uint4*>(sc + r * CB + swz(half * 512 + lane * 16, r & 7));
      const float2 s01 =
          e4m3x2_to_f32x2(*reinterpret_cast<const uint16_t*>(ss + r * SB + swz(half * 64 + lane * 2, r & 7)));
      const uint32_t ws[4] = {cw.x, cw.y, cw.z, cw.w};
      float b[2] = {0.f, 0.f};
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        uint32_t o[4];
        cvt_e2m1x8(ws[w], o);
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          const float2 f = f16x2_to_f32x2(o[p]);
          b[w >> 1] = fmaf(f.x, hv[8 * w + 2 * p], b[w >> 1]);
          b[w >> 1] = fmaf(f.y, hv[8 * w + 2 * p + 1], b[w >> 1]);
        }
      }
      v[rr] = fmaf(b[0], s01.x, b[1] * s01.y);
    }
    // transposing sum over the warp (as the output layer's): lane 4r ends with row grp * 8 + r
    float w4[4], w2[2];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      w4[i] = (b4 ? v[i + 4] : v[i]) + __shfl_xor_sync(0xffffffffu, b4 ? v[i] : v[i + 4], 16);
#pragma unroll
    for (int i = 0; i < 2; ++i)
      w2[i] = (b3 ? w4[i + 2] : w4[i]) + __shfl_xor_sync(0xffffffffu, b3 ? w4[i] : w4[i + 2], 8);
    float t = (b2 ? w2[1] : w2[0]) + __shfl_xor_sync(0xffffffffu, b2 ? w2[0] : w2[1], 4);
    t += __shfl_xor_sync(0xffffffffu, t, 2);
    t += __shfl_xor_sync(0xffffffffu, t, 1);
    t2[grp] = t;
    asm volatile("" ::: "memory");   // the second group's loads after the first group's sums
  }
  if (half && (lane & 3) == 0) {
    xch[lane >> 2] = t2[0];
    xch[8 + (lane >> 2)] = t2[1];
  }
  asm volatile("bar.sync %0, 64;" :: "r"(bar_id) : "memory");
  if (!half && (lane & 3) == 0) {
    float* dst = g.out + (size_t)slice * g.out_ld + tile * 16 + (lane >> 2);
    dst[0] = (t2[0] + xch[lane >> 2]) * g.ts0;
    dst[8] = (t2[1] + xch[8 + (lane >> 2)]) * g.ts0;
  }
}

__device__ __noinline__ bool consume_loop_t1_down(const GemvArgs& g, const uint8_t* gsm, uint32_t stage_bytes,
                                                  uint32_t scale_off, uint64_t* full_bar, uint64_t* empty_bar,
                                                  float (*xch_all)[2][16 * 32], int s, int half, int units) {
  const int lane = threadIdx.x & 31, NS = g.nstages;
  bool ok = true;
  int j = s;
  for (int u = blockIdx.x + s * gridDim.x; u < units; u += NS * gridDim.x, j += NS) {
    const int slice = u / g.ntiles, tile = u % g.ntiles;
    float hv[32];
    const float4* hp = reinterpret_cast<const float4*>(g.h1 + (size_t)slice * 2048 + half * 1024 + lane * 32);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float4 q = hp[i];
      hv[4 * i] = q.x;
      hv[4 * i + 1] = q.y;
      hv[4 * i + 2] = q.z;
      hv[4 * i + 3] = q.w;
    }
    if (!wait_parity(&full_bar[s], (j / NS) & 1)) ok = false;
    const uint8_t* sc = gsm + (size_t)s * stage_bytes;
    consume_unit_t1_down(g, sc, sc + scale_off, slice, tile, half, hv, xch_all[s][(j / NS) & 1], s + 1);
    __syncwarp();
    if (lane == 0 && half == 0) mbar_arrive(&empty_bar[s]);
  }
  return ok;
}

// T1: one token through the dense gate/up pass (d_model 1024 or 2048) or the
// dense down pass (K slices of 2048) on the FMA consumers.  The output layer
// picks its consumer at run time instead.
template <int MODE, bool T1>
__global__ void __launch_bounds__(32 * (2 * max_stages(MODE, T1) + 1), 1) nvfp4_gemv_kernel(GemvArgs g) {
  extern __shared__ __align__(128) uint8_t gsm[];
  __shared__ __align__(8) uint64_t full_bar[max_stages(MODE, T1)], empty_bar[max_stages(MODE, T1)];
  // partial sums a warp pair exchanges: [stage][unit parity][16 values][32 lanes]
  __shared__ float xch_all[max_stages(MODE, T1)][2][16 * 32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NS = g.nstages;
  const uint32_t rcodes = (uint32_t)g.KS / 2, rscales = (uint32_t)g.KS / 16;     // bytes per row
  const uint32_t stage_bytes = stage_bytes_of(g.KS), scale_off = 16 * rcodes;
  const int units = g.ntiles * g.nslices;
  griddep_launch();
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    fence_barrier_init();
  }
  __syncthreads();
  bool ok = true;
  if (warp == 0) {
    // the weights were written at init: no wait on the previous kernel
    if (lane == 0) {
      int j = 0;
      for (int u = blockIdx.x; u < units; u += gridDim.x, ++j) {
        const int s = j % NS;
        if (j >= NS && !wait_parity(&empty_bar[s], ((j / NS) - 1) & 1)) { ok = false; break; }
        const int slice = u / g.ntiles, tile = u % g.ntiles;
        uint8_t* dst = gsm + (size_t)s * stage_bytes;
        mbar_arrive_expect_tx(&full_bar[s], stage_bytes);
        bulk_load(dst, g.codes + slice * g.slice_codes + (size_t)tile * 16 * rcodes, 16 * rcodes, &full_bar[s]);
        bulk_load(dst + scale_off, g.scales + slice * g.slice_scales + (size_t)tile * 16 * rscales, 16 * rscales,
                  &full_bar[s]);
      }
    }
    // every copy issued here lands before the consumer that owns its stage
    // finishes, and the CTA leaves only after all consumers (below)
  } else if (warp - 1 < 2 * NS) {
    // warps 2s + 1 and 2s + 2 share stage s, each on one half of the K slice;
    // the activations and every output buffer belong to the previous kernels
    griddep_wait();
    const int s = (warp - 1) >> 1, half = (warp - 1) & 1;
    const bool head_t1 = MODE == kModeHead && g.T == 1 && g.x1 != nullptr && g.nslices == 1;
    if constexpr (MODE == kModeHead) {
      if (head_t1 && g.KS == 2048)
        ok = consume_loop_t1_head<2>(g, gsm, stage_bytes, scale_off, full_bar, empty_bar, s, half, units);
      else if (head_t1 && g.KS == 1024)
        ok = consume_loop_t1_head<1>(g, gsm, stage_bytes, scale_off, full_bar, empty_bar, s, half, units);
      else
        ok = consume_loop<MODE>(g, gsm, stage_bytes, scale_off, full_bar, empty_bar, xch_all, s, half, units);
    } else if constexpr (T1 && MODE == kModeDown) {
      ok = consume_loop_t1_down(g, gsm, stage_bytes, scale_off, full_bar, empty_bar, xch_all, s, half, units);
    } else if constexpr (T1 && MODE == kModeGateUp) {
      if (g.KS == 2048)
        ok = consume_loop_t1<MODE, 2>(g, gsm, stage_bytes, scale_off, full_bar, empty_bar, xch_all, s, half, units);
      else
        ok = consume_loop_t1<MODE, 1>(g, gsm, stage_bytes, scale_off, full_bar, empty_bar, xch_all, s, half, units);
    } else {
      ok = consume_loop<MODE>(g, gsm, stage_bytes, scale_off, full_bar, empty_bar, xch_all, s, half, units);
    }
  }
  if (!ok) latch_status(g.status, MOE_ERR_TIMEOUT);
  __syncthreads();
  if (threadIdx.x == 0 && (g.dbg & MOE_DEBUG_FORCE_TIMEOUT)) latch_status(g.status, MOE_ERR_TIMEOUT);
}

// Rows of the B operand a pass over T tokens reads: whole groups of 8 tokens
// (1, 2 or 4 groups).
__host__ __device__ __forceinline__ int rows_read(int T) {
  const int ng = (T + 7) / 8;
  return ng <= 2 ? 8 * ng : kTokPass;
}

// Block-wide maximum of non-negative floats (as ordered bit patterns) of 256 threads.
__device__ __forceinline__ float block_max256(float m, uint32_t* red) {
  const uint32_t w = __reduce_max_sync(0xffffffffu, __float_as_uint(m));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = w;
  __syncthreads();
  const uint32_t v = __reduce_max_sync(0xffffffffu, red[threadIdx.x & 7]);   // every warp sees all 8
  return __uint_as_float(v);
}

// bf16 x [T][K] -> prescaled f16 in the permuted chunk order, one CTA per row
// of the B operand (rows T .. rows_read(T) - 1 zero); unshift[t] = 2^-shift.
__global__ void __launch_bounds__(256) prep_x_kernel(const __nv_bfloat16* x, int T, int K, uint8_t* out,
                                                     float* unshift, uint32_t* hmax) {
  __shared__ uint32_t red[8];
  griddep_launch();
  griddep_wait();
  const int t = blockIdx.x;
  if (hmax && threadIdx.x == 0) hmax[t] = 0u;   // the dense FFN's gate/up pass folds max |h| in here
  uint8_t* dst = out + (size_t)t * K * 2;
  if (t >= T) {
    for (int i = threadIdx.x; i < K / 8; i += 256) reinterpret_cast<uint4*>(dst)[i] = make_uint4(0u, 0u, 0u, 0u);
    if (threadIdx.x == 0) unshift[t] = 0.f;
    return;
  }
  const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * K);
  float m = 0.f;
  for (int i = threadIdx.x; i < K / 8; i += 256) {
    const uint4 v = src[i];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q)
      m = fmaxf(m, fmaxf(fabsf(__uint_as_float(w[q] << 16)), fabsf(__uint_as_float(w[q] & 0xFFFF0000u))));
  }
  const int shift = prescale_shift(__float_as_uint(block_max256(m, red)));
  const float sc = pow2i(shift);
  for (int i = threadIdx.x; i < K / 8; i += 256) {
    const uint4 v = src[i];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t hv[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const __half2 hh = __floats2half2_rn(__uint_as_float(w[q] << 16) * sc, __uint_as_float(w[q] & 0xFFFF0000u) * sc);
      hv[q] = *reinterpret_cast<const uint32_t*>(&hh);
    }
    const int k0 = 8 * i, kp = k0 % 128, cc = kp / 32, kk = (kp % 32) / 4;
    uint8_t* base = dst + (size_t)(k0 / 128) * 256;
    *reinterpret_cast<uint2*>(base + perm_off(cc, kk)) = make_uint2(hv[0], hv[1]);
    *reinterpret_cast<uint2*>(base + perm_off(cc, kk + 1)) = make_uint2(hv[2], hv[3]);
  }
  if (threadIdx.x == 0) unshift[t] = pow2i(-shift);
}

// fp32 h [T][K] -> prescaled f16 hi + lo in the permuted chunk order.  The
// prescale comes from the token's max |h|, which the gate/up pass folded into
// hmax[t], so a row is split over K / 2048 CTAs (blockIdx.x = chunk,
// blockIdx.y = row; rows T.. are zero).
constexpr int kPrepHChunk = 2048;
__global__ void __launch_bounds__(256) prep_h_kernel(const float* h, int T, int K, const uint32_t* hmax,
                                                     uint8_t* hi, uint8_t* lo, float* unshift) {
  griddep_launch();
  griddep_wait();
  const int t = blockIdx.y;
  const int i0 = blockIdx.x * (kPrepHChunk / 4), i1 = min(K / 4, i0 + kPrepHChunk / 4);
  uint8_t* dh = hi + (size_t)t * K * 2;
  uint8_t* dl = lo + (size_t)t * K * 2;
  if (t >= T) {
    for (int i = i0 + (int)threadIdx.x; i < i1; i += 256) {
      const int k0 = 4 * i, kp = k0 % 128;
      const size_t off = (size_t)(k0 / 128) * 256 + perm_off(kp / 32, (kp % 32) / 4);
      *reinterpret_cast<uint2*>(dh + off) = make_uint2(0u, 0u);
      *reinterpret_cast<uint2*>(dl + off) = make_uint2(0u, 0u);
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) unshift[t] = 0.f;
    return;
  }
  const int shift = prescale_shift(hmax[t]);
  const float sc = pow2i(shift);
  const float4* src = reinterpret_cast<const float4*>(h + (size_t)t * K);
  for (int i = i0 + (int)threadIdx.x; i < i1; i += 256) {
    const float4 v = src[i];
    uint2 vh, vl;
    split_hi_lo(v.x * sc, v.y * sc, v.z * sc, v.w * sc, vh, vl);
    const int k0 = 4 * i, kp = k0 % 128;
    const size_t off = (size_t)(k0 / 128) * 256 + perm_off(kp / 32, (kp % 32) / 4);
    *reinterpret_cast<uint2*>(dh + off) = vh;
    *reinterpret_cast<uint2*>(dl + off) = vl;
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) unshift[t] = pow2i(-shift);
}

// y[t][r] = bf16(sum over the S K slices, in order, of partial[s][t][r] (+ x[t][r]))
__global__ void __launch_bounds__(256) reduce_down_kernel(const float* part, int S, int T, int d,
                                                          const __nv_bfloat16* x, int residual, __nv_bfloat16* y) {
  griddep_launch();
  griddep_wait();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= T * d) return;
  float acc = 0.f;
  for (int s = 0; s < S; ++s) acc += part[(size_t)s * T * d + i];
  if (residual) acc += __bfloat162float(x[i]);
  y[i] = __float2bfloat16_rn(acc);
}

// In place, one block per row of row_bytes (a multiple of 128): granule i of
// every 128-byte segment of row r moves to granule i ^ m(r % 8).
__global__ void swizzle_rows_kernel(uint8_t* __restrict__ buf, size_t row_bytes) {
  extern __shared__ __align__(16) uint8_t row_sm[];
  const size_t r = blockIdx.x;
  uint4* row = reinterpret_cast<uint4*>(buf + r * row_bytes);
  uint4* tmp = reinterpret_cast<uint4*>(row_sm);
  const int n = (int)(row_bytes / 16);
  for (int i = threadIdx.x; i < n; i += blockDim.x) tmp[i] = row[i];
  __syncthreads();
  const int m = swz_mask((int)(r & 7));
  for (int i = threadIdx.x; i < n; i += blockDim.x) row[(i & ~7) | ((i & 7) ^ m)] = tmp[i];
}

cudaError_t swizzle_rows(uint8_t* buf, size_t rows, size_t row_bytes) {
  if (row_bytes % 128 != 0 || rows == 0) return cudaSuccess;
  swizzle_rows_kernel<<<(unsigned)rows, 128, row_bytes>>>(buf, row_bytes);
  return cudaGetLastError();
}

// gate/up [f][K] canonical -> tiles of 8 gate rows then the matching 8 up rows
__global__ void interleave_gu_kernel(const uint8_t* __restrict__ gsrc, const uint8_t* __restrict__ usrc,
                                     size_t row_bytes, int f, uint8_t* __restrict__ dst) {
  const int r = blockIdx.x;        // destination row 0 .. 2f-1
  const int tile = r / 16, w = r % 16;
  const uint8_t* src = (w < 8 ? gsrc : usrc) + (size_t)(tile * 8 + (w & 7)) * row_bytes;
  for (size_t i = threadIdx.x; i < row_bytes; i += blockDim.x) dst[(size_t)r * row_bytes + i] = src[i];
}

// W_down [d][f] canonical -> K slices [S][d][KS] (codes KS/2 or scales KS/16 bytes per row and slice)
__global__ void slice_rows_kernel(const uint8_t* __restrict__ src, int d, size_t row_bytes, int S,
                                  uint8_t* __restrict__ dst) {
  const int r = blockIdx.x, s = blockIdx.y;
  const size_t sb = row_bytes / S;
  for (size_t i = threadIdx.x; i < sb; i += blockDim.x)
    dst[((size_t)s * d + r) * sb + i] = src[(size_t)r * row_bytes + (size_t)s * sb + i];
}

int stages_for(int KS, int mode, bool t1) {
  const int cap = max_stages(mode, t1);
  const int n = kStageBudget / (int)stage_bytes_of(KS);
  return n > cap ? cap : n;
}

size_t gemv_smem(int KS, int mode, bool t1) { return (size_t)stages_for(KS, mode, t1) * stage_bytes_of(KS); }

template <int MODE>
cudaError_t launch_gemv(GemvArgs g, int sm_count, cudaStream_t s) {
  const int units = g.ntiles * g.nslices;
  const int grid = units < sm_count ? units : sm_count;
  if constexpr (MODE == kModeDown) {
    if (g.T == 1 && g.h1 != nullptr && g.KS == 2048) {
      g.nstages = stages_for(g.KS, MODE, true);
      return launch_pdl(nvfp4_gemv_kernel<MODE, true>, dim3(grid), dim3(32 * (2 * g.nstages + 1)),
                        gemv_smem(g.KS, MODE, true), s, g);
    }
  }
  if constexpr (MODE == kModeGateUp) {
    if (g.T == 1 && g.x1 != nullptr && g.nslices == 1 && (g.KS == 1024 || g.KS == 2048)) {
      g.nstages = stages_for(g.KS, MODE, true);
      return launch_pdl(nvfp4_gemv_kernel<MODE, true>, dim3(grid), dim3(32 * (2 * g.nstages + 1)),
                        gemv_smem(g.KS, MODE, true), s, g);
    }
  }
  g.nstages = stages_for(g.KS, MODE, false);
  return launch_pdl(nvfp4_gemv_kernel<MODE, false>, dim3(grid), dim3(32 * (2 * g.nstages + 1)),
                    gemv_smem(g.KS, MODE, false), s, g);
}

}  // namespace

// ---------------------------------------------------------------------------
// host side: the dense context
// ---------------------------------------------------------------------------
}  // namespace nvmoe

struct moe_dense {
  int kind = 0;              // 0 lm_head, 1 dense FFN
  int device = 0, sm_count = 0;
  int d = 0, rows = 0, f = 0, max_tokens = 0;
  int S = 1, KS = 0;         // K slices of the down projection
  uint8_t* arena = nullptr;
  uint8_t* codes = nullptr;  // head [R][d/2]; FFN gate/up tiles [2f][d/2]
  uint8_t* scales = nullptr;
  uint8_t* dn_codes = nullptr;   // FFN: [S][d][KS/2]
  uint8_t* dn_scales = nullptr;  // FFN: [S][d][KS/16]
  float ts[3] = {0.f, 0.f, 0.f};
  uint8_t* x16 = nullptr;    // [kTokPass][d] f16
  float* xun = nullptr;      // [kTokPass]
  float* h = nullptr;        // FFN: [kTokPass][f]
  uint8_t* h_hi = nullptr;   // FFN: [kTokPass][f] f16
  uint8_t* h_lo = nullptr;
  float* hun = nullptr;      // FFN: [kTokPass]
  uint32_t* hmax = nullptr;  // FFN: [kTokPass] max |h| of each token (fp32 bits)
  float* part = nullptr;     // FFN: [S][kTokPass][d]
  int* status = nullptr;
};

namespace nvmoe {

namespace {

size_t carve_dense(moe_dense* x, uint8_t* base) {
  size_t off = 0;
  auto take = [&](size_t bytes) {
    off = (off + 255) & ~size_t(255);
    uint8_t* p = base ? base + off : nullptr;
    off += bytes;
    return p;
  };
  const size_t d = x->d;
  const size_t R = x->kind == 0 ? (size_t)x->rows : 2 * (size_t)x->f;
  x->codes = take(R * d / 2);
  x->scales = take(R * d / 16);
  x->x16 = take((size_t)kTokPass * d * 2);
  x->xun = reinterpret_cast<float*>(take(kTokPass * sizeof(float)));
  x->status = reinterpret_cast<int*>(take(sizeof(int)));
  if (x->kind == 1) {
    const size_t f = x->f;
    x->dn_codes = take(d * f / 2);
    x->dn_scales = take(d * f / 16);
    x->h = reinterpret_cast<float*>(take((size_t)kTokPass * f * sizeof(float)));
    x->h_hi = take((size_t)kTokPass * f * 2);
    x->h_lo = take((size_t)kTokPass * f * 2);
    x->hun = reinterpret_cast<float*>(take(kTokPass * sizeof(float)));
    x->hmax = reinterpret_cast<uint32_t*>(take(kTokPass * sizeof(uint32_t)));
    x->part = reinterpret_cast<float*>(take((size_t)x->S * kTokPass * d * sizeof(float)));
  }
  return off;
}

bool matrix_ok(const moe_matrix* m) { return m && m->codes && m->scales && m->tensor_scale; }

// K slices of the dense down projection: the largest K slice <= 2304 that is a
// multiple of 256 (a code row of the slice is whole 128-byte swizzle segments)
// and divides f (so a stage of 16 rows x K slice stays ~20 KB).
// K slices of the dense down projection: 2048 wide when they divide d_ff
// (the width the one-token FMA consumer takes), else the widest multiple of
// 256 up to 2304 that does.
int down_slices(int f) {
  if (f % 2048 == 0) return f / 2048;
  for (int ks = 2304; ks >= 256; ks -= 256)
    if (f % ks == 0) return f / ks;
  return -1;
}

moe_status alloc_dense(moe_dense* x) {
  x->arena = nullptr;
  const size_t bytes = carve_dense(x, nullptr);
  if (device_alloc(reinterpret_cast<void**>(&x->arena), bytes) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_OOM;
  }
  carve_dense(x, x->arena);
  return MOE_OK;
}

cudaError_t set_gemv_smem() {
  cudaError_t e = cudaSuccess;
  const int lim = kStageBudget;   // every ring fits: stages_for() fills at most this many bytes
  const cudaFuncAttribute a = cudaFuncAttributeMaxDynamicSharedMemorySize;
  if (e == cudaSuccess) e = cudaFuncSetAttribute(nvfp4_gemv_kernel<kModeHead, false>, a, lim);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(nvfp4_gemv_kernel<kModeGateUp, false>, a, lim);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(nvfp4_gemv_kernel<kModeGateUp, true>, a, lim);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(nvfp4_gemv_kernel<kModeDown, false>, a, lim);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(nvfp4_gemv_kernel<kModeDown, true>, a, lim);
  return e;
}

moe_status finish_init(moe_dense* x, cudaError_t e, moe_dense** out) {
  if (e == cudaSuccess) e = cudaMemset(x->status, 0, sizeof(int));
  if (e == cudaSuccess) e = set_gemv_smem();
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    cudaFree(x->arena);
    delete x;
    return e == cudaErrorMemoryAllocation ? MOE_ERR_OOM : MOE_ERR_CUDA;
  }
  *out = x;
  return MOE_OK;
}

bool is_pow2_between(int v, int lo, int hi) { return v >= lo && v <= hi && (v & (v - 1)) == 0; }

moe_status check_dense_call(moe_dense* x, const void* in, int T, const void* out) {
  if (!x || T < 0 || T > x->max_tokens) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!in || !out || (reinterpret_cast<uintptr_t>(in) & 15) || (reinterpret_cast<uintptr_t>(out) & 15)))
    return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

GemvArgs base_args(const moe_dense* x, int T) {
  GemvArgs g{};
  g.nslices = 1;
  g.T = T;
  g.status = x->status;
  g.dbg = 0;
  return g;
}

}  // namespace

}  // namespace nvmoe

using namespace nvmoe;

extern "C" {

moe_status moe_head_init(int vocab, int d_model, const moe_matrix* w, int max_tokens, int device, moe_dense** out) {
  if (!out) return MOE_ERR_INVALID_ARG;
  *out = nullptr;
  if (vocab <= 0 || d_model <= 0 || max_tokens <= 0 || !matrix_ok(w)) return MOE_ERR_INVALID_ARG;
  if (vocab % 16 != 0 || !is_pow2_between(d_model, 256, 4096) || max_tokens > 4096) return MOE_ERR_UNSUPPORTED;
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || device < 0 || device >= ndev) return MOE_ERR_INVALID_ARG;
  if (cudaSetDevice(device) != cudaSuccess) return MOE_ERR_CUDA;
  moe_dense* x = new moe_dense();
  x->kind = 0;
  x->device = device;
  x->d = d_model;
  x->rows = vocab;
  x->max_tokens = max_tokens;
  cudaDeviceGetAttribute(&x->sm_count, cudaDevAttrMultiProcessorCount, device);
  moe_status st = alloc_dense(x);
  if (st != MOE_OK) {
    delete x;
    return st;
  }
  const size_t R = vocab, d = d_model;
  cudaError_t e = cudaMemcpy(x->codes, w->codes, R * d / 2, cudaMemcpyDefault);
  if (e == cudaSuccess) e = cudaMemcpy(x->scales, w->scales, R * d / 16, cudaMemcpyDefault);
  if (e == cudaSuccess) e = cudaMemcpy(&x->ts[0], w->tensor_scale, sizeof(float), cudaMemcpyDefault);
  if (e == cudaSuccess) e = swizzle_rows(x->codes, R, d / 2);
  if (e == cudaSuccess) e = swizzle_rows(x->scales, R, d / 16);
  return finish_init(x, e, out);
}

moe_status moe_head_forward(moe_dense* x, const void* x_bf16, int T, float* logits, cudaStream_t s) {
  moe_status st = check_dense_call(x, x_bf16, T, logits);
  if (st != MOE_OK) return st;
  if (x->kind != 0) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  cudaSetDevice(x->device);
  const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x_bf16);
  for (int t0 = 0; t0 < T; t0 += kTokPass) {
    const int n = T - t0 < kTokPass ? T - t0 : kTokPass;
    if (launch_pdl(prep_x_kernel, dim3(rows_read(n)), dim3(256), 0, s, xb + (size_t)t0 * x->d, n, x->d, x->x16,
                   x->xun, (uint32_t*)nullptr) != cudaSuccess)
      return MOE_ERR_CUDA;
    GemvArgs g = base_args(x, n);
    g.codes = x->codes;
    g.scales = x->scales;
    g.ntiles = x->rows / 16;
    g.KS = x->d;
    g.K = x->d;
    g.b_hi = x->x16;
    g.unshift = x->xun;
    g.ts0 = x->ts[0];
    g.out = logits + (size_t)t0 * x->rows;
    g.out_ld = x->rows;
    g.x1 = n == 1 ? xb + (size_t)t0 * x->d : nullptr;
    if (launch_gemv<kModeHead>(g, x->sm_count, s) != cudaSuccess) return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

moe_status moe_ffn_init(int d_model, int d_ff, const moe_matrix* gate, const moe_matrix* up, const moe_matrix* down,
                        int max_tokens, int device, moe_dense** out) {
  if (!out) return MOE_ERR_INVALID_ARG;
  *out = nullptr;
  if (d_model <= 0 || d_ff <= 0 || max_tokens <= 0 || !matrix_ok(gate) || !matrix_ok(up) || !matrix_ok(down))
    return MOE_ERR_INVALID_ARG;
  if (!is_pow2_between(d_model, 256, 4096) || d_ff % 256 != 0 || d_ff > 65536 || max_tokens > 4096 ||
      down_slices(d_ff) < 1)
    return MOE_ERR_UNSUPPORTED;
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || device < 0 || device >= ndev) return MOE_ERR_INVALID_ARG;
  if (cudaSetDevice(device) != cudaSuccess) return MOE_ERR_CUDA;
  moe_dense* x = new moe_dense();
  x->kind = 1;
  x->device = device;
  x->d = d_model;
  x->f = d_ff;
  x->max_tokens = max_tokens;
  x->S = down_slices(d_ff);
  x->KS = d_ff / x->S;
  cudaDeviceGetAttribute(&x->sm_count, cudaDevAttrMultiProcessorCount, device);
  moe_status st = alloc_dense(x);
  if (st != MOE_OK) {
    delete x;
    return st;
  }
  const size_t d = d_model, f = d_ff;
  // canonical copies go through temporaries in the caller-independent part of the arena: the
  // B-operand buffers are large enough only for small layers, so use one device temporary
  uint8_t* tmp = nullptr;
  const size_t tmp_bytes = 2 * f * d / 2;
  cudaError_t e = device_alloc(reinterpret_cast<void**>(&tmp), tmp_bytes);
  if (e != cudaSuccess) {
    cudaGetLastError();
    cudaFree(x->arena);
    delete x;
    return MOE_ERR_OOM;
  }
  // gate / up codes, then scales, into 8 + 8 row tiles
  e = cudaMemcpy(tmp, gate->codes, f * d / 2, cudaMemcpyDefault);
  if (e == cudaSuccess) e = cudaMemcpy(tmp + f * d / 2, up->codes, f * d / 2, cudaMemcpyDefault);
  if (e == cudaSuccess) {
    interleave_gu_kernel<<<(unsigned)(2 * f), 128>>>(tmp, tmp + f * d / 2, d / 2, (int)f, x->codes);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpy(tmp, gate->scales, f * d / 16, cudaMemcpyDefault);
  if (e == cudaSuccess) e = cudaMemcpy(tmp + f * d / 16, up->scales, f * d / 16, cudaMemcpyDefault);
  if (e == cudaSuccess) {
    interleave_gu_kernel<<<(unsigned)(2 * f), 128>>>(tmp, tmp + f * d / 16, d / 16, (int)f, x->scales);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  // W_down into K slices
  if (e == cudaSuccess) e = cudaMemcpy(tmp, down->codes, d * f / 2, cudaMemcpyDefault);
  if (e == cudaSuccess) {
    slice_rows_kernel<<<dim3((unsigned)d, (unsigned)x->S), 128>>>(tmp, (int)d, f / 2, x->S, x->dn_codes);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpy(tmp, down->scales, d * f / 16, cudaMemcpyDefault);
  if (e == cudaSuccess) {
    slice_rows_kernel<<<dim3((unsigned)d, (unsigned)x->S), 128>>>(tmp, (int)d, f / 16, x->S, x->dn_scales);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  cudaFree(tmp);
  if (e == cudaSuccess) e = swizzle_rows(x->codes, 2 * f, d / 2);
  if (e == cudaSuccess) e = swizzle_rows(x->scales, 2 * f, d / 16);
  if (e == cudaSuccess) e = swizzle_rows(x->dn_codes, (size_t)x->S * d, x->KS / 2);
  if (e == cudaSuccess) e = swizzle_rows(x->dn_scales, (size_t)x->S * d, x->KS / 16);
  if (e == cudaSuccess) e = cudaMemcpy(&x->ts[0], gate->tensor_scale, sizeof(float), cudaMemcpyDefault);
  if (e == cudaSuccess) e = cudaMemcpy(&x->ts[1], up->tensor_scale, sizeof(float), cudaMemcpyDefault);
  if (e == cudaSuccess) e = cudaMemcpy(&x->ts[2], down->tensor_scale, sizeof(float), cudaMemcpyDefault);
  return finish_init(x, e, out);
}

moe_status moe_ffn_forward(moe_dense* x, const void* x_bf16, int T, void* y_bf16, int residual, cudaStream_t s) {
  moe_status st = check_dense_call(x, x_bf16, T, y_bf16);
  if (st != MOE_OK) return st;
  if (x->kind != 1 || (T > 0 && x_bf16 == y_bf16)) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  cudaSetDevice(x->device);
  const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x_bf16);
  __nv_bfloat16* yb = static_cast<__nv_bfloat16*>(y_bf16);
  const int d = x->d, f = x->f;
  for (int t0 = 0; t0 < T; t0 += kTokPass) {
    const int n = T - t0 < kTokPass ? T - t0 : kTokPass;
    if (launch_pdl(prep_x_kernel, dim3(rows_read(n)), dim3(256), 0, s, xb + (size_t)t0 * d, n, d, x->x16, x->xun,
                   x->hmax) != cudaSuccess)
      return MOE_ERR_CUDA;
    GemvArgs g = base_args(x, n);
    g.codes = x->codes;
    g.scales = x->scales;
    g.ntiles = 2 * f / 16;
    g.KS = d;
    g.K = d;
    g.b_hi = x->x16;
    g.unshift = x->xun;
    g.ts0 = x->ts[0];
    g.ts1 = x->ts[1];
    g.out = x->h;
    g.out_ld = f;
    g.hmax = x->hmax;
    g.x1 = n == 1 ? xb + (size_t)t0 * d : nullptr;
    if (launch_gemv<kModeGateUp>(g, x->sm_count, s) != cudaSuccess) return MOE_ERR_CUDA;
    // one token with 2048-wide K slices: the down pass reads h (fp32) itself, no hi / lo split
    const bool h_direct = n == 1 && x->KS == 2048;
    if (!h_direct &&
        launch_pdl(prep_h_kernel, dim3((unsigned)((f + kPrepHChunk - 1) / kPrepHChunk), (unsigned)rows_read(n)),
                   dim3(256), 0, s, (const float*)x->h, n, f, (const uint32_t*)x->hmax, x->h_hi, x->h_lo,
                   x->hun) != cudaSuccess)
      return MOE_ERR_CUDA;
    GemvArgs dn = base_args(x, n);
    dn.h1 = h_direct ? x->h : nullptr;
    dn.codes = x->dn_codes;
    dn.scales = x->dn_scales;
    dn.slice_codes = (size_t)d * x->KS / 2;
    dn.slice_scales = (size_t)d * x->KS / 16;
    dn.ntiles = d / 16;
    dn.nslices = x->S;
    dn.KS = x->KS;
    dn.K = f;
    dn.b_hi = x->h_hi;
    dn.b_lo = x->h_lo;
    dn.unshift = x->hun;
    dn.ts0 = x->ts[2];
    dn.out = x->part;
    dn.out_ld = d;
    if (launch_gemv<kModeDown>(dn, x->sm_count, s) != cudaSuccess) return MOE_ERR_CUDA;
    if (launch_pdl(reduce_down_kernel, dim3((n * d + 255) / 256), dim3(256), 0, s, (const float*)x->part, x->S, n,
                   d, xb + (size_t)t0 * d, residual, yb + (size_t)t0 * d) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

moe_status moe_dense_get_device_status(moe_dense* x) {
  if (!x) return MOE_ERR_INVALID_ARG;
  cudaSetDevice(x->device);
  if (cudaDeviceSynchronize() != cudaSuccess) return MOE_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, x->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemset(x->status, 0, sizeof(int)) != cudaSuccess) return MOE_ERR_CUDA;
  return static_cast<moe_status>(v);
}

int moe_dense_kernels_per_forward(moe_dense* x, int T) {
  if (!x || T <= 0) return 0;
  int n = 0;
  for (int t0 = 0; t0 < T; t0 += kTokPass) {
    const int m = T - t0 < kTokPass ? T - t0 : kTokPass;
    n += x->kind == 0 ? 2 : (m == 1 && x->KS == 2048 ? 4 : 5);
  }
  return n;
}

moe_status moe_dense_destroy(moe_dense* x) {
  if (!x) return MOE_OK;
  cudaSetDevice(x->device);
  cudaError_t e = cudaFree(x->arena);
  delete x;
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // extern "C"
