// Prefill: block-scaled FP4 x FP4 grouped GEMMs on the 5th-generation tensor
// cores (tcgen05.mma kind::mxf4nvf4, scales in tensor memory).
//
// The pages list prompt-processing kernels among the vendor's custom kernels
// ("Recursive Flint 40B-A2.5B：まず速さを第一に考えて作られたコーディングモデル",
// section "量子化のレシピは最も転用しやすい部分です") without describing them.
// Here prefill is the one place where the MoE layer is a dense contraction
// (~96 tokens per routed expert at 4096 tokens, all tokens for the shared
// expert), so it runs on the tensor cores with both operands in NVFP4:
//
//   1. plan:   padded position blocks per active expert (multiples of 128
//              tokens, so every 128-row block belongs to one expert), made by
//              the bucketing kernel;
//   2. x -> NVFP4 (16-element E4M3 block scales, tensor scale 1) gathered into
//              the padded blocks, scales written straight into the
//              scale-factor atoms the MMA reads;
//   3. GEMM gate/up: D[128 tokens, 256 weight rows] per (token block, 256-row
//              tile of the gate/up layout).  Such a tile holds two groups of
//              64 gate rows and the matching 64 up rows, so each epilogue
//              thread (one token, one TMEM lane) forms h = silu(g) * u for its
//              32 hidden units in registers and quantises it to NVFP4 (block
//              16, scale 1): 16 contiguous code bytes and 2 adjacent scale
//              bytes per token;
//   4. GEMM down: D[128 tokens, 128 output dims] * ts_down * w is added with
//              vector reductions into the token's row of an fp32 accumulator
//              that stays in L2 (the weighted scatter-combine; the order of a
//              token's seven contributions is not fixed), then one pass writes
//              bf16 y (+ the residual).  Batches whose accumulator would not
//              fit well inside L2 store per-position outputs instead and add
//              them in a fixed order afterwards.
//
// GEMM kernel: persistent, one CTA per SM, 512 TMEM columns.
//   gate/up: 128 x 256 tiles (an N = 256 MMA costs 40% more than an N = 128
//            one for twice the work, and its 12 scale copies per stage are 6
//            per 128 columns instead of 8), one 256-column accumulator, 576
//            threads; the epilogue warps free it as soon as their columns are
//            in registers, so the next tile's MMAs wait only for those loads;
//   down:    128 x 128 tiles, two 128-column accumulators (the epilogue of one
//            tile overlaps the MMAs of the next), 16 epilogue warps of 32
//            columns each (the vector reductions are its bound), 576 threads.
//   warp 0  TMA producer: 4-stage ring of {A 128x256 fp4 tokens (SW128),
//           B 128 or 256 x 256 fp4 weights (SW128), SFA 4 atoms, SFB 4 atoms
//           per 128 rows}
//   warp 1  TMEM owner + single-thread MMA issuer: per stage, scale atoms ->
//           TMEM (tcgen05.cp 32x128b.warpx4), 4 MMAs of K = 64
//   warps 2.. epilogue: 4 warps per TMEM lane quarter (lanes 32*(warp%4) ..),
//           tcgen05.ld 32 columns at a time.  The down GEMM's rows go through a
//           per-warp shared-memory tile so that each vector reduction covers
//           4 rows x 128 contiguous bytes instead of 32 scattered rows (2x the
//           reduction rate into L2).
// All waits are bounded; the first one that gives up latches MOE_ERR_TIMEOUT
// and sets a CTA-wide abort flag so that no other role waits afterwards.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "internal.h"
#include "sm100.cuh"

namespace nvmoe {

namespace {

using namespace sm100;

constexpr int kBM = 128;        // tokens per tile (MMA M, TMEM lanes)
constexpr int kStageK = 256;    // fp4 elements of K per stage (128 bytes per row)
constexpr int kBNGateUp = 256;  // gate/up: 128 tokens x 256 weight rows per tile
constexpr int kBNDown = 128;    // down: 128 tokens x 128 output dims per tile
constexpr int kStagesGateUp = 4;   // gate/up: 4 x 54 KB in flight
constexpr int kStagesDown = 4;     // down: 4 x 36 KB + the epilogue's row staging
constexpr uint32_t kTmemCols = 512;
constexpr int kSfColsPerStage = 16;           // 4 k-steps x 4 columns of scales per 128 rows

// shared-memory plan of the GEMM kernel (offsets from a 1024-aligned base)
constexpr int kA = kBM * 128;                 // 16 KB per stage
constexpr int kSF = 4 * 512;                  // 2 KB of scales per 128 rows per stage
constexpr int kEpiStride = 144;             // staged row: 32 fp32 + 16 bytes of padding (no bank conflicts)
// Tile of BN weight rows: epilogue warps (two per 64 columns, 32 columns
// each: BN / 16 warps), threads, the ring of NST stages {A, B, SFA, SFB}
// from a 1024-aligned base and (down GEMM only) the epilogue's staging rows.
// TMEM: the accumulator(s) (two of 128 columns for BN = 128 so that a tile's
// epilogue overlaps the next tile's MMAs; one of 256 for BN = 256), then a
// ring of token-side scales (16 columns per stage) and one of weight-side
// scales (16 columns per 128 rows per stage: a k-step takes 4 columns per
// 128 rows, rows 128..255 of a 256-row tile in the 4 columns after rows
// 0..127).
template <int NST, int BN, int EW>
struct Plan {
  static constexpr int epi_warps = EW;
  static constexpr int threads = 64 + 32 * epi_warps;
  static constexpr int kB = BN * 128;
  static constexpr int kSFB = (BN / 128) * kSF;
  static constexpr int stage_bytes = kA + kB + kSF + kSFB;
  static constexpr int offA = 0;
  static constexpr int offB = offA + NST * kA;
  static constexpr int offSFA = offB + NST * kB;
  static constexpr int offSFB = offSFA + NST * kSF;
  static constexpr int offEpi = offSFB + NST * kSFB;
  static constexpr int nacc = BN == 256 ? 1 : 2;
  static constexpr int sfaCol0 = nacc * BN;
  static constexpr int sfbCol0 = sfaCol0 + NST * kSfColsPerStage;
  static constexpr int sfbColsPerStage = (BN / 128) * kSfColsPerStage;
  static_assert(sfbCol0 + NST * sfbColsPerStage <= (int)kTmemCols, "scale-factor columns exceed TMEM");
};
constexpr int kEpiGateUp = kBNGateUp / 16;   // 32 hidden units (64 columns) per warp
constexpr int kEpiDown = 16;                  // 32 output columns per warp
using PlanGateUp = Plan<kStagesGateUp, kBNGateUp, kEpiGateUp>;
using PlanDown = Plan<kStagesDown, kBNDown, kEpiDown>;
constexpr int kSmemGateUp = PlanGateUp::offEpi + 1024;               // + alignment slack
constexpr int kSmemDown = PlanDown::offEpi + PlanDown::epi_warps * 32 * kEpiStride + 1024;

// largest a < na with tab[a] <= v (tab non-decreasing, tab[0] = 0)
__device__ __forceinline__ int find_seg(const int32_t* tab, int na, int v) {
  int lo = 0, hi = na - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(tab + mid) <= v) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// ---------------------------------------------------------------------------
// NVFP4 block quantisation with tensor scale 1 (same rules as the weights)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t q_e4m3(float v) {
  uint16_t out;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(out) : "f"(0.0f), "f"(v));
  return out & 0xFF;
}
// E2M1 code of v / dq, rounded to nearest with ties to the even code, decided
// without dividing: |v| is compared with each rounding midpoint times dq.
// Midpoints have at most 3 significant bits and dq (an E4M3 value) at most 4,
// so every product is exact and the comparison is that of the exact quotient.
__device__ __forceinline__ uint32_t e2m1_by_compare(float v, float dq) {
  const float a = fabsf(v);
  const uint32_t c = (a > 0.25f * dq) + (a >= 0.75f * dq) + (a > 1.25f * dq) + (a >= 1.75f * dq) +
                     (a > 2.5f * dq) + (a >= 3.5f * dq) + (a > 5.0f * dq);
  return (v < 0.f && c != 0u) ? (c | 8u) : c;
}

// byte offset of the scale of (row p, 16-block b) in a [rows/128][ksteps][512] atom array
__device__ __forceinline__ size_t sf_atom_offset(int p, int b, int ksteps) {
  return ((size_t)(p >> 7) * ksteps + (b >> 2)) * 512 + (p & 31) * 16 + ((p >> 5) & 3) * 4 + (b & 3);
}

// Active-expert tables copied to shared memory once per CTA, so that mapping a
// tile index to its expert costs shared-memory reads only (a binary search
// over global memory would put several dependent L2 round trips in front of
// every TMA issue).
constexpr int kMaxActive = 256 + 2 + 1;
struct ActTables {
  int ppos[kMaxActive];   // padded first row, total last
  int e[kMaxActive];
  int n[kMaxActive];
  int pos[kMaxActive];
};

// x -> NVFP4 (tensor scale 1), once per token, written straight into the
// token's k + S padded rows of the grouped-GEMM operand: the codes, and the
// block scales row-major (one byte per 16-element block; x_sf_atoms_kernel
// then builds the MMA's scale-factor atoms from them).  One warp per token;
// each lane quantises four consecutive 16-element blocks (one k-step) at a
// time, so a warp writes a row's scales as 128 contiguous bytes (written
// straight into the atoms, they were 32 scattered 4-byte stores per row, most
// of this kernel's store traffic).  The token's row of the fp32 output
// accumulator is cleared on the way.  Padding rows of the position blocks are
// not written: the GEMM rows are independent and the outputs of padding rows
// are never read.
constexpr int kMaxPerTok = 10;   // top_k (<= 8) + n_shared (<= 2)
__global__ void __launch_bounds__(256, 4) quant_scatter_x_kernel(Routing r, const __nv_bfloat16* __restrict__ x, int T,
                                                              int d, int k, int S, uint8_t* __restrict__ codes,
                                                              uint8_t* __restrict__ sf_rows, float* __restrict__ yacc) {
  __shared__ int s_pos[kMaxActive], s_ppos[kMaxActive], s_prow[8][kMaxPerTok];
  const int na = *r.n_active;
  for (int i = threadIdx.x; i <= na; i += blockDim.x) {
    s_pos[i] = i < na ? r.act_pos[i] : 0;
    s_ppos[i] = r.act_ppos[i];
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  if (t >= T) return;
  // lane j < k + S finds the padded row of the token's j-th position
  if (lane < k + S) {
    const int pos = lane < k ? __ldg(r.slot_pos + (size_t)t * k + lane) : T * k + (lane - k) * T + t;
    int lo = 0, hi = na - 1;               // last active expert whose first position is <= pos
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_pos[mid] <= pos) lo = mid; else hi = mid - 1;
    }
    s_prow[warp][lane] = s_ppos[lo] + (pos - s_pos[lo]);
  }
  __syncwarp();
  const int* pr = s_prow[warp];
  if (yacc)
    for (int i = lane; i < d / 4; i += 32)
      reinterpret_cast<float4*>(yacc + (size_t)t * d)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  const int nblk = d / 16;
  for (int b0 = 4 * lane; b0 < nblk; b0 += 128) {
    const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * d + b0 * 16);
    uint4 u[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) u[q] = __ldg(src + q);
    uint32_t cw[8], sc = 0;
#pragma unroll
    for (int blk = 0; blk < 4; ++blk) {
      const uint32_t w[8] = {u[2 * blk].x, u[2 * blk].y, u[2 * blk].z, u[2 * blk].w,
                             u[2 * blk + 1].x, u[2 * blk + 1].y, u[2 * blk + 1].z, u[2 * blk + 1].w};
      float v[16];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        v[2 * q] = __uint_as_float(w[q] << 16);
        v[2 * q + 1] = __uint_as_float(w[q] & 0xFFFF0000u);
      }
      float amax = 0.f;
#pragma unroll
      for (int q = 0; q < 16; ++q) amax = fmaxf(amax, fabsf(v[q]));
      const uint32_t s8 = q_e4m3(__fdiv_rn(amax, 6.0f));
      const float dq = e4m3_to_f32(s8);
      uint32_t lo = 0, hi = 0;
      // codes by comparison with midpoint x dq (exact products).  For a bf16
      // value this equals rounding the fp32 quotient v / dq: the exact quotient
      // is a midpoint itself or at least ~2^-8 (relative) away from every midpoint.
      if (dq > 0.f) {
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          lo |= e2m1_by_compare(v[q], dq) << (4 * q);
          hi |= e2m1_by_compare(v[8 + q], dq) << (4 * q);
        }
      }
      cw[2 * blk] = lo;
      cw[2 * blk + 1] = hi;
      sc |= s8 << (8 * blk);
    }
    for (int j = 0; j < k + S; ++j) {
      const int p = pr[j];
      uint4* dst = reinterpret_cast<uint4*>(codes + (size_t)p * (d / 2) + b0 * 8);
      dst[0] = make_uint4(cw[0], cw[1], cw[2], cw[3]);
      dst[1] = make_uint4(cw[4], cw[5], cw[6], cw[7]);
      *reinterpret_cast<uint32_t*>(sf_rows + (size_t)p * nblk + b0) = sc;   // blocks b0..b0+3: one k-step
    }
  }
}

// Row-major block scales [rows][d/16] -> the MMA's scale-factor atoms
// [rows/128][d/64][512] (row r, block 4 kk + j: byte (r % 32) * 16 + (r / 32) * 4
// + j of atom kk of r's 128-row block).  One CTA per 128-row block, through
// shared memory; a row's words sit (d/64 + 1) words apart, an odd stride, so
// the 32 lanes that gather the rows c, c + 32, c + 64, c + 96 of one 16-byte
// atom chunk read 32 different banks.  CTAs past the padded row count exit.
__global__ void __launch_bounds__(256) x_sf_atoms_kernel(Routing r, const uint8_t* __restrict__ rows_sf, int d,
                                                         uint8_t* __restrict__ atoms) {
  extern __shared__ uint32_t w[];
  const int b = blockIdx.x;
  if (b >= (r.act_ppos[*r.n_active] >> 7)) return;
  const int ks = d / 64, ws = ks + 1;
  // the block's 128 rows are contiguous: 32 * ks 16-byte loads, all of a
  // thread's issued before any is stored (one memory round trip, not one per load)
  const uint4* src = reinterpret_cast<const uint4*>(rows_sf + (size_t)b * 128 * (d / 16));
  constexpr int kPer = 8;
  const int n4 = 32 * ks;
  for (int i0 = 0; i0 < n4; i0 += kPer * 256) {
    uint4 v[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int i = i0 + u * 256 + (int)threadIdx.x;
      v[u] = i < n4 ? src[i] : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int i = i0 + u * 256 + (int)threadIdx.x;
      if (i < n4) {
        uint32_t* row = w + ((4 * i) / ks) * ws + (4 * i) % ks;   // 4 words of one row (ks is a multiple of 4)
        row[0] = v[u].x;
        row[1] = v[u].y;
        row[2] = v[u].z;
        row[3] = v[u].w;
      }
    }
  }
  __syncthreads();
  uint4* dst = reinterpret_cast<uint4*>(atoms + (size_t)b * ks * 512);
  for (int i = threadIdx.x; i < 32 * ks; i += blockDim.x) {
    const int kk = i >> 5, c = i & 31;
    dst[i] = make_uint4(w[c * ws + kk], w[(c + 32) * ws + kk], w[(c + 64) * ws + kk], w[(c + 96) * ws + kk]);
  }
}

// ---------------------------------------------------------------------------
// the grouped GEMM
// ---------------------------------------------------------------------------
struct GemmArgs {
  Routing r;
  const uint8_t* sfa;     // activation scale atoms [rows/128][K/64][512]
  const uint8_t* sfb;     // weight scale atoms [n_all][M/128][K/64][512]
  const float* tsc;       // [n_all][3]
  int M;                  // weight rows per expert (2f or d)
  int K;                  // contraction length
  // mode 0 outputs
  uint8_t* hq_codes;      // [rows][f/2]
  uint8_t* hq_sf;         // [rows/128][f/64][512]
  int f;
  // mode 1 output: with yacc, every position adds w * ts_down * D into its token's
  // row of yacc (fp32 [T][d]); without, it stores ts_down * D into its own row of
  // yexp (fp32 [positions][d]) for the fixed-order combine
  float* yacc;
  float* yexp;
  int d;
  int* status;
  int dbg;                // debug flags (MOE_DEBUG_FORCE_TIMEOUT)
};

// unit u -> (128-token block, 128-row weight tile)
struct UnitInfo {
  int a, e, p0, nt, ntile;
};

__device__ __forceinline__ UnitInfo decode_unit(const ActTables& t, int u, int ntiles, int na) {
  UnitInfo ui;
  const int tb = u / ntiles;
  ui.ntile = u % ntiles;
  ui.p0 = tb * kBM;
  int lo = 0, hi = na - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (t.ppos[mid] <= ui.p0) lo = mid; else hi = mid - 1;
  }
  ui.a = lo;
  ui.e = t.e[lo];
  ui.nt = min(kBM, t.n[lo] - (ui.p0 - t.ppos[lo]));   // real tokens in the block
  return ui;
}

__device__ __forceinline__ float silu_fast(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

// NVFP4 (scale 1) of 16 consecutive fp32 values held by one thread -> 8 code bytes, one scale byte
__device__ __forceinline__ uint32_t quant16(const float* v, uint2& codes) {
  float amax = 0.f;
#pragma unroll
  for (int q = 0; q < 16; ++q) amax = fmaxf(amax, fabsf(v[q]));
  const uint32_t s = q_e4m3(__fdiv_rn(amax, 6.0f));
  const float dq = e4m3_to_f32(s);
  uint32_t lo = 0, hi = 0;
  if (dq > 0.f) {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      lo |= e2m1_by_compare(v[q], dq) << (4 * q);
      hi |= e2m1_by_compare(v[8 + q], dq) << (4 * q);
    }
  }
  codes = make_uint2(lo, hi);
  return s;
}

template <int NST, int MODE, int BN, int EW>
__global__ void __launch_bounds__(Plan<NST, BN, EW>::threads, 1)
    moe_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, GemmArgs g) {
  extern __shared__ uint8_t smem_raw[];
  using P = Plan<NST, BN, EW>;
  constexpr int kEpi = P::epi_warps;
  static_assert(MODE == 1 || EW == BN / 16, "gate/up: one warp per 32 hidden units of a lane quarter");
  constexpr int kColsPerWarp = BN * 4 / EW;   // down: output columns of one epilogue warp
  static_assert(MODE == 0 || kColsPerWarp % 32 == 0, "down: whole 32-column chunks per warp");
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t full_bar[NST], empty_bar[NST], dfull_bar[2], dempty_bar[2];
  __shared__ uint32_t tmem_base_s;
  __shared__ volatile int abort_flag;
  __shared__ ActTables tab;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int na = *g.r.n_active;
  for (int i = threadIdx.x; i <= na; i += blockDim.x) {
    tab.ppos[i] = g.r.act_ppos[i];
    if (i < na) {
      tab.e[i] = g.r.act_e[i];
      tab.n[i] = g.r.act_n[i];
      tab.pos[i] = g.r.act_pos[i];
    }
  }
  const int ntiles = g.M / BN, ksteps = g.K / 64, kstages = g.K / kStageK;
  const int mtiles = g.M / 128;   // 128-row tiles of scale atoms per expert

  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&dfull_bar[b], 1);
      mbar_init(&dempty_bar[b], kEpi);
    }
    abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  if (warp == 1) tmem_alloc(&tmem_base_s, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;
  const int U = (tab.ppos[na] / kBM) * ntiles;



  auto bounded_wait = [&](uint64_t* bar, uint32_t parity) -> bool {
    if (abort_flag) return false;
    if (wait_parity(bar, parity)) return true;
    abort_flag = 1;
    latch_status(g.status, MOE_ERR_TIMEOUT);
    return false;
  };

  if (warp == 0) {
    // ------------------------------ producer ------------------------------
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      for (int u = blockIdx.x; u < U && !abort_flag; u += gridDim.x) {
        const UnitInfo ui = decode_unit(tab, u, ntiles, na);
        const int brow = ui.e * g.M + ui.ntile * BN;
        const uint8_t* sfa = g.sfa + (size_t)(ui.p0 / kBM) * ksteps * 512;
        const uint8_t* sfb = g.sfb + ((size_t)ui.e * mtiles + ui.ntile * (BN / 128)) * ksteps * 512;
        for (int ks = 0; ks < kstages; ++ks) {
          if (!bounded_wait(&empty_bar[stage], phase ^ 1)) break;
          mbar_arrive_expect_tx(&full_bar[stage], P::stage_bytes);
          tma_load_2d(smem + P::offA + stage * kA, &tmA, ks * 128, ui.p0, &full_bar[stage]);
#pragma unroll
          for (int h = 0; h < BN / 128; ++h)
            tma_load_2d(smem + P::offB + stage * P::kB + h * 128 * 128, &tmB, ks * 128, brow + h * 128,
                        &full_bar[stage]);
          bulk_load(smem + P::offSFA + stage * kSF, sfa + (size_t)ks * 4 * 512, kSF, &full_bar[stage]);
#pragma unroll
          for (int h = 0; h < BN / 128; ++h)
            bulk_load(smem + P::offSFB + stage * P::kSFB + h * kSF, sfb + ((size_t)h * ksteps + ks * 4) * 512, kSF,
                      &full_bar[stage]);
          if (++stage == NST) { stage = 0; phase ^= 1; }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------ MMA issuer ----------------------------
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      const uint32_t idesc = idesc_mxf4nvf4(kBM, BN);
      int i = 0;
      for (int u = blockIdx.x; u < U && !abort_flag; u += gridDim.x, ++i) {
        const int buf = i % P::nacc, use = i / P::nacc;
        if (!bounded_wait(&dempty_bar[buf], (use & 1) ^ 1)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + buf * BN;
        for (int ks = 0; ks < kstages; ++ks) {
          if (!bounded_wait(&full_bar[stage], phase)) break;
          tc_fence_after();
          const uint32_t sfa_t = tmem + P::sfaCol0 + stage * kSfColsPerStage;
          const uint32_t sfb_t = tmem + P::sfbCol0 + stage * P::sfbColsPerStage;
          const uint32_t sa = smem_u32(smem + P::offSFA + stage * kSF);
          const uint32_t sb = smem_u32(smem + P::offSFB + stage * P::kSFB);
          // k-step kk: SFA in 4 columns; SFB of rows 128h .. 128h+127 in the
          // 4 columns at kk * 4 * (BN / 128) + 4h
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            tmem_cp_sf_atom(sfa_t + kk * 4, desc_sf_atom(sa + kk * 512));
#pragma unroll
            for (int h = 0; h < BN / 128; ++h)
              tmem_cp_sf_atom(sfb_t + kk * 4 * (BN / 128) + h * 4, desc_sf_atom(sb + h * kSF + kk * 512));
          }
          const uint64_t adesc = desc_kmajor_sw128(smem_u32(smem + P::offA + stage * kA));
          const uint64_t bdesc = desc_kmajor_sw128(smem_u32(smem + P::offB + stage * P::kB));
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_mxf4nvf4(d_tmem, adesc + (uint64_t)(kk * 2), bdesc + (uint64_t)(kk * 2), idesc, sfa_t + kk * 4,
                         sfb_t + kk * 4 * (BN / 128), ks > 0 || kk > 0);
          tc_commit(&empty_bar[stage]);
          if (++stage == NST) { stage = 0; phase ^= 1; }
        }
        tc_commit(&dfull_bar[buf]);
      }
    }
  } else {
    // ------------------------------ epilogue ------------------------------
    // TMEM lane = token row of the block; this thread owns token row m and
    // slice `sub` of the tile (gate/up: 32 hidden units, i.e. 32 gate and 32
    // up columns; down: kColsPerWarp output columns).
    const int q = warp & 3, sub = (warp - 2) >> 2;
    const int m = q * 32 + lane;
    uint8_t* stage_rows = smem + P::offEpi + (warp - 2) * 32 * kEpiStride;
    int i = 0;
    // Every epilogue warp runs the same units and never leaves the loop early
    // (a failed wait only skips the work), so all of them always arrive.  A
    // warp frees the accumulator as soon as its columns are in registers, so
    // the next tile's MMAs overlap this tile's arithmetic and stores.
    auto release = [&](bool ok, int buf) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0 && ok) mbar_arrive(&dempty_bar[buf]);
    };
    for (int u = blockIdx.x; u < U; u += gridDim.x, ++i) {
      const UnitInfo ui = decode_unit(tab, u, ntiles, na);
      const int buf = i % P::nacc, use = i / P::nacc;
      const bool ok = __all_sync(0xffffffffu, bounded_wait(&dfull_bar[buf], use & 1));   // warp-uniform
      tc_fence_after();
      const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + buf * BN;
      const float* ts = g.tsc + ui.e * 3;
      const int p = ui.p0 + m;                    // padded row of this token
      if constexpr (MODE == 0) {
        // 128-column group grp holds 64 gate rows then the matching 64 up rows
        // of hidden units (BN / 2) * ntile + 64 * grp + 0..63; this warp forms
        // the 32 of them at 32 * h32
        const int grp = sub >> 1, h32 = sub & 1;
        const int hid0 = 64 * grp + 32 * h32;   // first hidden unit of the warp within the tile
        const float tg = ts[0], tu = ts[1];
        uint32_t gv[32], uv[32];
        if (ok) {
          tmem_ld32(taddr + 128 * grp + 32 * h32, gv);
          tmem_ld32(taddr + 128 * grp + 64 + 32 * h32, uv);
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) { gv[j] = 0u; uv[j] = 0u; }
        }
        release(ok, buf);
        float hv[32];
#pragma unroll
        for (int j = 0; j < 32; ++j)
          hv[j] = silu_fast(__uint_as_float(gv[j]) * tg) * (__uint_as_float(uv[j]) * tu);
        uint2 c0, c1;
        const uint32_t s0 = quant16(hv, c0), s1 = quant16(hv + 16, c1);
        if (ok) {
          const int hb = ui.ntile * (BN / 2) + hid0;   // first hidden unit
          *reinterpret_cast<uint4*>(g.hq_codes + (size_t)p * (g.f / 2) + hb / 2) = make_uint4(c0.x, c0.y, c1.x, c1.y);
          // its two 16-unit block scales: 2 adjacent bytes of one k-step atom of the down GEMM
          *reinterpret_cast<uint16_t*>(g.hq_sf + sf_atom_offset(p, hb / 16, g.f / 64)) =
              static_cast<uint16_t>(s0 | (s1 << 8));
        }
      } else {
        // weighted scatter-combine: w * ts_down * D is added into the token's
        // row of the fp32 accumulator (vector reductions in L2; the order in
        // which a token's top_k + shared contributions arrive is not fixed).
        // Without the accumulator, ts_down * D goes to the position's own row.
        const int i_tok = p - tab.ppos[ui.a];   // index among the expert's tokens
        const bool real = m < ui.nt;
        const int pos = tab.pos[ui.a] + i_tok;
        const bool acc = g.yacc != nullptr;
        const int row_out = !real ? 0 : acc ? __ldg(g.r.pos_tok + pos) : pos;
        const float wtd = (real && acc) ? __ldg(g.r.pos_w + pos) * ts[2] : ts[2];
        const unsigned real_mask = ok ? __ballot_sync(0xffffffffu, real) : 0u;
        float* base = (acc ? g.yacc : g.yexp) + ui.ntile * BN;
        constexpr int kChunks = kColsPerWarp / 32;
        uint32_t v[kChunks][32];
        if (ok) {
#pragma unroll
          for (int h = 0; h < kChunks; ++h) tmem_ld32(taddr + sub * kColsPerWarp + h * 32, v[h]);
        }
        release(ok, buf);
#pragma unroll
        for (int h = 0; h < kChunks && ok; ++h) {
          const int c0 = sub * kColsPerWarp + h * 32;
          __syncwarp();                         // the previous chunk's rows have been read
#pragma unroll
          for (int j = 0; j < 32; j += 4)
            *reinterpret_cast<float4*>(stage_rows + lane * kEpiStride + j * 4) =
                make_float4(__uint_as_float(v[h][j]) * wtd, __uint_as_float(v[h][j + 1]) * wtd,
                            __uint_as_float(v[h][j + 2]) * wtd, __uint_as_float(v[h][j + 3]) * wtd);
          __syncwarp();
          // 8 lanes per row: each instruction covers 4 rows x 128 contiguous bytes
#pragma unroll
          for (int rr = 0; rr < 32; rr += 4) {
            const int row = rr + (lane >> 3), qq = lane & 7;
            const int dst_row = __shfl_sync(0xffffffffu, row_out, row);
            if ((real_mask >> row) & 1u) {
              const float4 x = *reinterpret_cast<const float4*>(stage_rows + row * kEpiStride + qq * 16);
              float* dst = base + (size_t)dst_row * g.d + c0 + qq * 4;
              if (acc)
                asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};"
                             :: "l"(dst), "f"(x.x), "f"(x.y), "f"(x.z), "f"(x.w) : "memory");
              else
                *reinterpret_cast<float4*>(dst) = x;
            }
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  // every wait has completed or given up; the debug flag reports a timeout anyway
  if (threadIdx.x == 0 && (g.dbg & MOE_DEBUG_FORCE_TIMEOUT)) latch_status(g.status, MOE_ERR_TIMEOUT);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 2-D byte tensor [rows][row_bytes], boxes of box_rows x 128 bytes, 128-byte swizzle
bool make_tmap(CUtensorMap* m, const void* base, uint64_t rows, uint64_t row_bytes, uint32_t box_rows) {
  return make_tmap_u8(m, base, rows, row_bytes, 128, box_rows, true);
}

// weight scales [n][M][K/16] -> atoms [n][M/128][K/64][512]; one thread per output byte
__global__ void weight_sf_atoms_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst, size_t n, int M,
                                       int K) {
  const size_t total = n * (size_t)M * (K / 16);
  const size_t o = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (o >= total) return;
  const int ksteps = K / 64, mtiles = M / 128;
  const size_t atom = o / 512;
  const int w = (int)(o % 512);
  const int ks = (int)(atom % ksteps);
  const size_t rest = atom / ksteps;
  const int mt = (int)(rest % mtiles);
  const size_t e = rest / mtiles;
  const int lr = w / 16, col = (w % 16) / 4, kb = w % 4;
  const int row = mt * 128 + col * 32 + lr;
  dst[o] = src[(e * M + row) * (K / 16) + ks * 4 + kb];
}

}  // namespace

bool make_tmap_u8(CUtensorMap* m, const void* base, uint64_t rows, uint64_t row_bytes, uint32_t box_bytes,
                  uint32_t box_rows, bool swizzle128) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {row_bytes, rows};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_bytes, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The L2-resident accumulator pays while it stays well inside the 126 MB L2
// next to the streamed weights (48 MB: 6144 tokens at d_model 2048); larger
// batches store per-position outputs and combine them in a fixed order.
bool prefill_accumulates(const moe_config& c, int T) { return (size_t)T * c.d_model * sizeof(float) <= (48u << 20); }

bool prefill_supported(const moe_config& c) {
  return c.weight_format == MOE_W_NVFP4 && c.d_model % 256 == 0 && c.d_ff % 256 == 0 && c.d_model <= 8192;
}

size_t prefill_max_rows(const moe_config& c) {
  const size_t T = c.max_tokens, k = c.top_k, S = c.n_shared, E = c.n_experts;
  return (T * (k + S) + 128 * (E + S) + 127) / 128 * 128;
}

cudaError_t prefill_prepare(moe_ctx* c) {
  const int d = c->cfg.d_model, f = c->cfg.d_ff, n = c->n_all;
  const size_t t1 = (size_t)n * 2 * f * (d / 16), t2 = (size_t)n * d * (f / 16);
  weight_sf_atoms_kernel<<<(unsigned)((t1 + 255) / 256), 256>>>(c->gu_scales, c->pf_sfa_gu, n, 2 * f, d);
  weight_sf_atoms_kernel<<<(unsigned)((t2 + 255) / 256), 256>>>(c->dn_scales, c->pf_sfa_dn, n, d, f);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const size_t rows = prefill_max_rows(c->cfg);
  bool ok = make_tmap(&c->pf_tm[0], c->gu_codes, (uint64_t)n * 2 * f, d / 2, kBM) &&
            make_tmap(&c->pf_tm[1], c->dn_codes, (uint64_t)n * d, f / 2, kBM) &&
            make_tmap(&c->pf_tm[2], c->pf_xq, rows, d / 2, kBM) &&
            make_tmap(&c->pf_tm[3], c->pf_hq, rows, f / 2, kBM);
  if (!ok) return cudaErrorInvalidValue;
  e = cudaFuncSetAttribute(moe_gemm_kernel<kStagesGateUp, 0, kBNGateUp, kEpiGateUp>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemGateUp);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(moe_gemm_kernel<kStagesDown, 1, kBNDown, kEpiDown>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kSmemDown);
}

cudaError_t launch_prefill_experts(const moe_ctx* c, const __nv_bfloat16* x, int T, cudaStream_t s) {
  const int d = c->cfg.d_model, f = c->cfg.d_ff;
  cudaError_t e;
  // the row-major scales [rows][d/16] follow the atoms in the same allocation
  uint8_t* xsf_rows = c->pf_xsf + prefill_max_rows(c->cfg) * (d / 16);
  quant_scatter_x_kernel<<<(T + 7) / 8, 256, 0, s>>>(c->r, x, T, d, c->cfg.top_k, c->cfg.n_shared, c->pf_xq,
                                                     xsf_rows, prefill_accumulates(c->cfg, T) ? c->yacc : nullptr);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // at most this many padded 128-row blocks (the kernel reads the actual count)
  const int max_blocks = (int)(((size_t)T * (c->cfg.top_k + c->cfg.n_shared) + 127) / 128) + c->n_all;
  x_sf_atoms_kernel<<<max_blocks, 256, (size_t)128 * (d / 64 + 1) * 4, s>>>(c->r, xsf_rows, d, c->pf_xsf);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  GemmArgs g{};
  g.r = c->r;
  g.tsc = c->tsc;
  g.status = c->status;
  g.dbg = c->debug_flags;
  g.f = f;
  g.d = d;
  // gate/up + SwiGLU + h quantisation
  g.sfa = c->pf_xsf;
  g.sfb = c->pf_sfa_gu;
  g.M = 2 * f;
  g.K = d;
  g.hq_codes = c->pf_hq;
  g.hq_sf = c->pf_hsf;
  moe_gemm_kernel<kStagesGateUp, 0, kBNGateUp, kEpiGateUp>
      <<<c->sm_count, PlanGateUp::threads, kSmemGateUp, s>>>(c->pf_tm[2], c->pf_tm[0], g);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // down projection -> per-slot outputs
  g.sfa = c->pf_hsf;
  g.sfb = c->pf_sfa_dn;
  g.M = d;
  g.K = f;
  g.yacc = prefill_accumulates(c->cfg, T) ? c->yacc : nullptr;
  g.yexp = c->yexp;
  moe_gemm_kernel<kStagesDown, 1, kBNDown, kEpiDown>
      <<<c->sm_count, PlanDown::threads, kSmemDown, s>>>(c->pf_tm[3], c->pf_tm[1], g);
  return cudaGetLastError();
}

// y = bf16(yacc (+ x)), four elements per thread
namespace {
__global__ void __launch_bounds__(256) prefill_finish_kernel(const float* __restrict__ yacc,
                                                             const __nv_bfloat16* __restrict__ x, size_t n4,
                                                             int residual, __nv_bfloat16* __restrict__ y) {
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n4) return;
  float4 a = reinterpret_cast<const float4*>(yacc)[i];
  if (residual) {
    const uint2 xv = reinterpret_cast<const uint2*>(x)[i];
    a.x += __uint_as_float(xv.x << 16);
    a.y += __uint_as_float(xv.x & 0xFFFF0000u);
    a.z += __uint_as_float(xv.y << 16);
    a.w += __uint_as_float(xv.y & 0xFFFF0000u);
  }
  __nv_bfloat162 lo = __floats2bfloat162_rn(a.x, a.y), hi = __floats2bfloat162_rn(a.z, a.w);
  reinterpret_cast<uint2*>(y)[i] = make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
}
}  // namespace

cudaError_t launch_prefill_finish(const moe_ctx* c, const __nv_bfloat16* x, int T, __nv_bfloat16* y, int residual,
                                  cudaStream_t s) {
  if (!prefill_accumulates(c->cfg, T)) return launch_combine(c, x, T, y, residual, s);
  const size_t n4 = (size_t)T * c->cfg.d_model / 4;
  prefill_finish_kernel<<<(unsigned)((n4 + 255) / 256), 256, 0, s>>>(c->yacc, x, n4, residual, y);
  return cudaGetLastError();
}

// h codes / scales of the last prefill, in slot order (see moe_debug_prefill_h)
namespace {
__global__ void gather_h_kernel(Routing r, int T, int k, int S, int f, const uint8_t* __restrict__ hq,
                                const uint8_t* __restrict__ hsf, uint8_t* __restrict__ out_codes,
                                uint8_t* __restrict__ out_sf) {
  const int slot = blockIdx.x;
  int pos;
  if (slot < T * k) pos = r.slot_pos[slot];
  else pos = slot;  // shared experts: positions T*k + s*T + t == slot
  const int na = *r.n_active;
  const int a = find_seg(r.act_pos, na, pos);
  const int p = r.act_ppos[a] + (pos - r.act_pos[a]);
  for (int i = threadIdx.x; i < f / 2; i += blockDim.x) out_codes[(size_t)slot * (f / 2) + i] = hq[(size_t)p * (f / 2) + i];
  for (int b = threadIdx.x; b < f / 16; b += blockDim.x)
    out_sf[(size_t)slot * (f / 16) + b] = hsf[sf_atom_offset(p, b, f / 64)];
}
}  // namespace

cudaError_t launch_gather_prefill_h(const moe_ctx* c, int T, uint8_t* codes, uint8_t* sf, cudaStream_t s) {
  const int slots = T * (c->cfg.top_k + c->cfg.n_shared);
  if (slots == 0) return cudaSuccess;
  gather_h_kernel<<<slots, 128, 0, s>>>(c->r, T, c->cfg.top_k, c->cfg.n_shared, c->cfg.d_ff, c->pf_hq, c->pf_hsf,
                                        codes, sf);
  return cudaGetLastError();
}

}  // namespace nvmoe
