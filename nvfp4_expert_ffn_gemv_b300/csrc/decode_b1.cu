// Batch-1 decode fast path: two kernels per token, chained with programmatic
// dependent launch (PDL).
//
//   router_b1:  one warp per expert computes its fp32 logit x . W_r[:, e] (+bias)
//               from the transposed router; the W_r row is loaded before the
//               kernel waits on its predecessor, so it streams while the
//               previous token (or layer) is still finishing.
//   top-k:      not a kernel of its own: every CTA of the two kernels below
//               selects the top-k experts and their renormalised softmax
//               weights from the 256 logits with one warp (the same
//               deterministic selection everywhere), so no CTA waits for a
//               single selecting CTA.
//   experts_b1: every CTA owns a slice of the shared expert's hidden rows and a
//               slice of the 6 routed experts' hidden rows (a flat split of the
//               6 x d_ff rows, so all CTAs move the same number of bytes).
//               Before waiting it starts TMA bulk copies of its shared-expert
//               rows; after the wait it selects the experts and copies its
//               routed rows.  Then, per hidden row j it owns:
//                 g_j, u_j  = NVFP4 rows of W_gate / W_up . x
//                 h_j       = silu(g_j) * u_j * w_slot * ts_down   -> global
//   down_b1:    every CTA owns 16 output rows; it fetches those rows of
//               W_down for all 7 slots (routing is already known) while the
//               experts kernel runs, waits for h, and writes
//                 y[r] = sum_slots W_down[r, :] . h_slot  (+ x[r])  in bf16,
//               summing the slots in a fixed order (deterministic).
//
// The pages frame decode as a weight-bandwidth problem ("Recursive Flint
// 40B-A2.5B：まず速さを第一に考えて作られたコーディングモデル", section "このアーキ
// テクチャはメモリ帯域幅に関する主張である"); this path touches each chosen weight
// byte exactly once, with a kernel boundary only between router and experts.
//
// Arithmetic: E2M1 codes are expanded by the hardware cvt to exact f16, x is
// held as f16 after an exact power-of-two prescale (max|x| mapped into
// [2^14, 2^15)), and the products are accumulated in fp32 with the
// mixed-precision FMA (f16 x f16 + f32): every product is exact, only the
// fp32 sums round.  W_down is applied on the tensor cores (mma.sync, exact
// f16 weights against h split into f16 hi + lo, fp32 accumulation).
#include "internal.h"
#include "mma_frag.cuh"
#include "sm100.cuh"

namespace nvmoe {

namespace {

using namespace sm100;

__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

using frag::cvt_e2m1x8;

// acc += lo(a) * lo(b) and acc2 += hi(a) * hi(b), f16 inputs, fp32 accumulate
__device__ __forceinline__ void fma2_mixed(uint32_t a, uint32_t b, float& acc, float& acc2) {
  asm("{\n\t.reg .f16 al, ah, bl, bh;\n\tmov.b32 {al, ah}, %2;\n\tmov.b32 {bl, bh}, %3;\n\t"
      "fma.rn.f32.f16 %0, al, bl, %0;\n\tfma.rn.f32.f16 %1, ah, bh, %1;\n\t}"
      : "+f"(acc), "+f"(acc2) : "r"(a), "r"(b));
}

// One L2 load that the compiler may neither repeat nor drop (a plain __ldcg
// can be rematerialised inside later loops, re-paying the L2 latency each
// time).  No memory clobber, so several of these stay in flight together.
__device__ __forceinline__ float ld_once_f32(const float* p) {
  float v;
  asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(p));
  return v;
}

// 2^k as a float for -126 <= k <= 127
__device__ __forceinline__ float exp2i(int k) { return __uint_as_float((uint32_t)(k + 127) << 23); }

// top-k over E <= 256 logits by one warp; equal values (+0 and -0 included) to
// the lower expert, NaN lowest.
// Only compile-time register indices, so nothing spills to local memory.
__device__ __forceinline__ void warp_topk(const float* logits, int E, int k, int* idx, float* wts) {
  const int lane = threadIdx.x & 31;
  uint32_t key[8];
  float val[8];
  // all 8 loads are issued before any of them is used
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = lane + 32 * i;
    val[i] = ld_once_f32(logits + (e < E ? e : 0));
  }
#pragma unroll
  for (int i = 0; i < 8; ++i)
    if (lane + 32 * i >= E) val[i] = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = lane + 32 * i;
    const uint32_t u = __float_as_uint(val[i] == 0.f ? 0.f : val[i]);   // -0 ties +0
    uint32_t kk = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    if (val[i] != val[i]) kk = 1u;
    key[i] = e < E ? max(kk, 1u) : 0u;
  }
  float my_sel = 0.f;
  int my_e = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    if (j < k) {
      // lane-local argmax over 8 keys as a 3-level tree (ties -> lower index)
      uint32_t k01 = key[1] > key[0] ? key[1] : key[0]; int i01 = key[1] > key[0] ? 1 : 0;
      uint32_t k23 = key[3] > key[2] ? key[3] : key[2]; int i23 = key[3] > key[2] ? 3 : 2;
      uint32_t k45 = key[5] > key[4] ? key[5] : key[4]; int i45 = key[5] > key[4] ? 5 : 4;
      uint32_t k67 = key[7] > key[6] ? key[7] : key[6]; int i67 = key[7] > key[6] ? 7 : 6;
      uint32_t ka = k23 > k01 ? k23 : k01; int ia = k23 > k01 ? i23 : i01;
      uint32_t kb = k67 > k45 ? k67 : k45; int ib = k67 > k45 ? i67 : i45;
      const uint32_t best = kb > ka ? kb : ka;
      const int bi = kb > ka ? ib : ia;
      const uint32_t top = __reduce_max_sync(0xffffffffu, best);
      const uint32_t win =
          __reduce_min_sync(0xffffffffu, (best == top && top != 0) ? (uint32_t)(lane + 32 * bi) : 0xFFFFu);
      float bv = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (i == bi) bv = val[i];
        if (lane + 32 * i == (int)win) key[i] = 0;
      }
      const float sv = __shfl_sync(0xffffffffu, bv, (int)(win & 31));
      if (lane == j) { my_sel = sv; my_e = (int)win < E ? (int)win : 0; }   // k <= E leaves a candidate
    }
  }
  // softmax over the chosen logits, one per lane (lane 0 holds the largest)
  const float m = __shfl_sync(0xffffffffu, my_sel, 0);
  const float z = lane < k ? expf(my_sel - m) : 0.f;
  float sum = z;
#pragma unroll
  for (int o = 4; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);   // k <= 8 lanes
  sum = __shfl_sync(0xffffffffu, sum, 0);
  if (lane < k) {
    idx[lane] = my_e;
    wts[lane] = z / sum;
  }
}

// ---------------------------------------------------------------------------
// router: logits only
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(64) router_b1_kernel(const float* __restrict__ rt, const float* __restrict__ bias,
                                                       int has_bias, const __nv_bfloat16* x, float* logits, int E) {
  constexpr int Q = D / 128;  // float4 of W_r per lane
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  const int e = blockIdx.x * 2 + w;
  float4 wv[Q];
  if (e < E) {
    const float4* p = reinterpret_cast<const float4*>(rt + (size_t)e * D);
#pragma unroll
    for (int q = 0; q < Q; ++q) wv[q] = __ldg(p + l + 32 * q);
  }
  griddep_launch();
  griddep_wait();
  if (e < E) {
    const uint2* xp = reinterpret_cast<const uint2*>(x);
    float acc = 0.f, acc2 = 0.f;
#pragma unroll
    for (int q = 0; q < Q; ++q) {
      const uint2 xv = __ldcg(xp + l + 32 * q);
      acc = fmaf(__uint_as_float(xv.x << 16), wv[q].x, acc);
      acc2 = fmaf(__uint_as_float(xv.x & 0xFFFF0000u), wv[q].y, acc2);
      acc = fmaf(__uint_as_float(xv.y << 16), wv[q].z, acc);
      acc2 = fmaf(__uint_as_float(xv.y & 0xFFFF0000u), wv[q].w, acc2);
    }
    const float s = warp_sum(acc + acc2);
    if (l == 0) logits[e] = s + (has_bias ? bias[e] : 0.f);
  }
}

// ---------------------------------------------------------------------------
// experts
// ---------------------------------------------------------------------------
struct B1Args {
  const float* logits;     // [E] router output
  int32_t* idx_out;        // [k] chosen experts (written by CTA 0, for inspection)
  float* w_out;            // [k] their combine weights
  const __nv_bfloat16* x;
  const uint8_t* rows;     // [n_all][f][gate/up record]
  const float* tsc;
  float* h_out;            // [k + S][f] fp32: w_slot * ts_down * silu(g) * u
  int* status;
  int f, E, k, S, rmax;
  int dbg;                 // debug flags (MOE_DEBUG_FORCE_TIMEOUT)
};

struct Seg {
  int e;       // expert
  int slot;    // routed slot 0..k-1, or k + s for shared expert s
  int j0;      // first hidden row within the expert
  int len;     // rows
  int row0;    // first local row
  float wt;    // combine weight (1 for shared experts)
};

constexpr int kMaxSeg = 8;
constexpr int kB1Threads = 512;
constexpr int kB1Warps = kB1Threads / 32;

// Split [a, b) of a stacked f-space (f = 1 << lf rows per slot) into per-expert
// segments.  Slot s is shared expert e0 + s (weight 1, h slot k + s) when
// `experts` is null, else routed slot s: experts[s] with weight wts[s].
__device__ __forceinline__ int make_segments(Seg* seg, int nseg, int a, int b, int lf, int e0, int k,
                                             const int* experts, const float* wts, int& row) {
  const int f = 1 << lf;
  while (a < b && nseg < kMaxSeg) {
    const int slot = a >> lf, j0 = a & (f - 1);
    const int len = min(b, (slot + 1) << lf) - a;
    Seg& s = seg[nseg++];
    s.e = experts ? experts[slot] : e0 + slot;
    s.slot = experts ? slot : k + slot;
    s.j0 = j0;
    s.len = len;
    s.row0 = row;
    s.wt = experts ? wts[slot] : 1.f;
    row += len;
    a += len;
  }
  return nseg;
}

// Gate/up record of hidden row j (D = d_model):
//   [gate codes D/2][up codes D/2][gate scales D/16][up scales D/16]
// with lane-ordered scales (lane l's 2*CPL bytes contiguous), records of an
// expert stored consecutively, so a CTA that owns rows [j0, j0+len) of an
// expert fetches them with one bulk copy.
template <int D>
struct B1Row {
  static constexpr int kUp = D / 2;
  static constexpr int kGateSc = D;
  static constexpr int kUpSc = D + D / 16;
  static constexpr int kGu = D + D / 8;
};

// Lane 0 posts the byte count, then lane i < n issues segment s0 + i.
template <int D>
__device__ __forceinline__ void issue_segment_copies(const B1Args& a, const Seg* seg, int s0, int s1,
                                                     uint8_t* sm_gu, uint64_t* bar) {
  const int lane = threadIdx.x & 31;
  uint32_t bytes = 0;
  for (int s = s0; s < s1; ++s) bytes += seg[s].len * B1Row<D>::kGu;
  if (lane == 0 && bytes) mbar_arrive_expect_tx(bar, bytes);
  __syncwarp();
  if (lane < s1 - s0) {
    const Seg& g = seg[s0 + lane];
    bulk_load(sm_gu + (size_t)g.row0 * B1Row<D>::kGu, a.rows + ((size_t)g.e * a.f + g.j0) * B1Row<D>::kGu,
              g.len * B1Row<D>::kGu, bar);
  }
}

// Dot of one NVFP4 row (CPL 16-byte chunks per lane) with the lane's f16 x
// registers; returns the lane's partial (block scales applied, not reduced).
template <int CPL>
__device__ __forceinline__ float row_dot_partial(const uint8_t* codes, const uint8_t* sc, const uint32_t (&xh)[CPL][16]) {
  const int lane = threadIdx.x & 31;
  float dot = 0.f;
#pragma unroll
  for (int q = 0; q < CPL; ++q) {
    const uint4 cw = *reinterpret_cast<const uint4*>(codes + (lane + 32 * q) * 16);
    const uint32_t ws[4] = {cw.x, cw.y, cw.z, cw.w};
    float b[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      uint32_t o[4];
      cvt_e2m1x8(ws[v], o);
#pragma unroll
      for (int p = 0; p < 4; ++p) fma2_mixed(o[p], xh[q][4 * v + p], b[v >> 1][0], b[v >> 1][1]);
    }
    const uint32_t s2 = *reinterpret_cast<const uint16_t*>(sc + lane * 2 * CPL + 2 * q);
    const float2 s01 = e4m3x2_to_f32x2(s2);
    dot = fmaf(b[0][0] + b[0][1], s01.x, dot);
    dot = fmaf(b[1][0] + b[1][1], s01.y, dot);
  }
  return dot;
}

// ---------------------------------------------------------------------------
// experts: gate/up + SwiGLU for this CTA's hidden rows -> h
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(kB1Threads, 1) experts_b1_kernel(B1Args a) {
  constexpr int CPL = D / 1024;  // 16-byte code chunks per lane per row
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* sm_gu = smem;                                                 // [rmax][gate/up record]
  // x in fp32, float4 f of 32-column chunk c = l + 32q stored at float4 slot
  // (8q + f) * 32 + l: the 32 lanes of a warp, each reading float4 f of its
  // own chunk, touch 512 consecutive bytes (a chunk-contiguous layout would
  // put all 32 lanes on the same four banks)
  float* xs = reinterpret_cast<float*>(sm_gu + (size_t)a.rmax * B1Row<D>::kGu);  // [D]
  __shared__ Seg seg[kMaxSeg];
  __shared__ int nseg_sh, nseg_all, n_rows, nsh_rows_s, top_idx[8];
  __shared__ float top_w[8];
  __shared__ uint32_t wmax[kB1Warps];
  __shared__ __align__(8) uint64_t bars[2];  // shared-expert rows, routed rows
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x, c = blockIdx.x;
  const int f = a.f;
  const int lf = 31 - __clz(f);

  if (threadIdx.x == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    fence_barrier_init();
  }
  __syncthreads();

  // ---- shared experts: independent of routing, copy before waiting ----
  if (warp == 0) {
    if (lane == 0) {
      int row = 0;
      const int Nsh = a.S * f;
      nseg_sh = make_segments(seg, 0, c * Nsh / G, (c + 1) * Nsh / G, lf, a.E, a.k, nullptr, nullptr, row);
      n_rows = row;
      nsh_rows_s = row;
    }
    __syncwarp();
    issue_segment_copies<D>(a, seg, 0, nseg_sh, sm_gu, &bars[0]);
    asm volatile("bar.arrive 1, 64;" ::: "memory");   // segment table handed to warp 1
  }
  griddep_wait();

  if (warp == 1) {
    // ---- routed experts: top-k of the logits (the router grid has completed).
    // Warp 1 rather than warp 0: the warp that issued the shared-expert bulk
    // copies runs several times slower for a while afterwards. ----
    asm volatile("bar.sync 1, 64;" ::: "memory");
    warp_topk(a.logits, a.E, a.k, top_idx, top_w);
    __syncwarp();
    if (c == 0 && lane < a.k) {
      a.idx_out[lane] = top_idx[lane];
      a.w_out[lane] = top_w[lane];
    }
    if (lane == 0) {
      int row = n_rows;
      const int Nr = a.k * f;
      nseg_all = make_segments(seg, nseg_sh, c * Nr / G, (c + 1) * Nr / G, lf, 0, a.k, top_idx, top_w, row);
      n_rows = row;
    }
    __syncwarp();
    issue_segment_copies<D>(a, seg, nseg_sh, nseg_all, sm_gu, &bars[1]);
  } else {
    // ---- x -> shared memory (fp32), block max of |x| (every warp but warp 1) ----
    float m = 0.f;
    for (int i = warp == 0 ? lane : threadIdx.x - 32; i < D / 8; i += kB1Threads - 32) {
      const uint4 t = __ldcg(reinterpret_cast<const uint4*>(a.x) + i);
      const uint32_t u[4] = {t.x, t.y, t.z, t.w};
      float4 lo, hi;
      lo.x = __uint_as_float(u[0] << 16); lo.y = __uint_as_float(u[0] & 0xFFFF0000u);
      lo.z = __uint_as_float(u[1] << 16); lo.w = __uint_as_float(u[1] & 0xFFFF0000u);
      hi.x = __uint_as_float(u[2] << 16); hi.y = __uint_as_float(u[2] & 0xFFFF0000u);
      hi.z = __uint_as_float(u[3] << 16); hi.w = __uint_as_float(u[3] & 0xFFFF0000u);
      const int ch = i >> 2;                                              // 32-column chunk
      const int slot = ((ch >> 5) * 8 + (i & 3) * 2) * 32 + (ch & 31);
      reinterpret_cast<float4*>(xs)[slot] = lo;
      reinterpret_cast<float4*>(xs)[slot + 32] = hi;
      m = fmaxf(m, fmaxf(fmaxf(fabsf(lo.x), fabsf(lo.y)), fmaxf(fabsf(lo.z), fabsf(lo.w))));
      m = fmaxf(m, fmaxf(fmaxf(fabsf(hi.x), fabsf(hi.y)), fmaxf(fabsf(hi.z), fabsf(hi.w))));
    }
    const uint32_t mb = __reduce_max_sync(0xffffffffu, __float_as_uint(m));
    if (lane == 0) wmax[warp] = mb;
  }
  __syncthreads();
  // the down-projection kernel may start fetching its weights now
  griddep_launch();

  // ---- x as prescaled f16 registers: lane l holds the columns of chunks l + 32q ----
  uint32_t mb = 0;
  for (int w = 0; w < kB1Warps; ++w)
    if (w != 1) mb = max(mb, wmax[w]);
  const int ex = (int)((mb >> 23) & 0xFF) - 127;
  const int shift = (mb == 0u) ? 0 : max(-126, min(127, 14 - ex));
  uint32_t xh[CPL][16];
  {
    const float sc = exp2i(shift);
#pragma unroll
    for (int q = 0; q < CPL; ++q) {
      const float4* xp = reinterpret_cast<const float4*>(xs) + q * 8 * 32 + lane;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float4 v = xp[i * 32];
        __half2 h0 = __floats2half2_rn(v.x * sc, v.y * sc), h1 = __floats2half2_rn(v.z * sc, v.w * sc);
        xh[q][2 * i] = *reinterpret_cast<uint32_t*>(&h0);
        xh[q][2 * i + 1] = *reinterpret_cast<uint32_t*>(&h1);
      }
    }
  }
  const int nrows = n_rows, nsh_rows = nsh_rows_s, nsegs = nseg_all;
  bool ok = true;

  // ---- one warp per hidden row: gate and up dots, SwiGLU, fold w * ts_down ----
  const float unshift = exp2i(-shift);
  bool waited_sh = false, waited_rt = false;
  for (int row = warp; row < nrows; row += kB1Warps) {
    if (row < nsh_rows) {
      if (!waited_sh) { ok &= wait_parity(&bars[0], 0); waited_sh = true; }
    } else if (!waited_rt) {
      ok &= wait_parity(&bars[1], 0);
      waited_rt = true;
    }
    const uint8_t* base = sm_gu + (size_t)row * B1Row<D>::kGu;
    float g = row_dot_partial<CPL>(base, base + B1Row<D>::kGateSc, xh);
    float u = row_dot_partial<CPL>(base + B1Row<D>::kUp, base + B1Row<D>::kUpSc, xh);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      g += __shfl_xor_sync(0xffffffffu, g, o);
      u += __shfl_xor_sync(0xffffffffu, u, o);
    }
    if (lane == 0) {
      int s = 0;
      while (s + 1 < nsegs && row >= seg[s + 1].row0) ++s;
      const Seg& sg = seg[s];
      const float gg = g * unshift * a.tsc[sg.e * 3 + 0];
      const float uu = u * unshift * a.tsc[sg.e * 3 + 1];
      a.h_out[(size_t)sg.slot * f + sg.j0 + (row - sg.row0)] = silu_f(gg) * uu * sg.wt * a.tsc[sg.e * 3 + 2];
    }
  }
  if (!ok) latch_status(a.status, MOE_ERR_TIMEOUT);
  // after every wait completed, the debug flag reports a timeout anyway
  if (threadIdx.x == 0 && (a.dbg & MOE_DEBUG_FORCE_TIMEOUT)) latch_status(a.status, MOE_ERR_TIMEOUT);
}

// ---------------------------------------------------------------------------
// down projection + combine: CTA owns kRD output rows, sums every slot
// ---------------------------------------------------------------------------
// The 16 rows of a CTA are one MMA tile (m16n8k16): A = W_down rows (E2M1 code
// times E4M3 block scale, exact in f16), B column 0 = hi and column 1 = lo of
// h (f16 split after a per-slot power-of-two prescale), so every k step costs
// one MMA and the products are exact.  The k range (slots x d_ff) is cut into
// 128-wide chunks; warp w takes chunks w, w + 8, ... (two accumulators, so
// the MMA chain of a chunk is four steps deep) and the eight warp sums are
// added in a fixed order.
constexpr int kRD = 16;          // output rows per CTA (one MMA tile)
constexpr int kDThreads = 256;
constexpr int kDWarps = kDThreads / 32;
constexpr int kMaxSlots = 12;

struct DnArgs {
  const float* logits;
  const float* h;                 // [k + S][f]
  const __nv_bfloat16* x;
  __nv_bfloat16* y;
  const uint8_t* dn_codes;        // [n_all][d][f/2]
  const uint8_t* dn_scales;       // [n_all][d][f/16]
  int* status;
  int d, f, E, k, S, residual;
  int dbg;                        // debug flags (MOE_DEBUG_FORCE_TIMEOUT)
};

// shared-memory plan of down_b1 for NS slots (byte offsets)
template <int F>
struct DnB1Smem {
  static constexpr int FB = F / 2, FS = F / 16;   // code / scale bytes per row
  __host__ __device__ static size_t codes(int) { return 0; }  // [NS][kRD][FB]
  __host__ __device__ static size_t scales(int ns) { return (size_t)ns * kRD * FB; }  // [NS][kRD][FS]
  __host__ __device__ static size_t hi(int ns) { return scales(ns) + (size_t)ns * kRD * FS; }  // [NS][F] f16, k-permuted
  __host__ __device__ static size_t lo(int ns) { return hi(ns) + (size_t)ns * F * 2; }  // [NS][F] f16, k-permuted
  __host__ __device__ static size_t unshift(int ns) { return lo(ns) + (size_t)ns * F * 2; }  // [kMaxSlots] fp32
  __host__ __device__ static size_t red(int ns) { return unshift(ns) + kMaxSlots * sizeof(float); }  // [kDWarps][kRD] fp32
  __host__ __device__ static size_t total(int ns) { return red(ns) + kDWarps * kRD * sizeof(float); }
};

template <int F>
__global__ void __launch_bounds__(kDThreads) down_b1_kernel(DnArgs a) {
  static_assert(F % 128 == 0, "down_b1 works on 128-wide k chunks of d_ff");
  using L = DnB1Smem<F>;
  constexpr int FB = L::FB, FS = L::FS, NCH = F / 128;
  extern __shared__ __align__(128) uint8_t smem[];
  const int NS = a.k + a.S;
  uint8_t* sc_codes = smem + L::codes(NS);
  uint8_t* sc_scales = smem + L::scales(NS);
  uint8_t* h_hi = smem + L::hi(NS);
  uint8_t* h_lo = smem + L::lo(NS);
  float* unshift = reinterpret_cast<float*>(smem + L::unshift(NS));
  float* red = reinterpret_cast<float*>(smem + L::red(NS));
  __shared__ __align__(8) uint64_t bar;
  __shared__ int sel_idx[8];
  __shared__ float sel_w[8];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r0 = blockIdx.x * kRD;

  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  // the logits are final (the router finished before the experts kernel passed
  // its wait, and that kernel released this one afterwards): select the same
  // experts and fetch their W_down rows now (warp 1: warp 0 initialised the
  // mbarrier and runs slowly for a while afterwards)
  if (warp == 1) {
    warp_topk(a.logits, a.E, a.k, sel_idx, sel_w);
    __syncwarp();
    int e = 0;
    if (lane < NS) e = lane < a.k ? sel_idx[lane] : a.E + (lane - a.k);
    if (lane == 0) mbar_arrive_expect_tx(&bar, (uint32_t)NS * kRD * (FB + FS));
    __syncwarp();
    if (lane < NS) {
      bulk_load(sc_codes + (size_t)lane * kRD * FB, a.dn_codes + ((size_t)e * a.d + r0) * FB, kRD * FB, &bar);
      bulk_load(sc_scales + (size_t)lane * kRD * FS, a.dn_scales + ((size_t)e * a.d + r0) * FS, kRD * FS, &bar);
    }
  }
  griddep_launch();
  griddep_wait();
  // h of every slot (written by the experts kernel) -> prescaled f16 hi + lo,
  // k-permuted per 128 chunk; warp w converts slots w, w + 8
  for (int s = warp; s < NS; s += kDWarps) {
    const float4* src = reinterpret_cast<const float4*>(a.h + (size_t)s * F);
    float4 v[F / 128];
    float m = 0.f;
#pragma unroll
    for (int i = 0; i < F / 128; ++i) {
      v[i] = __ldcg(src + lane + 32 * i);
      m = fmaxf(m, fmaxf(fmaxf(fabsf(v[i].x), fabsf(v[i].y)), fmaxf(fabsf(v[i].z), fabsf(v[i].w))));
    }
    const int shift = frag::prescale_shift(__reduce_max_sync(0xffffffffu, __float_as_uint(m)));
    const float sc = frag::pow2i(shift);
#pragma unroll
    for (int i = 0; i < F / 128; ++i) {
      const int k0 = 4 * (lane + 32 * i), kp = k0 % 128;
      const size_t off = (size_t)s * F * 2 + (k0 / 128) * 256 + frag::perm_off(kp / 32, (kp % 32) / 4);
      uint2 hi, lo;
      frag::split_hi_lo(v[i].x * sc, v[i].y * sc, v[i].z * sc, v[i].w * sc, hi, lo);
      *reinterpret_cast<uint2*>(h_hi + off) = hi;
      *reinterpret_cast<uint2*>(h_lo + off) = lo;
    }
    if (lane == 0) unshift[s] = frag::pow2i(-shift);
  }
  __syncthreads();
  const bool ok = wait_parity(&bar, 0);
  if (!ok) latch_status(a.status, MOE_ERR_TIMEOUT);
  if (threadIdx.x == 0 && (a.dbg & MOE_DEBUG_FORCE_TIMEOUT)) latch_status(a.status, MOE_ERR_TIMEOUT);

  // MMA lane roles: gq = lane / 4 is the A row (and B column), c = lane % 4
  // the quad position; B columns 0 (hi) and 1 (lo) come from lanes 0..7.
  const int gq = lane >> 2, c = lane & 3;
  float y0 = 0.f, y8 = 0.f;
  for (int u = warp; u < NS * NCH; u += kDWarps) {
    const int s = u / NCH, ch = u - s * NCH;
    const uint8_t* cg = sc_codes + ((size_t)s * kRD + gq) * FB + ch * 64 + c * 16;
    const uint4 wg = *reinterpret_cast<const uint4*>(cg);
    const uint4 wg8 = *reinterpret_cast<const uint4*>(cg + 8 * FB);
    const uint8_t* sp = sc_scales + ((size_t)s * kRD + gq) * FS + ch * 8 + c * 2;
    const uint32_t s2 = frag::cvt_e4m3x2_f16x2(*reinterpret_cast<const uint16_t*>(sp));
    const uint32_t s28 = frag::cvt_e4m3x2_f16x2(*reinterpret_cast<const uint16_t*>(sp + 8 * FS));
    const uint8_t* hb = (gq == 0 ? h_hi : h_lo) + (size_t)s * F * 2 + ch * 256;
    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int wd = 0; wd < 4; ++wd) {
      const uint32_t sg = wd < 2 ? frag::bcast_lo(s2) : frag::bcast_hi(s2);
      const uint32_t sg8 = wd < 2 ? frag::bcast_lo(s28) : frag::bcast_hi(s28);
      uint32_t afp[2][4];
      frag::a_frag_pair(afp[0], afp[1], frag::word_of(wg, wd), frag::word_of(wg8, wd), sg, sg8);
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        const uint2 b = gq < 2 ? frag::lds64(hb + frag::perm_off(c, 2 * wd + h2)) : make_uint2(0u, 0u);
        frag::mma_f16(acc[h2], afp[h2], b.x, b.y);
      }
    }
    // lanes with c == 0 hold columns 0 (hi) and 1 (lo) of rows gq and gq + 8
    const float us = unshift[s];
    y0 = fmaf((acc[0][0] + acc[0][1]) + (acc[1][0] + acc[1][1]), us, y0);
    y8 = fmaf((acc[0][2] + acc[0][3]) + (acc[1][2] + acc[1][3]), us, y8);
  }
  if (c == 0) {
    red[warp * kRD + gq] = y0;
    red[warp * kRD + gq + 8] = y8;
  }
  __syncthreads();
  if (threadIdx.x < kRD) {
    float y = 0.f;
#pragma unroll
    for (int w = 0; w < kDWarps; ++w) y += red[w * kRD + threadIdx.x];
    if (a.residual) y += __bfloat162float(a.x[r0 + threadIdx.x]);
    a.y[r0 + threadIdx.x] = __float2bfloat16_rn(y);
  }
}

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

int ceil_div(long a, long b) { return (int)((a + b - 1) / b); }

}  // namespace

bool b1_supported(const moe_config& c) {
  return c.weight_format == MOE_W_NVFP4 && (c.d_model == 2048 || c.d_model == 4096) && c.d_ff == 512 &&
         c.n_experts <= 256 && c.top_k <= 8 && c.n_shared >= 1 && c.top_k + c.n_shared <= kMaxSlots;
}

// Choose the expert grid and shared-memory plan (also used by moe_init to size buffers).
bool b1_plan(const moe_config& c, int sm_count, int ctas_per_sm, int* grid, int* rmax, int* nbmax, size_t* smem) {
  const int G = sm_count * ctas_per_sm;
  const int f = c.d_ff, D = c.d_model;
  const int Ls = ceil_div((long)c.n_shared * f, G), Lr = ceil_div((long)c.top_k * f, G);
  const int segs_s = ceil_div(Ls, f) + 1, segs_r = ceil_div(Lr, f) + 1;
  if (segs_s > 8 || segs_r > 8 || segs_s + segs_r > kMaxSeg) return false;
  *grid = G;
  *rmax = Ls + Lr;
  *nbmax = 0;
  *smem = (size_t)(*rmax) * (D + D / 8) + (size_t)D * sizeof(float) + 64;
  return *smem <= 200 * 1024 && D % kRD == 0;
}

size_t b1_row_bytes(int d) { return (size_t)d + d / 8; }

static size_t down_smem(const moe_config& c) {
  return DnB1Smem<512>::total(c.top_k + c.n_shared);   // b1_supported() requires d_ff = 512
}

// The three kernels of a token overlap through PDL only if an SM can hold an
// experts CTA and a down CTA (and a router CTA) at once, so every one of them
// asks for the largest shared-memory carveout: with a carveout sized for one
// kernel alone, the next kernel's CTAs would wait for the SM to drain.
template <typename K>
cudaError_t max_carveout(K kern) {
  return cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
}

cudaError_t prepare_b1_kernels(const moe_ctx* c) {
  if (!c->b1_enabled) return cudaSuccess;
  const bool d2k = c->cfg.d_model == 2048;
  cudaError_t e = d2k ? cudaFuncSetAttribute(experts_b1_kernel<2048>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)c->b1_smem)
                      : cudaFuncSetAttribute(experts_b1_kernel<4096>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)c->b1_smem);
  if (e == cudaSuccess) e = d2k ? max_carveout(experts_b1_kernel<2048>) : max_carveout(experts_b1_kernel<4096>);
  if (e == cudaSuccess) e = d2k ? max_carveout(router_b1_kernel<2048>) : max_carveout(router_b1_kernel<4096>);
  if (e == cudaSuccess) e = max_carveout(down_b1_kernel<512>);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(down_b1_kernel<512>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)down_smem(c->cfg));
}

cudaError_t launch_router_b1(const moe_ctx* c, const __nv_bfloat16* x, cudaStream_t s) {
  const int E = c->cfg.n_experts;
  const dim3 grid((E + 1) / 2), block(64);
  if (c->cfg.d_model == 2048)
    return launch_pdl(router_b1_kernel<2048>, grid, block, 0, s, (const float*)c->router_t, (const float*)c->bias,
                      c->has_bias, x, c->logits, E);
  return launch_pdl(router_b1_kernel<4096>, grid, block, 0, s, (const float*)c->router_t, (const float*)c->bias,
                    c->has_bias, x, c->logits, E);
}

cudaError_t launch_experts_b1(const moe_ctx* c, const __nv_bfloat16* x, __nv_bfloat16* y, int residual,
                              cudaStream_t s) {
  B1Args a;
  a.logits = c->logits;
  a.idx_out = c->r.idx;
  a.w_out = c->r.w;
  a.x = x;
  a.rows = c->b1_rows;
  a.tsc = c->tsc;
  a.h_out = c->h;
  a.status = c->status;
  a.f = c->cfg.d_ff;
  a.E = c->cfg.n_experts;
  a.k = c->cfg.top_k;
  a.S = c->cfg.n_shared;
  a.rmax = c->b1_rmax;
  a.dbg = c->debug_flags;
  cudaError_t e = c->cfg.d_model == 2048
                      ? launch_pdl(experts_b1_kernel<2048>, dim3(c->b1_grid), dim3(kB1Threads), c->b1_smem, s, a)
                      : launch_pdl(experts_b1_kernel<4096>, dim3(c->b1_grid), dim3(kB1Threads), c->b1_smem, s, a);
  if (e != cudaSuccess) return e;
  DnArgs d;
  d.logits = c->logits;
  d.h = c->h;
  d.x = x;
  d.y = y;
  d.dn_codes = c->dn_codes;
  d.dn_scales = c->dn_scales;
  d.status = c->status;
  d.d = c->cfg.d_model;
  d.f = c->cfg.d_ff;
  d.E = c->cfg.n_experts;
  d.k = c->cfg.top_k;
  d.S = c->cfg.n_shared;
  d.residual = residual;
  d.dbg = c->debug_flags;
  return launch_pdl(down_b1_kernel<512>, dim3(d.d / kRD), dim3(kDThreads), down_smem(c->cfg), s, d);
}

}  // namespace nvmoe
