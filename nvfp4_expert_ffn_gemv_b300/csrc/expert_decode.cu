// Decode experts: fused NVFP4 dequantisation + SwiGLU GEMV (gate/up), then the
// down projection, for every (active expert, token) pair the router produced.
//
// The Flint pages frame decode as moving weights from memory to the ALUs
// ("Recursive Flint 40B-A2.5B：まず速さを第一に考えて作られたコーディングモデル",
// section "このアーキテクチャはメモリ帯域幅に関する主張である"), so both kernels
// stream each chosen expert's NVFP4 bytes exactly once per call with 16-byte
// coalesced loads and do all arithmetic in registers:
//   value = e2m1 * e4m3 * ts;  per 16-element block the kernel sums e2m1 * x
//   (exact products, fp32 sum), multiplies once by the block's E4M3 scale and
//   once per row by the tensor scale.
// Activations stay exact (bf16 -> fp32) and h is kept in fp32.
//
// Work units (grid-stride over a device-side count, so one launch serves any
// routing):  gate/up unit = (active expert, 16 consecutive rows of h) -> 32
// weight rows;  down unit = (active expert, 64 output rows).  Each unit loops
// over the expert's tokens in groups of kTG.
#include "internal.h"

namespace nvmoe {

namespace {

constexpr int kTG = 8;         // tokens per pass over a unit's weights
constexpr int kThreads = 256;  // 8 warps

struct ExpertArgs {
  Routing r;
  const __nv_bfloat16* x;  // [T][d]
  const uint8_t* gu_codes;
  const uint8_t* gu_scales;
  const uint8_t* dn_codes;
  const uint8_t* dn_scales;
  const __nv_bfloat16* gu_bf16;
  const __nv_bfloat16* dn_bf16;
  const float* tsc;
  float* h;     // [P][f]
  float* yexp;  // [P][d]
  int d, f, T;
};

// 32 consecutive weights of one row starting at column c*32, times 32 x values
// per token, accumulated into acc[t].
template <bool kBF16>
__device__ __forceinline__ void load_chunk(const ExpertArgs& a, const uint8_t* codes_row,
                                           const uint8_t* scales_row, const __nv_bfloat16* bf_row,
                                           int c, uint4 (&raw)[4], uint32_t& sc) {
  if constexpr (kBF16) {
    const uint4* p = reinterpret_cast<const uint4*>(bf_row + c * 32);
#pragma unroll
    for (int q = 0; q < 4; ++q) raw[q] = __ldg(p + q);
    sc = 0;
  } else {
    raw[0] = __ldg(reinterpret_cast<const uint4*>(codes_row + c * 16));
    sc = __ldg(reinterpret_cast<const uint16_t*>(scales_row + c * 2));
  }
}

template <bool kBF16>
__device__ __forceinline__ void fma_chunk(const uint4 (&raw)[4], uint32_t sc, const float* xs,
                                          int x_stride, int c, int nt, float (&acc)[kTG]) {
  float wv[32];
  float s0 = 1.f, s1 = 1.f;
  if constexpr (kBF16) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t u[4] = {raw[q].x, raw[q].y, raw[q].z, raw[q].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        wv[q * 8 + 2 * i] = __uint_as_float(u[i] << 16);
        wv[q * 8 + 2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
      }
    }
  } else {
    decode32_e2m1(raw[0], wv);
    const float2 s = e4m3x2_to_f32x2(sc);
    s0 = s.x;
    s1 = s.y;
  }
#pragma unroll
  for (int t = 0; t < kTG; ++t) {
    if (t < nt) {
      const float4* xp = reinterpret_cast<const float4*>(xs + (size_t)t * x_stride + c * 32);
      float b0 = 0.f, b1 = 0.f;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float4 xv = xp[q];
        b0 = fmaf(wv[4 * q + 0], xv.x, b0);
        b0 = fmaf(wv[4 * q + 1], xv.y, b0);
        b0 = fmaf(wv[4 * q + 2], xv.z, b0);
        b0 = fmaf(wv[4 * q + 3], xv.w, b0);
      }
#pragma unroll
      for (int q = 4; q < 8; ++q) {
        const float4 xv = xp[q];
        b1 = fmaf(wv[4 * q + 0], xv.x, b1);
        b1 = fmaf(wv[4 * q + 1], xv.y, b1);
        b1 = fmaf(wv[4 * q + 2], xv.z, b1);
        b1 = fmaf(wv[4 * q + 3], xv.w, b1);
      }
      acc[t] = fmaf(b0, s0, acc[t]);
      acc[t] = fmaf(b1, s1, acc[t]);
    }
  }
}

// A warp computes ROWS rows of a weight matrix with C chunks (of 32 columns)
// per row against kTG tokens in shared memory; row_ptr(i) gives the i-th row.
// Results (unscaled by the tensor scale) go to out[i * kTG + t].
template <int C, int ROWS, bool kBF16, typename RowFn>
__device__ __forceinline__ void warp_rows(const ExpertArgs& a, RowFn row_of, const float* xs,
                                          int x_stride, int nt, float* out) {
  constexpr int LPR = C < 32 ? C : 32;   // lanes per row
  constexpr int RPP = 32 / LPR;          // rows per pass
  constexpr int NPASS = ROWS / RPP;      // passes
  constexpr int CPL = C / LPR;           // chunks per lane per pass
  static_assert(ROWS % RPP == 0, "rows per warp must be a multiple of rows per pass");
  const int lane = threadIdx.x & 31;
  const int sub = lane / LPR, cl = lane % LPR;
  uint4 raw[NPASS][CPL][kBF16 ? 4 : 1];
  uint32_t sc[NPASS][CPL];
#pragma unroll
  for (int p = 0; p < NPASS; ++p) {
    const int i = p * RPP + sub;
    const uint8_t* cr;
    const uint8_t* sr;
    const __nv_bfloat16* br;
    row_of(i, cr, sr, br);
#pragma unroll
    for (int q = 0; q < CPL; ++q) {
      uint4 tmp[4];
      load_chunk<kBF16>(a, cr, sr, br, cl + LPR * q, tmp, sc[p][q]);
#pragma unroll
      for (int z = 0; z < (kBF16 ? 4 : 1); ++z) raw[p][q][z] = tmp[z];
    }
  }
#pragma unroll
  for (int p = 0; p < NPASS; ++p) {
    float acc[kTG];
#pragma unroll
    for (int t = 0; t < kTG; ++t) acc[t] = 0.f;
#pragma unroll
    for (int q = 0; q < CPL; ++q) {
      uint4 tmp[4];
#pragma unroll
      for (int z = 0; z < 4; ++z) tmp[z] = raw[p][q][kBF16 ? z : 0];
      fma_chunk<kBF16>(tmp, sc[p][q], xs, x_stride, cl + LPR * q, nt, acc);
    }
#pragma unroll
    for (int t = 0; t < kTG; ++t) {
      if (t < nt) {
        const float v = segment_sum(acc[t], LPR);
        if (cl == 0) out[(p * RPP + sub) * kTG + t] = v;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// gate/up + SwiGLU
// ---------------------------------------------------------------------------
template <int CD, bool kBF16>
__global__ void __launch_bounds__(kThreads) gateup_decode_kernel(ExpertArgs a) {
  extern __shared__ float4 smem4[];
  float* xs = reinterpret_cast<float*>(smem4);      // [kTG][d]
  __shared__ float res[32 * kTG];                   // [32 rows][kTG]
  const int d = a.d, f = a.f;
  const int units_per_e = f / 16;
  const int n_units = *a.r.n_active * units_per_e;
  const int warp = threadIdx.x >> 5;
  for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
    const int ai = u / units_per_e, j0 = (u % units_per_e) * 16;
    const int e = a.r.act_e[ai], pos0 = a.r.act_pos[ai], n = a.r.act_n[ai];
    const float ts_g = kBF16 ? 1.f : a.tsc[e * 3 + 0];
    const float ts_u = kBF16 ? 1.f : a.tsc[e * 3 + 1];
    for (int tok0 = 0; tok0 < n; tok0 += kTG) {
      const int nt = min(kTG, n - tok0);
      __syncthreads();
      for (int i = threadIdx.x; i < nt * (d / 8); i += kThreads) {
        const int t = i / (d / 8), c8 = i % (d / 8);
        const int tok = a.r.pos_tok[pos0 + tok0 + t];
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(a.x + (size_t)tok * d) + c8);
        float4* dst = reinterpret_cast<float4*>(xs + (size_t)t * d + c8 * 8);
        dst[0] = make_float4(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xFFFF0000u),
                             __uint_as_float(v.y << 16), __uint_as_float(v.y & 0xFFFF0000u));
        dst[1] = make_float4(__uint_as_float(v.z << 16), __uint_as_float(v.z & 0xFFFF0000u),
                             __uint_as_float(v.w << 16), __uint_as_float(v.w & 0xFFFF0000u));
      }
      __syncthreads();
      // warp w: rows 4w..4w+3 of the unit; rows 0..15 gate, 16..31 up
      auto row_of = [&](int i, const uint8_t*& cr, const uint8_t*& sr, const __nv_bfloat16*& br) {
        const int r = warp * 4 + i;
        const int j = j0 + (r & 15);
        const int gr = (r < 16) ? gu_row_of_gate(j) : gu_row_of_up(j);
        const size_t row = (size_t)e * 2 * f + gr;
        cr = a.gu_codes + row * (d / 2);
        sr = a.gu_scales + row * (d / 16);
        br = a.gu_bf16 + row * d;
      };
      warp_rows<CD, 4, kBF16>(a, row_of, xs, d, nt, res + warp * 4 * kTG);
      __syncthreads();
      for (int i = threadIdx.x; i < 16 * nt; i += kThreads) {
        const int jj = i & 15, t = i >> 4;
        const float g = res[jj * kTG + t] * ts_g;
        const float uv = res[(16 + jj) * kTG + t] * ts_u;
        a.h[(size_t)(pos0 + tok0 + t) * f + j0 + jj] = silu_f(g) * uv;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// down projection: yexp[p] = W_down h[p]
// ---------------------------------------------------------------------------
template <int CF, bool kBF16>
__global__ void __launch_bounds__(kThreads) down_decode_kernel(ExpertArgs a) {
  extern __shared__ float4 smem4[];
  float* hs = reinterpret_cast<float*>(smem4);      // [kTG][f]
  __shared__ float res[64 * kTG];
  const int d = a.d, f = a.f;
  const int units_per_e = d / 64;
  const int n_units = *a.r.n_active * units_per_e;
  const int warp = threadIdx.x >> 5;
  for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
    const int ai = u / units_per_e, r0 = (u % units_per_e) * 64;
    const int e = a.r.act_e[ai], pos0 = a.r.act_pos[ai], n = a.r.act_n[ai];
    const float ts_d = kBF16 ? 1.f : a.tsc[e * 3 + 2];
    for (int tok0 = 0; tok0 < n; tok0 += kTG) {
      const int nt = min(kTG, n - tok0);
      __syncthreads();
      for (int i = threadIdx.x; i < nt * (f / 4); i += kThreads) {
        const int t = i / (f / 4), c4 = i % (f / 4);
        reinterpret_cast<float4*>(hs + (size_t)t * f)[c4] =
            reinterpret_cast<const float4*>(a.h + (size_t)(pos0 + tok0 + t) * f)[c4];
      }
      __syncthreads();
      auto row_of = [&](int i, const uint8_t*& cr, const uint8_t*& sr, const __nv_bfloat16*& br) {
        const size_t row = (size_t)e * d + r0 + warp * 8 + i;
        cr = a.dn_codes + row * (f / 2);
        sr = a.dn_scales + row * (f / 16);
        br = a.dn_bf16 + row * f;
      };
      warp_rows<CF, 8, kBF16>(a, row_of, hs, f, nt, res + warp * 8 * kTG);
      __syncthreads();
      for (int i = threadIdx.x; i < 64 * nt; i += kThreads) {
        const int rr = i & 63, t = i >> 6;
        a.yexp[(size_t)(pos0 + tok0 + t) * d + r0 + rr] = res[rr * kTG + t] * ts_d;
      }
    }
  }
}

ExpertArgs make_args(const moe_ctx* c, const __nv_bfloat16* x, int T) {
  ExpertArgs a;
  a.r = c->r;
  a.x = x;
  a.gu_codes = c->gu_codes;
  a.gu_scales = c->gu_scales;
  a.dn_codes = c->dn_codes;
  a.dn_scales = c->dn_scales;
  a.gu_bf16 = c->gu_bf16;
  a.dn_bf16 = c->dn_bf16;
  a.tsc = c->tsc;
  a.h = c->h;
  a.yexp = c->yexp;
  a.d = c->cfg.d_model;
  a.f = c->cfg.d_ff;
  a.T = T;
  return a;
}

// Launch (prepare == false) or, once at context set-up, raise the kernel's
// dynamic shared-memory limit (prepare == true), so forward calls make no
// attribute changes and can be captured in a CUDA graph.
template <typename K>
cudaError_t launch_k(K kern, int grid, size_t smem, cudaStream_t s, const ExpertArgs& a, bool prepare) {
  if (prepare) return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  kern<<<grid, kThreads, smem, s>>>(a);
  return cudaGetLastError();
}

int max_active(const moe_ctx* c, int T) {
  const int routed = T * c->cfg.top_k < c->cfg.n_experts ? T * c->cfg.top_k : c->cfg.n_experts;
  return routed + c->cfg.n_shared;
}

}  // namespace

cudaError_t gateup_decode(const moe_ctx* c, const __nv_bfloat16* x, int T, cudaStream_t s,
                          bool prepare) {
  const ExpertArgs a = make_args(c, x, T);
  const int units = max_active(c, T) * (a.f / 16);
  const int grid = units < 2 * c->sm_count ? units : 2 * c->sm_count;
  const size_t smem = (size_t)kTG * a.d * sizeof(float);
  const bool bf = c->cfg.weight_format == MOE_W_BF16;
  switch (a.d) {
#define GU_CASE(D)                                                                          \
  case D:                                                                                   \
    return bf ? launch_k(gateup_decode_kernel<D / 32, true>, grid, smem, s, a, prepare)              \
              : launch_k(gateup_decode_kernel<D / 32, false>, grid, smem, s, a, prepare);
    GU_CASE(256)
    GU_CASE(512)
    GU_CASE(1024)
    GU_CASE(2048)
    GU_CASE(4096)
#undef GU_CASE
    default:
      return cudaErrorInvalidValue;
  }
}

cudaError_t down_decode(const moe_ctx* c, int T, cudaStream_t s, bool prepare) {
  const ExpertArgs a = make_args(c, nullptr, T);
  const int units = max_active(c, T) * (a.d / 64);
  const int grid = units < 2 * c->sm_count ? units : 2 * c->sm_count;
  const size_t smem = (size_t)kTG * a.f * sizeof(float);
  const bool bf = c->cfg.weight_format == MOE_W_BF16;
  switch (a.f) {
#define DN_CASE(F)                                                                          \
  case F:                                                                                   \
    return bf ? launch_k(down_decode_kernel<F / 32, true>, grid, smem, s, a, prepare)                \
              : launch_k(down_decode_kernel<F / 32, false>, grid, smem, s, a, prepare);
    DN_CASE(128)
    DN_CASE(256)
    DN_CASE(512)
    DN_CASE(1024)
#undef DN_CASE
    default:
      return cudaErrorInvalidValue;
  }
}

cudaError_t launch_gateup_decode(const moe_ctx* c, const __nv_bfloat16* x, int T, cudaStream_t s) {
  return gateup_decode(c, x, T, s, false);
}

cudaError_t launch_down_decode(const moe_ctx* c, int T, cudaStream_t s) {
  return down_decode(c, T, s, false);
}

cudaError_t prepare_decode_kernels(const moe_ctx* c) {
  cudaError_t e = gateup_decode(c, nullptr, 1, nullptr, true);
  if (e != cudaSuccess) return e;
  return down_decode(c, 1, nullptr, true);
}

// ---------------------------------------------------------------------------
// combine: y[t] = sum_j w[t,j] yexp[pos(t,j)] + sum_s yexp[T*k + s*T + t] (+ x[t])
// Fixed summation order (j ascending, then shared), so results are deterministic.
// Below 1024 tokens CTA (t, q) takes the q-th of 4 column ranges of token t,
// one 16-byte column group per thread, so a 64-token batch spreads over 256
// CTAs and every thread's loads are in flight together (64 tokens: 114.3 ->
// 113.1 us a step).  Larger batches have CTAs enough with one per token (the
// split made 32768 tokens 1% slower).
// ---------------------------------------------------------------------------
namespace {
template <bool SPLIT>
__global__ void __launch_bounds__(256) combine_kernel(Routing r, const float* __restrict__ yexp,
                                                      const __nv_bfloat16* __restrict__ x,
                                                      __nv_bfloat16* __restrict__ y, int T, int d,
                                                      int k, int S, int residual) {
  const int t = blockIdx.x;
  int pos[8];
  float w[8];
  for (int j = 0; j < k; ++j) {
    pos[j] = r.slot_pos[t * k + j];
    w[j] = r.w[t * k + j];
  }
  int c0 = threadIdx.x, c1 = d / 4;
  if (SPLIT) {
    const int per = (c1 + gridDim.y - 1) / gridDim.y;
    c0 = blockIdx.y * per + threadIdx.x;
    c1 = min(c1, ((int)blockIdx.y + 1) * per);
  }
  for (int c = c0; c < c1; c += blockDim.x) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < k; ++j) {
      const float4 v = reinterpret_cast<const float4*>(yexp + (size_t)pos[j] * d)[c];
      acc.x = fmaf(w[j], v.x, acc.x);
      acc.y = fmaf(w[j], v.y, acc.y);
      acc.z = fmaf(w[j], v.z, acc.z);
      acc.w = fmaf(w[j], v.w, acc.w);
    }
    for (int s = 0; s < S; ++s) {
      const float4 v = reinterpret_cast<const float4*>(yexp + (size_t)(T * k + s * T + t) * d)[c];
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    if (residual) {
      const uint2 xv = reinterpret_cast<const uint2*>(x + (size_t)t * d)[c];
      acc.x += __uint_as_float(xv.x << 16);
      acc.y += __uint_as_float(xv.x & 0xFFFF0000u);
      acc.z += __uint_as_float(xv.y << 16);
      acc.w += __uint_as_float(xv.y & 0xFFFF0000u);
    }
    __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
    __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
    uint2 out;
    out.x = *reinterpret_cast<uint32_t*>(&lo);
    out.y = *reinterpret_cast<uint32_t*>(&hi);
    reinterpret_cast<uint2*>(y + (size_t)t * d)[c] = out;
  }
}
}  // namespace

cudaError_t launch_combine(const moe_ctx* c, const __nv_bfloat16* x, int T, __nv_bfloat16* y,
                           int residual, cudaStream_t s) {
  if (T < 1024)
    combine_kernel<true><<<dim3(T, 4), 128, 0, s>>>(c->r, c->yexp, x, y, T, c->cfg.d_model, c->cfg.top_k,
                                                    c->cfg.n_shared, residual);
  else
    combine_kernel<false><<<T, 256, 0, s>>>(c->r, c->yexp, x, y, T, c->cfg.d_model, c->cfg.top_k,
                                            c->cfg.n_shared, residual);
  return cudaGetLastError();
}

}  // namespace nvmoe
