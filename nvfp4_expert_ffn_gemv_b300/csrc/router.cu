// Router: fp32 logits x W_r (+ bias), top-k selection and renormalised softmax.
//
// Flint pages ("Recursive Flint 40B-A2.5B：まず速さを第一に考えて作られたコーディング
// モデル", section "このアーキテクチャはメモリ帯域幅に関する主張である"): 256 routed
// experts, 6 chosen per token.  The scoring function is not on the pages; the
// reading used is a softmax router whose k best logits are kept and
// renormalised, ties broken towards the lower expert index.
//
// Two kernels:
//   router_partial: split-K GEMV/GEMM.  Block (kc, tile) multiplies a tile of TT
//     tokens (8, or 32 from 256 tokens up) by the K-chunk kc of W_r [d][E];
//     thread e owns expert e, so every W_r row is read as one coalesced 1 KB
//     line and feeds TT FMAs; a thread's W_r loads of a chunk are all in
//     flight together.  Partial sums go to scratch.
//   router_topk: one CTA per token; thread e sums its nkc partials in a fixed
//     order (deterministic) and adds the bias, then one warp runs k rounds of
//     argmax over the (up to) 256 logits (8 per lane) and writes idx and the
//     softmax weights.
#include <atomic>

#include "internal.h"

namespace nvmoe {

namespace {

constexpr int kSlab = 256;  // rows of W_r staged per x slab

// Transposed x slab xs[kk][t] (row stride TT + 4) for k0 <= k < k0 + slab:
// thread i loads the TT / NPART values t = (i / kSlab) * TT / NPART + .. of
// row kk = i % kSlab at once, so all of a thread's L2 loads are in flight
// together (blockDim == kSlab * NPART).
template <int TT, int NPART>
__device__ __forceinline__ void stage_x_slab(const __nv_bfloat16* __restrict__ x, int d, int t0, int nt, int k0,
                                             int slab, float* xs) {
  constexpr int TP = TT / NPART;
  const int kk = threadIdx.x % kSlab;
  const int tb = (threadIdx.x / kSlab) * TP;
  float v[TP];
#pragma unroll
  for (int t = 0; t < TP; ++t)
    v[t] = (tb + t < nt && kk < slab) ? __bfloat162float(x[(size_t)(t0 + tb + t) * d + k0 + kk]) : 0.f;
  if (kk < slab) {
#pragma unroll
    for (int q = 0; q < TP / 4; ++q)
      *reinterpret_cast<float4*>(xs + kk * (TT + 4) + tb + 4 * q) = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2],
                                                                               v[4 * q + 3]);
  }
}

// A thread requests WPRE rows of its W_r column before it uses any of them
// (the first batch even before the x slab is staged, so the two latencies
// overlap): a K chunk of up to WPRE rows costs one memory round trip.
template <int TT>
__global__ void __launch_bounds__(256) router_partial_kernel(
    const __nv_bfloat16* __restrict__ x, const float* __restrict__ wr, float* __restrict__ part,
    int T, int d, int E, int kc_len) {
  constexpr int XS = TT + 4;  // padded row of the transposed x slab
  constexpr int WPRE = TT <= 8 ? 64 : 16;
  __shared__ __align__(16) float xs[kSlab][XS];
  const int kc = blockIdx.x;
  const int t0 = blockIdx.y * TT;
  const int e = threadIdx.x;
  const int nt = min(TT, T - t0);
  float acc[TT];
#pragma unroll
  for (int t = 0; t < TT; ++t) acc[t] = 0.f;
  const int kbeg = kc * kc_len;
  for (int k0 = kbeg; k0 < kbeg + kc_len; k0 += kSlab) {
    const int slab = min(kSlab, kbeg + kc_len - k0);
    const float* wp = wr + (size_t)k0 * E + (e < E ? e : 0);
    float wv[WPRE];
#pragma unroll
    for (int i = 0; i < WPRE; ++i) wv[i] = (e < E && i < slab) ? __ldg(wp + (size_t)i * E) : 0.f;
    __syncthreads();
    stage_x_slab<TT, 1>(x, d, t0, nt, k0, slab, &xs[0][0]);
    __syncthreads();
    if (e < E) {
      for (int kb = 0; kb < slab; kb += WPRE) {
        if (kb > 0) {
#pragma unroll
          for (int i = 0; i < WPRE; ++i) wv[i] = kb + i < slab ? __ldg(wp + (size_t)(kb + i) * E) : 0.f;
        }
#pragma unroll
        for (int i = 0; i < WPRE; ++i) {
          if (kb + i < slab) {
            const float4* xv = reinterpret_cast<const float4*>(&xs[kb + i][0]);
#pragma unroll
            for (int q = 0; q < TT / 4; ++q) {
              const float4 v = xv[q];
              acc[4 * q + 0] = fmaf(v.x, wv[i], acc[4 * q + 0]);
              acc[4 * q + 1] = fmaf(v.y, wv[i], acc[4 * q + 1]);
              acc[4 * q + 2] = fmaf(v.z, wv[i], acc[4 * q + 2]);
              acc[4 * q + 3] = fmaf(v.w, wv[i], acc[4 * q + 3]);
            }
          }
        }
      }
    }
  }
  if (e < E) {
#pragma unroll
    for (int t = 0; t < TT; ++t)
      if (t < nt) part[((size_t)kc * T + t0 + t) * E + e] = acc[t];
  }
}

// Same partial sums as router_partial_kernel (same k order, so bit-identical),
// for 32-token tiles: W_r is streamed through shared memory in 32-row
// sub-slabs by a 4-deep cp.async ring, and each of 512 threads accumulates 4
// experts x 4 tokens, so one k step costs it two 16-byte shared loads for 16
// FMAs, with 16 warps per SM to hide their latency.
constexpr int kWRows = 32;
constexpr int kWStages = 4;
constexpr int kStagedTT = 32;
constexpr int kStagedThreads = 512;

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const uint32_t sa = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" :: "r"(sa), "l"(gmem) : "memory");
}

constexpr size_t staged_smem_bytes() {
  return (size_t)kSlab * (kStagedTT + 4) * 4 + (size_t)kWStages * kWRows * 256 * 4;
}

__global__ void __launch_bounds__(kStagedThreads, 1) router_partial_staged_kernel(
    const __nv_bfloat16* __restrict__ x, const float* __restrict__ wr, float* __restrict__ part,
    int T, int d, int E, int kc_len) {
  constexpr int TT = kStagedTT;
  constexpr int XS = TT + 4;
  extern __shared__ __align__(16) float rsm[];
  float* xs = rsm;                      // [kSlab][XS]
  float* ws = rsm + kSlab * XS;         // [kWStages][kWRows][256]
  const int kc = blockIdx.x;
  const int t0 = blockIdx.y * TT;
  const int eq = threadIdx.x & 63;      // experts 4eq .. 4eq+3
  const int tq = threadIdx.x >> 6;      // tokens 4tq .. 4tq+3 of the tile
  const int nt = min(TT, T - t0);
  const int kbeg = kc * kc_len;
  const int nsub = kc_len / kWRows;
  const int e4 = E / 4;
  auto issue = [&](int sub) {
    if (sub < nsub) {
      const float* src = wr + (size_t)(kbeg + sub * kWRows) * E;
      float* dst = ws + (sub % kWStages) * kWRows * 256;
      for (int i = threadIdx.x; i < kWRows * e4; i += blockDim.x) {
        const int r = i / e4, q = i % e4;
        cp_async16(dst + r * 256 + 4 * q, src + (size_t)r * E + 4 * q);
      }
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  for (int s = 0; s < kWStages - 1; ++s) issue(s);
  for (int sub = 0; sub < nsub; ++sub) {
    __syncthreads();  // compute(sub - 1) is done: its W stage and (on a slab edge) xs are free
    const int kin = (sub * kWRows) % kSlab;
    if (kin == 0) {
      const int k0 = kbeg + sub * kWRows;
      stage_x_slab<TT, kStagedThreads / kSlab>(x, d, t0, nt, k0, min(kSlab, kbeg + kc_len - k0), xs);
    }
    issue(sub + kWStages - 1);
    asm volatile("cp.async.wait_group %0;" :: "n"(kWStages - 1) : "memory");
    __syncthreads();
    if (4 * eq < E) {
      const float* wrow = ws + (sub % kWStages) * kWRows * 256 + 4 * eq;
      const float* xrow = xs + kin * XS + 4 * tq;
#pragma unroll 8
      for (int r = 0; r < kWRows; ++r) {
        const float4 w = *reinterpret_cast<const float4*>(wrow + r * 256);
        const float4 xa = *reinterpret_cast<const float4*>(xrow + r * XS);
        const float wv[4] = {w.x, w.y, w.z, w.w};
        const float xv[4] = {xa.x, xa.y, xa.z, xa.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(xv[j], wv[i], acc[i][j]);
      }
    }
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");
  if (4 * eq < E) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int t = 4 * tq + j;
      if (t < nt)
        *reinterpret_cast<float4*>(part + ((size_t)kc * T + t0 + t) * E + 4 * eq) =
            make_float4(acc[0][j], acc[1][j], acc[2][j], acc[3][j]);
    }
  }
}

// k rounds of warp argmax over the (up to) 256 logits v[i] of expert lane + 32 i
// (larger value first, equal values -- +0 and -0 included -- to the lower
// expert, NaN below every number); logits_out (debug, or NULL) receives the
// values ranked;
// lanes j < K write idx and the renormalised softmax weight of token t's
// choice j.  Each value maps to an order-preserving unsigned key, so a round
// is a lane-local 8-way argmax, one warp max of the keys and one warp min of
// the expert index among the lanes that hold the maximum.
__device__ __forceinline__ void warp_select(const float (&v)[8], int E, int K, int t, int32_t* __restrict__ idx,
                                            float* __restrict__ wout, int* status, float* __restrict__ logits_out) {
  const int lane = threadIdx.x & 31;
  if (logits_out) {
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (lane + 32 * i < E) logits_out[(size_t)t * E + lane + 32 * i] = v[i];
  }
  uint32_t key[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    // -0 and +0 are equal logits: both get the key of +0
    const uint32_t u = __float_as_uint(v[i] == 0.f ? 0.f : v[i]);
    uint32_t kk = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    if (v[i] != v[i]) kk = 1u;
    key[i] = lane + 32 * i < E ? max(kk, 1u) : 0u;   // 0: no expert
  }
  float my_v = 0.f;
  uint32_t my_e = 0u;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    if (j < K) {
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
        if (i == bi) bv = v[i];
        if (lane + 32 * i == (int)win) key[i] = 0;
      }
      const float sv = __shfl_sync(0xffffffffu, bv, (int)(win & 31));
      if (lane == j) { my_v = sv; my_e = win; }
    }
  }
  // softmax over the chosen logits, one per lane (lane 0 holds the largest)
  const float m = __shfl_sync(0xffffffffu, my_v, 0);
  const float z = lane < K ? expf(my_v - m) : 0.f;
  float sum = z;
#pragma unroll
  for (int o = 4; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);   // K <= 8 lanes
  sum = __shfl_sync(0xffffffffu, sum, 0);
  if (lane < K) {
    int ee = (int)my_e;
    if (ee >= E) { latch_status(status, MOE_ERR_DEVICE_CHECK); ee = 0; }
    idx[(size_t)t * K + lane] = ee;
    wout[(size_t)t * K + lane] = z / sum;
  }
}

// Many K chunks: one CTA per token; thread e sums its nkc partials in order.
__global__ void __launch_bounds__(256) router_topk_kernel(
    const float* __restrict__ part, const float* __restrict__ bias, int has_bias, int T, int E,
    int K, int nkc, int32_t* __restrict__ idx, float* __restrict__ wout, int* status, float* logits_out) {
  __shared__ float lg[256];
  const int t = blockIdx.x;
  const int e = threadIdx.x;
  if (e < E) {
    // partial sums in a fixed order; 16 independent loads in flight per step
    float v = 0.f;
    for (int kc0 = 0; kc0 < nkc; kc0 += 16) {
      float pv[16];
#pragma unroll
      for (int q = 0; q < 16; ++q)
        pv[q] = (kc0 + q < nkc) ? __ldg(part + ((size_t)(kc0 + q) * T + t) * E + e) : 0.f;
#pragma unroll
      for (int q = 0; q < 16; ++q)
        if (kc0 + q < nkc) v += pv[q];
    }
    if (has_bias) v += bias[e];
    lg[e] = v;
  }
  __syncthreads();
  if (threadIdx.x >= 32) return;
  float v[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int ee = threadIdx.x + 32 * i;
    v[i] = ee < E ? lg[ee] : 0.f;
  }
  warp_select(v, E, K, t, idx, wout, status, logits_out);
}

// Few K chunks (nkc <= 4): one warp per token, the same sums in the same order.
__global__ void __launch_bounds__(256) router_topk_warp_kernel(
    const float* __restrict__ part, const float* __restrict__ bias, int has_bias, int T, int E,
    int K, int nkc, int32_t* __restrict__ idx, float* __restrict__ wout, int* status, float* logits_out) {
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  float p[4][8];
#pragma unroll
  for (int q = 0; q < 4; ++q)
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int ee = lane + 32 * i;
      p[q][i] = (ee < E && q < nkc) ? __ldg(part + ((size_t)q * T + t) * E + ee) : 0.f;
    }
  float v[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int ee = lane + 32 * i;
    float s = 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (q < nkc) s += p[q][i];
    if (ee < E && has_bias) s += bias[ee];
    v[i] = s;
  }
  warp_select(v, E, K, t, idx, wout, status, logits_out);
}

int router_tile(int T) { return T >= 256 ? 32 : 8; }

}  // namespace

cudaError_t launch_router_topk(const float* part, const float* bias, int has_bias, int T, int E, int K, int nkc,
                               int32_t* idx, float* w, int* status, float* logits_out, cudaStream_t s) {
  if (nkc <= 4)
    router_topk_warp_kernel<<<(T + 7) / 8, 256, 0, s>>>(part, bias, has_bias, T, E, K, nkc, idx, w, status,
                                                         logits_out);
  else
    router_topk_kernel<<<T, 256, 0, s>>>(part, bias, has_bias, T, E, K, nkc, idx, w, status, logits_out);
  return cudaGetLastError();
}

namespace {

cudaError_t launch_router_kernels(const __nv_bfloat16* x, int T, const float* wr, const float* bias,
                                  int has_bias, int d, int E, int K, float* part, int32_t* idx, float* w,
                                  int* status, float* logits_out, cudaStream_t s) {
  const int nkc = router_chunks(d, T);
  const int tt = router_tile(T);
  const dim3 g1(nkc, (T + tt - 1) / tt);
  const bool staged = E % 4 == 0 && (reinterpret_cast<uintptr_t>(wr) & 15u) == 0 && (d / nkc) % kWRows == 0;
  if (tt == 32 && staged)
    router_partial_staged_kernel<<<g1, kStagedThreads, staged_smem_bytes(), s>>>(x, wr, part, T, d, E, d / nkc);
  else if (tt == 32)
    router_partial_kernel<32><<<g1, 256, 0, s>>>(x, wr, part, T, d, E, d / nkc);
  else
    router_partial_kernel<8><<<g1, 256, 0, s>>>(x, wr, part, T, d, E, d / nkc);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  return launch_router_topk(part, bias, has_bias, T, E, K, nkc, idx, w, status, logits_out, s);
}

// Scratch of the allocation-free router entry point: the split-K partial
// logits [nkc][T][E] of one call.  Every element the top-k kernel reads is
// written by the partial kernel of the same call, so nothing here has to start
// at zero.  One copy per device: calls that overlap on the GPU race on it.
constexpr size_t kStaticPartials = size_t(1) << 20;  // fp32 elements, 4 MiB
static __device__ __align__(256) float g_static_partials[kStaticPartials];

constexpr int kMaxCachedDevices = 64;
std::atomic<float*> g_static_partials_addr[kMaxCachedDevices];

}  // namespace

cudaError_t prepare_router_kernels() {
  return cudaFuncSetAttribute(router_partial_staged_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)staged_smem_bytes());
}

// K chunks of the split-K router for T tokens: about 256 CTAs, at most 64
// chunks and at least 32 rows per chunk, a power of two that divides d, and
// never more than 4096 / T chunks (so the partials hold at most
// max(T, 4096) x E values).
int router_chunks(int d, int T) {
  const int tt = router_tile(T);
  const int tiles = (T + tt - 1) / tt;
  int kc = 256 / (tiles > 0 ? tiles : 1);
  if (kc > 64) kc = 64;
  if (kc > d / 32) kc = d / 32;
  if (T > 0 && kc > 4096 / T) kc = 4096 / T;
  if (kc < 1) kc = 1;
  int p = 1;
  while (p * 2 <= kc) p *= 2;
  return p;
}

cudaError_t launch_router(const moe_ctx* c, const __nv_bfloat16* x, int T, cudaStream_t s) {
  return launch_router_kernels(x, T, c->router, c->bias, c->has_bias, c->cfg.d_model, c->cfg.n_experts,
                               c->cfg.top_k, c->router_partial, c->r.idx, c->r.w, c->status, debug_logits(c), s);
}

size_t router_static_capacity() { return kStaticPartials; }

cudaError_t launch_router_static(const __nv_bfloat16* x, int T, const float* wr, const float* bias, int d,
                                 int E, int K, int32_t* idx, float* w, cudaStream_t s) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  float* part = dev < kMaxCachedDevices ? g_static_partials_addr[dev].load(std::memory_order_acquire)
                                        : nullptr;
  if (!part) {
    err = cudaGetSymbolAddress((void**)&part, g_static_partials);
    if (err != cudaSuccess) return err;
    if ((err = prepare_router_kernels()) != cudaSuccess) return err;
    if (dev < kMaxCachedDevices) g_static_partials_addr[dev].store(part, std::memory_order_release);
  }
  return launch_router_kernels(x, T, wr, bias, bias != nullptr, d, E, K, part, idx, w, nullptr, nullptr, s);
}

}  // namespace nvmoe
