// Router: fp32 logits x W_r (+ bias), top-k selection and renormalised softmax.
//
// Flint pages ("Recursive Flint 40B-A2.5B：まず速さを第一に考えて作られたコーディング
// モデル", section "このアーキテクチャはメモリ帯域幅に関する主張である"): 256 routed
// experts, 6 chosen per token.  The scoring function is not on the pages; the
// reading used is a softmax router whose k best logits are kept and
// renormalised, ties broken towards the lower expert index.
//
// Two kernels:
//   router_partial: split-K GEMV/GEMM.  Block (kc, tile) multiplies a tile of 8
//     tokens by the K-chunk kc of W_r [d][E]; thread e owns expert e, so every
//     W_r row is read as one coalesced 1 KB line.  Partial sums go to scratch.
//   router_topk: one warp per token sums the partials in a fixed order
//     (deterministic), adds the bias, runs k rounds of warp argmax over the
//     (up to) 256 logits (8 per lane) and writes idx and the softmax weights.
#include <atomic>

#include "internal.h"

namespace nvmoe {

namespace {

constexpr int kTT = 8;      // tokens per router tile
constexpr int kSlab = 256;  // rows of W_r staged per x slab

__global__ void __launch_bounds__(256) router_partial_kernel(
    const __nv_bfloat16* __restrict__ x, const float* __restrict__ wr, float* __restrict__ part,
    int T, int d, int E, int kc_len) {
  __shared__ float xs[kTT][kSlab];
  const int kc = blockIdx.x;
  const int t0 = blockIdx.y * kTT;
  const int e = threadIdx.x;
  const int nt = min(kTT, T - t0);
  float acc[kTT];
#pragma unroll
  for (int t = 0; t < kTT; ++t) acc[t] = 0.f;
  const int kbeg = kc * kc_len;
  for (int k0 = kbeg; k0 < kbeg + kc_len; k0 += kSlab) {
    const int slab = min(kSlab, kbeg + kc_len - k0);
    __syncthreads();
    for (int i = threadIdx.x; i < kTT * slab; i += blockDim.x) {
      const int t = i / slab, kk = i % slab;
      xs[t][kk] = (t < nt) ? __bfloat162float(x[(size_t)(t0 + t) * d + k0 + kk]) : 0.f;
    }
    __syncthreads();
    if (e < E) {
      const float* wp = wr + (size_t)k0 * E + e;
#pragma unroll 8
      for (int kk = 0; kk < slab; ++kk) {
        const float wv = __ldg(wp + (size_t)kk * E);
#pragma unroll
        for (int t = 0; t < kTT; ++t) acc[t] = fmaf(xs[t][kk], wv, acc[t]);
      }
    }
  }
  if (e < E) {
    for (int t = 0; t < nt; ++t) part[((size_t)kc * T + t0 + t) * E + e] = acc[t];
  }
}

// a beats b: larger value first, NaN counts as -inf, ties to the lower index
__device__ __forceinline__ bool beats(float va, int ia, float vb, int ib) {
  const float a = (va != va) ? -INFINITY : va;
  const float b = (vb != vb) ? -INFINITY : vb;
  return a > b || (a == b && ia < ib);
}

__global__ void __launch_bounds__(256) router_topk_kernel(
    const float* __restrict__ part, const float* __restrict__ bias, int has_bias, int T, int E,
    int K, int nkc, int32_t* __restrict__ idx, float* __restrict__ wout, int* status) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + warp;
  if (t >= T) return;
  float v[8];
  bool taken[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = lane + 32 * i;
    taken[i] = e >= E;
    v[i] = 0.f;
  }
  // partial sums in a fixed order; 8 independent loads in flight per step
  for (int kc0 = 0; kc0 < nkc; kc0 += 8) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane + 32 * i;
      if (e < E) {
        float pv[8];
#pragma unroll
        for (int q = 0; q < 8; ++q)
          pv[q] = (kc0 + q < nkc) ? __ldg(part + ((size_t)(kc0 + q) * T + t) * E + e) : 0.f;
#pragma unroll
        for (int q = 0; q < 8; ++q) v[i] += pv[q];
      }
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = lane + 32 * i;
    if (e < E && has_bias) v[i] += bias[e];
  }
  float sel_v[8];
  int sel_e[8];
  for (int j = 0; j < K; ++j) {
    float bv = 0.f;
    int be = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane + 32 * i;
      if (!taken[i] && (be == 0x7fffffff || beats(v[i], e, bv, be))) { bv = v[i]; be = e; }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oe = __shfl_xor_sync(0xffffffffu, be, o);
      if (oe != 0x7fffffff && (be == 0x7fffffff || beats(ov, oe, bv, be))) { bv = ov; be = oe; }
    }
    sel_v[j] = bv;
    sel_e[j] = be;
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (lane + 32 * i == be) taken[i] = true;
  }
  if (lane == 0) {
    const float m = sel_v[0];
    float z[8], sum = 0.f;
    for (int j = 0; j < K; ++j) { z[j] = __expf(sel_v[j] - m); sum += z[j]; }
    for (int j = 0; j < K; ++j) {
      int e = sel_e[j];
      if (e < 0 || e >= E) { latch_status(status, MOE_ERR_DEVICE_CHECK); e = 0; }
      idx[(size_t)t * K + j] = e;
      wout[(size_t)t * K + j] = z[j] / sum;
    }
  }
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

int router_chunks(int d, int T) {
  const int tiles = (T + kTT - 1) / kTT;
  int kc = 512 / (tiles > 0 ? tiles : 1);
  if (kc > 64) kc = 64;
  if (kc > d / 32) kc = d / 32;
  if (kc < 1) kc = 1;
  int p = 1;  // power of two that divides d
  while (p * 2 <= kc) p *= 2;
  return p;
}

cudaError_t launch_router(const moe_ctx* c, const __nv_bfloat16* x, int T, cudaStream_t s) {
  const int d = c->cfg.d_model, E = c->cfg.n_experts;
  const int nkc = router_chunks(d, T);
  dim3 g1(nkc, (T + kTT - 1) / kTT);
  router_partial_kernel<<<g1, 256, 0, s>>>(x, c->router, c->router_partial, T, d, E, d / nkc);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  router_topk_kernel<<<(T + 7) / 8, 256, 0, s>>>(c->router_partial, c->bias, c->has_bias, T, E,
                                                 c->cfg.top_k, nkc, c->r.idx, c->r.w, c->status);
  return cudaGetLastError();
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
    if (dev < kMaxCachedDevices) g_static_partials_addr[dev].store(part, std::memory_order_release);
  }
  const int nkc = router_chunks(d, T);
  router_partial_kernel<<<dim3(nkc, (T + kTT - 1) / kTT), 256, 0, s>>>(x, wr, part, T, d, E, d / nkc);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  router_topk_kernel<<<(T + 7) / 8, 256, 0, s>>>(part, bias, bias != nullptr, T, E, K, nkc, idx, w,
                                                 nullptr);
  return cudaGetLastError();
}

}  // namespace nvmoe
