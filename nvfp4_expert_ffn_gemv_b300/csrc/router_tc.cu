// Router logits of long batches (prefill) on the 5th-generation tensor cores.
//
// logits[t, e] = sum_k x[t, k] W_r[k, e] is a dense [T x d] x [d x E]
// contraction once T is in the thousands (4096 x 2048 x 256: 2.1e9 FMAs, about
// 60 us of fp32 FMA on every SM).  It runs here as tcgen05.mma kind::f16 with
// BF16 operands and FP32 accumulation, at the fp32 precision of the router:
//   - x is bf16 already, so the A operand is the input itself (loaded by TMA);
//   - W_r (fp32) is split once at set-up into three bf16 matrices
//     W1 = bf16(W), W2 = bf16(W - W1), W3 = bf16(W - W1 - W2), whose sum is W
//     exactly (each step keeps the next 8 significant bits, and each
//     difference is exact in fp32);
//   - every product x * Wi is exact in fp32 and the tensor core sums the
//     three splits into one fp32 accumulator, so the logits differ from an
//     fp32 CUDA-core dot product only in the order of the fp32 additions.
// Each CTA takes one 128-token block and one of nkc K chunks and writes its
// fp32 partial logits; the router's top-k kernel adds the nkc partials in a
// fixed order (and the bias) and selects the experts.
//
// CTA of 192 threads: warp 0 TMA producer (4-stage ring of {x tile 128 x 64,
// one W split 256 x 64}, both 128-byte swizzled), warp 1 TMEM owner and MMA
// issuer (4 MMAs of K = 16 per stage), warps 2-5 epilogue (TMEM lanes = token
// rows, 32 columns per tcgen05.ld).  All waits are bounded.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "internal.h"
#include "sm100.cuh"

namespace nvmoe {

namespace {

using namespace sm100;

constexpr int kRM = 128;            // tokens per CTA (MMA M)
constexpr int kRK = 64;             // bf16 elements of K per stage (128-byte rows)
constexpr int kRStages = 4;
constexpr int kRThreads = 192;
constexpr int kRSplits = 3;
constexpr int kRA = kRM * 128;      // 16 KB
constexpr int kRBMax = 256 * 128;   // 32 KB (E padded to at most 256 rows)
constexpr int kRSmem = kRStages * (kRA + kRBMax) + 1024;

struct RouterTcArgs {
  float* part;      // [nkc][T][E]
  int T, E, Ep, kc_len;
  int* status;
  int dbg;          // debug flags (MOE_DEBUG_FORCE_TIMEOUT)
};

__global__ void __launch_bounds__(kRThreads, 1)
    router_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                     RouterTcArgs g) {
  extern __shared__ uint8_t rsmem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(rsmem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;                           // [kRStages][kRA]
  uint8_t* sB = smem + kRStages * kRA;          // [kRStages][kRBMax]
  __shared__ __align__(8) uint64_t full_bar[kRStages], empty_bar[kRStages], done_bar;
  __shared__ uint32_t tmem_base_s;
  __shared__ volatile int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.x * kRM;
  const int kc = blockIdx.y;
  const int k0 = kc * g.kc_len;
  const int nkb = g.kc_len / kRK;
  const int nstages = nkb * kRSplits;
  const uint32_t tcols = g.Ep <= 32 ? 32u : (g.Ep <= 64 ? 64u : (g.Ep <= 128 ? 128u : 256u));

  if (threadIdx.x == 0) {
    for (int s = 0; s < kRStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    mbar_init(&done_bar, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmX);
    prefetch_tmap(&tmW);
  }
  if (warp == 1) tmem_alloc(&tmem_base_s, tcols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;

  auto bounded_wait = [&](uint64_t* bar, uint32_t parity) -> bool {
    if (abort_flag) return false;
    if (wait_parity(bar, parity)) return true;
    abort_flag = 1;
    latch_status(g.status, MOE_ERR_TIMEOUT);
    return false;
  };

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      for (int i = 0; i < nstages; ++i) {
        const int kb = i / kRSplits, sp = i % kRSplits;
        if (!bounded_wait(&empty_bar[stage], phase ^ 1)) break;
        mbar_arrive_expect_tx(&full_bar[stage], (uint32_t)(kRA + g.Ep * 128));
        tma_load_2d(sA + stage * kRA, &tmX, k0 + kb * kRK, t0, &full_bar[stage]);
        tma_load_2d(sB + stage * kRBMax, &tmW, k0 + kb * kRK, sp * g.Ep, &full_bar[stage]);
        if (++stage == kRStages) { stage = 0; phase ^= 1; }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      const uint32_t idesc = idesc_bf16_f32(kRM, g.Ep);
      bool ok = true;
      for (int i = 0; i < nstages; ++i) {
        if (!bounded_wait(&full_bar[stage], phase)) { ok = false; break; }
        tc_fence_after();
        const uint64_t adesc = desc_kmajor_sw128(smem_u32(sA + stage * kRA));
        const uint64_t bdesc = desc_kmajor_sw128(smem_u32(sB + stage * kRBMax));
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_bf16(tmem, adesc + (uint64_t)(kk * 2), bdesc + (uint64_t)(kk * 2), idesc, i > 0 || kk > 0);
        tc_commit(&empty_bar[stage]);
        if (++stage == kRStages) { stage = 0; phase ^= 1; }
      }
      (void)ok;
      tc_commit(&done_bar);
    }
  } else {
    const int q = warp & 3;
    const int m = q * 32 + lane;
    const int t = t0 + m;
    const bool ok = __all_sync(0xffffffffu, bounded_wait(&done_bar, 0));   // warp-uniform for tcgen05.ld
    tc_fence_after();
    float* dst = g.part + ((size_t)kc * g.T + t) * g.E;
    for (int c0 = 0; c0 < g.Ep; c0 += 32) {
      uint32_t v[32];
      if (ok) tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + c0, v);
      if (ok && t < g.T) {
        if (c0 + 32 <= g.E && (g.E & 3) == 0) {
#pragma unroll
          for (int j = 0; j < 32; j += 4)
            *reinterpret_cast<float4*>(dst + c0 + j) = make_float4(__uint_as_float(v[j]), __uint_as_float(v[j + 1]),
                                                                   __uint_as_float(v[j + 2]),
                                                                   __uint_as_float(v[j + 3]));
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (c0 + j < g.E) dst[c0 + j] = __uint_as_float(v[j]);
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
    tmem_dealloc(tmem, tcols);
  }
}

// W_r [d][E] fp32 -> three bf16 splits [3][Ep][d] (expert rows, K contiguous),
// rows E..Ep-1 zero.  One thread per (e, k).
__global__ void split_router_kernel(const float* __restrict__ wr, int d, int E, int Ep,
                                    __nv_bfloat16* __restrict__ out) {
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (size_t)Ep * d) return;
  const int e = (int)(i / d), k = (int)(i % d);
  const float w = e < E ? wr[(size_t)k * E + e] : 0.f;
  const __nv_bfloat16 w1 = __float2bfloat16_rn(w);
  const float r1 = w - __bfloat162float(w1);
  const __nv_bfloat16 w2 = __float2bfloat16_rn(r1);
  const float r2 = r1 - __bfloat162float(w2);
  const __nv_bfloat16 w3 = __float2bfloat16_rn(r2);
  const size_t plane = (size_t)Ep * d;
  out[i] = w1;
  out[plane + i] = w2;
  out[2 * plane + i] = w3;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_tiled() {
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

// bf16 matrix [rows][cols] row-major, boxes of box_rows x 64 elements, 128-byte swizzle
bool make_tmap_bf16(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  auto fn = encode_tiled();
  if (!fn) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {kRK, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

int router_tc_padded_experts(const moe_config& c) { return (c.n_experts + 15) / 16 * 16; }

bool router_tc_supported(const moe_config& c) {
  return c.n_experts <= 256 && c.d_model % (kRTcChunks * kRK) == 0;
}

cudaError_t router_tc_prepare(moe_ctx* c) {
  const int d = c->cfg.d_model, E = c->cfg.n_experts, Ep = router_tc_padded_experts(c->cfg);
  const size_t n = (size_t)Ep * d;
  split_router_kernel<<<(unsigned)((n + 255) / 256), 256>>>(c->router, d, E, Ep, c->rt_wsplit);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (!make_tmap_bf16(&c->rt_tmw, c->rt_wsplit, (uint64_t)kRSplits * Ep, d, (uint32_t)Ep))
    return cudaErrorInvalidValue;
  return cudaFuncSetAttribute(router_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kRSmem);
}

cudaError_t launch_router_tc(const moe_ctx* c, const __nv_bfloat16* x, int T, cudaStream_t s) {
  const int d = c->cfg.d_model, E = c->cfg.n_experts, Ep = router_tc_padded_experts(c->cfg);
  CUtensorMap tmx;
  if (!make_tmap_bf16(&tmx, x, (uint64_t)T, d, kRM)) return cudaErrorInvalidValue;
  RouterTcArgs g;
  g.part = c->rt_part;
  g.T = T;
  g.E = E;
  g.Ep = Ep;
  g.kc_len = d / kRTcChunks;
  g.status = c->status;
  g.dbg = c->debug_flags;
  router_tc_kernel<<<dim3((T + kRM - 1) / kRM, kRTcChunks), kRThreads, kRSmem, s>>>(tmx, c->rt_tmw, g);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_router_topk(c->rt_part, c->bias, c->has_bias, T, E, c->cfg.top_k, kRTcChunks, c->r.idx, c->r.w,
                            c->status, debug_logits(c), s);
}

}  // namespace nvmoe
