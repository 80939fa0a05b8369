// C ABI of the NVFP4 MoE library: argument checks, device arena, weight
// repacking and the per-call kernel sequence.  See include/nvfp4_moe.h.
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <vector>

#include "internal.h"

using namespace nvmoe;

namespace {

bool is_pow2_in(int v, int lo, int hi) { return v >= lo && v <= hi && (v & (v - 1)) == 0; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Carver {
  size_t off = 0;
  template <typename T>
  T* take(uint8_t* base, size_t count) {
    off = (off + 255) & ~size_t(255);
    T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
    off += count * sizeof(T);
    return p;
  }
};

moe_status check_matrix_nvfp4(const moe_matrix& m) {
  return (m.codes && m.scales && m.tensor_scale) ? MOE_OK : MOE_ERR_INVALID_ARG;
}

size_t router_partial_floats(const moe_config& c) {
  size_t best = 0;
  for (int T = 1; T <= c.max_tokens; ++T) {
    const size_t v = (size_t)router_chunks(c.d_model, T) * T;
    best = std::max(best, v);
  }
  return std::max(best, (size_t)c.max_tokens) * c.n_experts;
}

// Lay out (base == nullptr: only measure) every buffer of the context.
size_t carve(moe_ctx* x, uint8_t* base) {
  const moe_config& c = x->cfg;
  const size_t n = x->n_all, d = c.d_model, f = c.d_ff;
  const size_t T = c.max_tokens, k = c.top_k, S = c.n_shared, E = c.n_experts;
  const size_t P = T * (k + S);
  Carver cv;
  if (c.weight_format == MOE_W_NVFP4) {
    x->gu_codes = cv.take<uint8_t>(base, n * 2 * f * d / 2);
    x->gu_scales = cv.take<uint8_t>(base, n * 2 * f * d / 16);
    x->dn_codes = cv.take<uint8_t>(base, n * d * f / 2);
    x->dn_scales = cv.take<uint8_t>(base, n * d * f / 16);
  } else {
    x->gu_bf16 = cv.take<__nv_bfloat16>(base, n * 2 * f * d);
    x->dn_bf16 = cv.take<__nv_bfloat16>(base, n * d * f);
  }
  x->tsc = cv.take<float>(base, n * 3);
  x->router = cv.take<float>(base, d * E);
  x->bias = cv.take<float>(base, E);
  x->router_partial = cv.take<float>(base, router_partial_floats(c));
  x->r.idx = cv.take<int32_t>(base, T * k);
  x->r.w = cv.take<float>(base, T * k);
  x->r.counts = cv.take<int32_t>(base, E);
  x->r.offsets = cv.take<int32_t>(base, E + 1);
  x->r.slot_pos = cv.take<int32_t>(base, T * k);
  x->r.pos_tok = cv.take<int32_t>(base, P);
  x->r.pos_w = cv.take<float>(base, P);
  x->r.act_e = cv.take<int32_t>(base, E + S);
  x->r.act_pos = cv.take<int32_t>(base, E + S);
  x->r.act_n = cv.take<int32_t>(base, E + S);
  x->r.n_active = cv.take<int32_t>(base, 1);
  x->r.act_ppos = cv.take<int32_t>(base, E + S + 1);
  x->r.blk_a = cv.take<int32_t>(base, (T * (k + S) + 127) / 128 + E + S);
  x->r.chunk_cnt = cv.take<int32_t>(base, ((T + 31) / 32) * E);
  x->r.group_cnt = cv.take<int32_t>(base, ((T + 255) / 256) * E);
  x->r.rank = cv.take<int32_t>(base, T * k);
  x->dbg_logits = cv.take<float>(base, T * E);
  x->h = cv.take<float>(base, P * f);
  x->yexp = cv.take<float>(base, P * d);
  if (x->pf_enabled && prefill_accumulates(c, (int)T)) x->yacc = cv.take<float>(base, T * d);
  else if (x->pf_enabled && prefill_accumulates(c, 1))
    x->yacc = cv.take<float>(base, (size_t)(48u << 20) / (d * sizeof(float)) * d);
  x->status = cv.take<int>(base, 1);
  if (x->b1_enabled) {
    x->router_t = cv.take<float>(base, d * E);
    x->b1_rows = cv.take<uint8_t>(base, n * f * b1_row_bytes((int)d));
    x->logits = cv.take<float>(base, E);
  }
  x->max_positions = (int)P;
  if (x->rt_enabled) {
    x->rt_wsplit = cv.take<__nv_bfloat16>(base, (size_t)3 * router_tc_padded_experts(c) * d);
    x->rt_part = cv.take<float>(base, (size_t)kRTcChunks * T * E);
  }
  if (x->mma_enabled) {
    x->x16 = cv.take<uint8_t>(base, T * d * 2);
    x->xunshift = cv.take<float>(base, T);
  }
  if (x->pf_enabled) {
    const size_t rows = prefill_max_rows(c);
    x->pf_sfa_gu = cv.take<uint8_t>(base, n * 2 * f * d / 16);
    x->pf_sfa_dn = cv.take<uint8_t>(base, n * d * f / 16);
    x->pf_xq = cv.take<uint8_t>(base, rows * d / 2);
    // x scale atoms, followed by the same scales row-major (the quantiser's output)
    x->pf_xsf = cv.take<uint8_t>(base, 2 * rows * d / 16);
    x->pf_hq = cv.take<uint8_t>(base, rows * f / 2);
    x->pf_hsf = cv.take<uint8_t>(base, rows * f / 16);
  }
  return cv.off;
}

moe_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return MOE_OK;
  if (e == cudaErrorMemoryAllocation) return MOE_ERR_OOM;
  return MOE_ERR_CUDA;
}

#define CK(call)                                         \
  do {                                                   \
    cudaError_t e_ = (call);                             \
    if (e_ != cudaSuccess) return cuda_status(e_);       \
  } while (0)

// Copy one canonical gate or up stack into the tile-interleaved gate/up layout.
cudaError_t copy_gu_rows(uint8_t* dst_base, const void* src, size_t row_bytes, int f, int n_src,
                         int expert0, int upper_half) {
  for (int t = 0; t < f / 64; ++t) {
    uint8_t* dst = dst_base + ((size_t)expert0 * 2 * f + (size_t)t * 128 + upper_half * 64) * row_bytes;
    const uint8_t* s = static_cast<const uint8_t*>(src) + (size_t)t * 64 * row_bytes;
    cudaError_t e = cudaMemcpy2D(dst, 2 * (size_t)f * row_bytes, s, (size_t)f * row_bytes,
                                 64 * row_bytes, n_src, cudaMemcpyDefault);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

void ensure_device(int dev) {
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess || cur != dev) cudaSetDevice(dev);
}

}  // namespace

namespace nvmoe {

// Test hook (moe_debug_fail_alloc): the n-th device allocation from now on fails.
static std::atomic<int> g_fail_alloc_countdown{0};

cudaError_t device_alloc(void** p, size_t bytes) {
  int n = g_fail_alloc_countdown.load();
  while (n > 0 && !g_fail_alloc_countdown.compare_exchange_weak(n, n - 1)) {
  }
  if (n == 1) return cudaErrorMemoryAllocation;   // this call was the n-th: fail without allocating
  return cudaMalloc(p, bytes);
}

}  // namespace nvmoe

extern "C" {

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported configuration";
    case MOE_ERR_OOM: return "device out of memory";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_TIMEOUT: return "device-side wait timed out";
    case MOE_ERR_DEVICE_CHECK: return "device-side consistency check failed";
  }
  return "unknown status";
}

moe_status moe_init(const moe_config* cfg, const moe_weights* wts, int device, moe_ctx** out) {
  if (!cfg || !wts || !out) return MOE_ERR_INVALID_ARG;
  *out = nullptr;
  const moe_config c = *cfg;
  if (c.d_model <= 0 || c.n_experts <= 0 || c.top_k <= 0 || c.d_ff <= 0 || c.max_tokens <= 0 ||
      c.n_shared < 0)
    return MOE_ERR_INVALID_ARG;
  if (c.weight_format != MOE_W_NVFP4 && c.weight_format != MOE_W_BF16) return MOE_ERR_INVALID_ARG;
  if (c.top_k > c.n_experts) return MOE_ERR_INVALID_ARG;
  if (!is_pow2_in(c.d_model, 256, 4096) || !is_pow2_in(c.d_ff, 128, 1024) || c.n_experts > 256 ||
      c.top_k > 8 || c.n_shared > 2 || c.max_tokens > 65536)
    return MOE_ERR_UNSUPPORTED;
  if (c.n_shared > 0 && c.d_ff_shared != c.d_ff) return MOE_ERR_UNSUPPORTED;
  if (!wts->router) return MOE_ERR_INVALID_ARG;
  const moe_matrix* mats[6] = {&wts->gate, &wts->up, &wts->down,
                               &wts->shared_gate, &wts->shared_up, &wts->shared_down};
  for (int i = 0; i < (c.n_shared > 0 ? 6 : 3); ++i) {
    if (c.weight_format == MOE_W_NVFP4) {
      if (check_matrix_nvfp4(*mats[i]) != MOE_OK) return MOE_ERR_INVALID_ARG;
    } else if (!mats[i]->bf16) {
      return MOE_ERR_INVALID_ARG;
    }
  }
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || device < 0 || device >= ndev)
    return MOE_ERR_INVALID_ARG;
  CK(cudaSetDevice(device));

  moe_ctx* x = new moe_ctx();
  x->cfg = c;
  x->device = device;
  x->n_all = c.n_experts + c.n_shared;
  cudaDeviceGetAttribute(&x->sm_count, cudaDevAttrMultiProcessorCount, device);
  if (b1_supported(c))
    x->b1_enabled = b1_plan(c, x->sm_count, 1, &x->b1_grid, &x->b1_rmax, &x->b1_nbmax, &x->b1_smem);
  x->pf_enabled = prefill_supported(c);
  x->mma_enabled = mma_decode_supported(c);
  x->rt_enabled = x->pf_enabled && router_tc_supported(c) && c.max_tokens >= kRTcMinTokens;
  x->arena_bytes = carve(x, nullptr);
  if (device_alloc(reinterpret_cast<void**>(&x->arena), x->arena_bytes) != cudaSuccess) {
    cudaGetLastError();
    delete x;
    return MOE_ERR_OOM;
  }
  carve(x, x->arena);

  auto fail = [&](cudaError_t e) {
    cudaFree(x->arena);
    delete x;
    return cuda_status(e);
  };
  const size_t d = c.d_model, f = c.d_ff, E = c.n_experts, S = c.n_shared;
  cudaError_t e = cudaSuccess;
  if (c.weight_format == MOE_W_NVFP4) {
    struct { const moe_matrix* m; int n; int e0; } sets[2] = {{&wts->gate, (int)E, 0},
                                                              {&wts->shared_gate, (int)S, (int)E}};
    for (int si = 0; si < 2 && e == cudaSuccess; ++si) {
      if (sets[si].n == 0) continue;
      const moe_matrix* g = sets[si].m;
      const moe_matrix* u = g + 1;
      const moe_matrix* dn = g + 2;
      const int n = sets[si].n, e0 = sets[si].e0;
      if (e == cudaSuccess) e = copy_gu_rows(x->gu_codes, g->codes, d / 2, (int)f, n, e0, 0);
      if (e == cudaSuccess) e = copy_gu_rows(x->gu_codes, u->codes, d / 2, (int)f, n, e0, 1);
      if (e == cudaSuccess) e = copy_gu_rows(x->gu_scales, g->scales, d / 16, (int)f, n, e0, 0);
      if (e == cudaSuccess) e = copy_gu_rows(x->gu_scales, u->scales, d / 16, (int)f, n, e0, 1);
      if (e == cudaSuccess)
        e = cudaMemcpy(x->dn_codes + (size_t)e0 * d * f / 2, dn->codes, (size_t)n * d * f / 2,
                       cudaMemcpyDefault);
      if (e == cudaSuccess)
        e = cudaMemcpy(x->dn_scales + (size_t)e0 * d * f / 16, dn->scales, (size_t)n * d * f / 16,
                       cudaMemcpyDefault);
    }
    std::vector<float> tsh(x->n_all * 3), tmp(std::max(E, S) + 1);
    for (int si = 0; si < 2 && e == cudaSuccess; ++si) {
      const moe_matrix* base = si == 0 ? &wts->gate : &wts->shared_gate;
      const int n = si == 0 ? (int)E : (int)S, e0 = si == 0 ? 0 : (int)E;
      for (int m = 0; m < 3 && n > 0 && e == cudaSuccess; ++m) {
        e = cudaMemcpy(tmp.data(), base[m].tensor_scale, sizeof(float) * n, cudaMemcpyDefault);
        for (int i = 0; i < n; ++i) tsh[(size_t)(e0 + i) * 3 + m] = tmp[i];
      }
    }
    if (e == cudaSuccess)
      e = cudaMemcpy(x->tsc, tsh.data(), sizeof(float) * tsh.size(), cudaMemcpyHostToDevice);
  } else {
    const size_t rb = d * sizeof(__nv_bfloat16);
    uint8_t* gu = reinterpret_cast<uint8_t*>(x->gu_bf16);
    if (e == cudaSuccess) e = copy_gu_rows(gu, wts->gate.bf16, rb, (int)f, (int)E, 0, 0);
    if (e == cudaSuccess) e = copy_gu_rows(gu, wts->up.bf16, rb, (int)f, (int)E, 0, 1);
    if (S > 0 && e == cudaSuccess) e = copy_gu_rows(gu, wts->shared_gate.bf16, rb, (int)f, (int)S, (int)E, 0);
    if (S > 0 && e == cudaSuccess) e = copy_gu_rows(gu, wts->shared_up.bf16, rb, (int)f, (int)S, (int)E, 1);
    if (e == cudaSuccess)
      e = cudaMemcpy(x->dn_bf16, wts->down.bf16, E * d * f * 2, cudaMemcpyDefault);
    if (S > 0 && e == cudaSuccess)
      e = cudaMemcpy(x->dn_bf16 + E * d * f, wts->shared_down.bf16, S * d * f * 2, cudaMemcpyDefault);
    std::vector<float> ones(x->n_all * 3, 1.0f);
    if (e == cudaSuccess)
      e = cudaMemcpy(x->tsc, ones.data(), sizeof(float) * ones.size(), cudaMemcpyHostToDevice);
  }
  if (e == cudaSuccess) e = cudaMemcpy(x->router, wts->router, d * E * sizeof(float), cudaMemcpyDefault);
  x->has_bias = wts->router_bias != nullptr;
  if (e == cudaSuccess) {
    e = x->has_bias ? cudaMemcpy(x->bias, wts->router_bias, E * sizeof(float), cudaMemcpyDefault)
                    : cudaMemset(x->bias, 0, E * sizeof(float));
  }
  if (e == cudaSuccess) e = cudaMemset(x->status, 0, sizeof(int));
  if (e == cudaSuccess) e = prepare_router_kernels();
  if (e == cudaSuccess) e = prepare_bucket_kernel();
  if (e == cudaSuccess) e = prepare_decode_kernels(x);
  if (e == cudaSuccess && x->mma_enabled) e = prepare_mma_decode(x);
  if (e == cudaSuccess && x->rt_enabled) e = router_tc_prepare(x);
  if (e == cudaSuccess && x->pf_enabled) {
    e = prefill_prepare(x);
    if (e == cudaSuccess) e = cudaMemset(x->pf_hq, 0, prefill_max_rows(c) * (f / 2));
    if (e == cudaSuccess) e = cudaMemset(x->pf_hsf, 0, prefill_max_rows(c) * (f / 16));
  }
  if (e == cudaSuccess && x->b1_enabled) {
    e = repack_b1_layouts(x);
    if (e == cudaSuccess) e = prepare_b1_kernels(x);
  }
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return fail(e);
  *out = x;
  return MOE_OK;
}

moe_status moe_destroy(moe_ctx* x) {
  if (!x) return MOE_OK;
  ensure_device(x->device);
  cudaError_t e = cudaFree(x->arena);
  delete x;
  return cuda_status(e);
}

// Remember what the last routing of the context was (for moe_debug_logits).
static void note_routing(moe_ctx* x, int T, int b1) {
  x->last_route_T = T;
  x->last_route_b1 = b1;
  x->last_route_kept = b1 || (x->debug_flags & MOE_DEBUG_KEEP_LOGITS) != 0;
}

static moe_status check_fwd(moe_ctx* x, const void* in, int T, const void* out) {
  if (!x) return MOE_ERR_INVALID_ARG;
  if (T < 0 || T > x->cfg.max_tokens) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!in || !aligned16(in))) return MOE_ERR_INVALID_ARG;
  if (T > 0 && out && !aligned16(out)) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

moe_status moe_route(moe_ctx* x, const void* x_bf16, int T, int32_t* idx, float* w, int32_t* counts,
                     cudaStream_t s) {
  moe_status st = check_fwd(x, x_bf16, T, nullptr);
  if (st != MOE_OK) return st;
  if (T == 0) return MOE_OK;
  ensure_device(x->device);
  const auto* xb = static_cast<const __nv_bfloat16*>(x_bf16);
  CK(launch_router(x, xb, T, s));
  CK(launch_bucket(x, T, s));
  note_routing(x, T, 0);
  const size_t tk = (size_t)T * x->cfg.top_k;
  if (idx) CK(cudaMemcpyAsync(idx, x->r.idx, tk * sizeof(int32_t), cudaMemcpyDeviceToDevice, s));
  if (w) CK(cudaMemcpyAsync(w, x->r.w, tk * sizeof(float), cudaMemcpyDeviceToDevice, s));
  if (counts)
    CK(cudaMemcpyAsync(counts, x->r.counts, x->cfg.n_experts * sizeof(int32_t),
                       cudaMemcpyDeviceToDevice, s));
  return MOE_OK;
}

// True when the GPU can dereference p: device, managed or registered / pinned host memory.
static bool device_reachable(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.type != cudaMemoryTypeUnregistered;
}

moe_status moe_route_noalloc(const void* x_bf16, int T, const float* router, const float* router_bias,
                             int d_model, int n_experts, int top_k, int32_t* idx, float* w, cudaStream_t s) {
  if (T < 0 || d_model < 256 || d_model > 4096 || d_model % 256 != 0 || n_experts < 1 || n_experts > 256 ||
      top_k < 1 || top_k > 8 || top_k > n_experts)
    return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x_bf16 || !router || !idx || !w) return MOE_ERR_INVALID_ARG;
  if (!device_reachable(x_bf16) || !device_reachable(router) || !device_reachable(idx) ||
      !device_reachable(w) || (router_bias && !device_reachable(router_bias)))
    return MOE_ERR_INVALID_ARG;
  if ((size_t)router_chunks(d_model, T) * T * n_experts > router_static_capacity()) return MOE_ERR_UNSUPPORTED;
  CK(launch_router_static(static_cast<const __nv_bfloat16*>(x_bf16), T, router, router_bias, d_model,
                          n_experts, top_k, idx, w, s));
  return MOE_OK;
}

moe_status moe_forward_decode(moe_ctx* x, const void* x_bf16, int T, void* y_bf16, int residual,
                              cudaStream_t s) {
  moe_status st = check_fwd(x, x_bf16, T, y_bf16);
  if (st != MOE_OK) return st;
  if (T > 0 && !y_bf16) return MOE_ERR_INVALID_ARG;
  if (T > 0 && x_bf16 == y_bf16) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  ensure_device(x->device);
  const auto* xb = static_cast<const __nv_bfloat16*>(x_bf16);
  if (T == 1 && x->b1_enabled) {
    // the three kernels of a token form one PDL chain: profile it as a whole
    if (x->prof_start) CK(cudaEventRecordWithFlags(x->prof_start, s, cudaEventRecordExternal));
    CK(launch_router_b1(x, xb, s));
    CK(launch_experts_b1(x, xb, static_cast<__nv_bfloat16*>(y_bf16), residual, s));
    note_routing(x, 1, 1);
    if (x->prof_stop) CK(cudaEventRecordWithFlags(x->prof_stop, s, cudaEventRecordExternal));
    return MOE_OK;
  }
  CK(launch_router(x, xb, T, s));
  CK(launch_bucket(x, T, s));
  note_routing(x, T, 0);
  if (x->prof_start) CK(cudaEventRecordWithFlags(x->prof_start, s, cudaEventRecordExternal));
  if (x->mma_enabled) {
    CK(launch_mma_decode(x, xb, T, s));
  } else {
    CK(launch_gateup_decode(x, xb, T, s));
    CK(launch_down_decode(x, T, s));
  }
  if (x->prof_stop) CK(cudaEventRecordWithFlags(x->prof_stop, s, cudaEventRecordExternal));
  CK(launch_combine(x, xb, T, static_cast<__nv_bfloat16*>(y_bf16), residual, s));
  return MOE_OK;
}

moe_status moe_forward_prefill(moe_ctx* x, const void* x_bf16, int T, void* y_bf16, int residual,
                               cudaStream_t s) {
  moe_status st = check_fwd(x, x_bf16, T, y_bf16);
  if (st != MOE_OK) return st;
  if (T > 0 && !y_bf16) return MOE_ERR_INVALID_ARG;
  if (T > 0 && x_bf16 == y_bf16) return MOE_ERR_INVALID_ARG;
  if (!x->pf_enabled) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  ensure_device(x->device);
  const auto* xb = static_cast<const __nv_bfloat16*>(x_bf16);
  if (x->rt_enabled && T >= kRTcMinTokens) {
    CK(launch_router_tc(x, xb, T, s));
  } else {
    CK(launch_router(x, xb, T, s));
  }
  CK(launch_bucket(x, T, s));
  note_routing(x, T, 0);
  if (x->prof_start) CK(cudaEventRecordWithFlags(x->prof_start, s, cudaEventRecordExternal));
  CK(launch_prefill_experts(x, xb, T, s));
  if (x->prof_stop) CK(cudaEventRecordWithFlags(x->prof_stop, s, cudaEventRecordExternal));
  CK(launch_prefill_finish(x, xb, T, static_cast<__nv_bfloat16*>(y_bf16), residual, s));
  x->last_prefill_T = T;
  return MOE_OK;
}

moe_status moe_debug_prefill_h(moe_ctx* x, int T, uint8_t* h_codes, uint8_t* h_scales, cudaStream_t s) {
  if (!x || !h_codes || !h_scales || T < 0 || T > x->cfg.max_tokens) return MOE_ERR_INVALID_ARG;
  if (!x->pf_enabled) return MOE_ERR_UNSUPPORTED;
  if (T != x->last_prefill_T) return MOE_ERR_INVALID_ARG;
  ensure_device(x->device);
  CK(launch_gather_prefill_h(x, T, h_codes, h_scales, s));
  return MOE_OK;
}

moe_status moe_debug_routing(moe_ctx* x, int T, int32_t* idx, float* w, cudaStream_t s) {
  if (!x || !idx || !w || T < 0 || T > x->cfg.max_tokens) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  ensure_device(x->device);
  const size_t tk = (size_t)T * x->cfg.top_k;
  CK(cudaMemcpyAsync(idx, x->r.idx, tk * sizeof(int32_t), cudaMemcpyDeviceToDevice, s));
  CK(cudaMemcpyAsync(w, x->r.w, tk * sizeof(float), cudaMemcpyDeviceToDevice, s));
  return MOE_OK;
}

moe_status moe_quantize_nvfp4(const float* w, int n, int rows, int K, uint8_t* codes, uint8_t* scales,
                              float* ts, cudaStream_t s) {
  if (!w || !codes || !scales || !ts || n <= 0 || rows <= 0 || K <= 0 || K % 16 != 0 || n > 65535)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(w) || (reinterpret_cast<uintptr_t>(codes) & 7u) || (reinterpret_cast<uintptr_t>(ts) & 3u))
    return MOE_ERR_INVALID_ARG;
  CK(launch_quantize_nvfp4(w, n, rows, K, codes, scales, ts, s));
  return MOE_OK;
}

moe_status moe_set_profile_events(moe_ctx* x, cudaEvent_t start, cudaEvent_t stop) {
  if (!x) return MOE_ERR_INVALID_ARG;
  x->prof_start = start;
  x->prof_stop = stop;
  return MOE_OK;
}

moe_status moe_set_debug(moe_ctx* x, int flags) {
  if (!x || (flags & ~(MOE_DEBUG_KEEP_LOGITS | MOE_DEBUG_FORCE_TIMEOUT))) return MOE_ERR_INVALID_ARG;
  x->debug_flags = flags;
  return MOE_OK;
}

moe_status moe_debug_logits(moe_ctx* x, int T, float* logits, cudaStream_t s) {
  if (!x || !logits || T <= 0 || T != x->last_route_T || !x->last_route_kept) return MOE_ERR_INVALID_ARG;
  ensure_device(x->device);
  const float* src = x->last_route_b1 ? x->logits : x->dbg_logits;
  CK(cudaMemcpyAsync(logits, src, (size_t)T * x->cfg.n_experts * sizeof(float), cudaMemcpyDeviceToDevice, s));
  return MOE_OK;
}

moe_status moe_debug_wait_selftest(moe_ctx* x, int spin_limit, cudaStream_t s) {
  if (!x || spin_limit < 1) return MOE_ERR_INVALID_ARG;
  ensure_device(x->device);
  CK(launch_wait_selftest(x->status, (uint32_t)spin_limit, s));
  return MOE_OK;
}

moe_status moe_debug_fail_alloc(int n) {
  if (n < 0) return MOE_ERR_INVALID_ARG;
  g_fail_alloc_countdown.store(n);
  return MOE_OK;
}

moe_status moe_get_device_status(moe_ctx* x) {
  if (!x) return MOE_ERR_INVALID_ARG;
  ensure_device(x->device);
  CK(cudaDeviceSynchronize());
  int v = 0;
  CK(cudaMemcpy(&v, x->status, sizeof(int), cudaMemcpyDeviceToHost));
  CK(cudaMemset(x->status, 0, sizeof(int)));
  return static_cast<moe_status>(v);
}

int moe_kernels_per_forward(moe_ctx* x, int T, int prefill) {
  if (!x || T <= 0) return 0;
  if (!prefill && T == 1 && x->b1_enabled) return 3;
  const int nb = bucket_kernel_count(T);
  if (prefill) return 7 + nb;   // router x2, bucketing, quantise + scatter x, scale atoms, GEMM x2, finish
  if (x->mma_enabled) return 6 + nb;   // router x2, bucketing, x prescale, gate/up, down, combine
  return 5 + nb;
}

}  // extern "C"
