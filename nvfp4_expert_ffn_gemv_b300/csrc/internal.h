// Host-side context and kernel launchers of the NVFP4 MoE library.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

struct moe_ctx {
  moe_config cfg;
  int device = 0;
  int n_all = 0;        // routed + shared experts
  int sm_count = 0;

  // one device arena holding every buffer below
  uint8_t* arena = nullptr;
  size_t arena_bytes = 0;

  // weights (library layouts, see common.cuh)
  uint8_t* gu_codes = nullptr;
  uint8_t* gu_scales = nullptr;
  uint8_t* dn_codes = nullptr;
  uint8_t* dn_scales = nullptr;
  float* tsc = nullptr;
  __nv_bfloat16* gu_bf16 = nullptr;
  __nv_bfloat16* dn_bf16 = nullptr;
  float* router = nullptr;   // [d][E]
  float* bias = nullptr;     // [E] (zeros when absent)
  int has_bias = 0;

  // scratch, sized for cfg.max_tokens
  float* router_partial = nullptr;
  nvmoe::Routing r{};
  float* h = nullptr;        // [P][f] fp32, P = T*k + S*T positions
  float* yexp = nullptr;     // [P][d] fp32 per-position expert outputs (batched decode)
  float* yacc = nullptr;     // [max_tokens][d] fp32 prefill accumulator of the weighted expert outputs
  int* status = nullptr;     // device status word
  int max_positions = 0;

  // batched decode on the tensor cores (see decode_mma.cu)
  int mma_enabled = 0;
  uint8_t* x16 = nullptr;        // [max_tokens][d] f16, prescaled, k-permuted
  float* xunshift = nullptr;     // [max_tokens]

  // tensor-core router for long batches (see router_tc.cu)
  int rt_enabled = 0;
  __nv_bfloat16* rt_wsplit = nullptr;  // [3][Ep][d] bf16 splits of W_r^T
  float* rt_part = nullptr;            // [kRTcChunks][max_tokens][E] partial logits
  CUtensorMap rt_tmw;

  // batch-1 decode fast path (see decode_b1.cu / repack.cu)
  int b1_enabled = 0;
  int b1_grid = 0, b1_rmax = 0, b1_nbmax = 0;
  size_t b1_smem = 0;
  float* router_t = nullptr;     // [E][d]
  uint8_t* b1_rows = nullptr;    // [n_all][f][1.125 d] gate/up records per hidden row
  float* logits = nullptr;       // [E]

  // prefill (see prefill.cu)
  int pf_enabled = 0;
  int last_prefill_T = -1;
  uint8_t* pf_sfa_gu = nullptr;  // gate/up weight scale atoms [n_all][2f/128][d/64][512]
  uint8_t* pf_sfa_dn = nullptr;  // W_down scale atoms [n_all][d/128][f/64][512]
  uint8_t* pf_xq = nullptr;      // x in NVFP4, padded positions [rows][d/2]
  uint8_t* pf_xsf = nullptr;     // its scale atoms [rows/128][d/64][512]
  uint8_t* pf_hq = nullptr;      // h in NVFP4 [rows][f/2]
  uint8_t* pf_hsf = nullptr;     // its scale atoms [rows/128][f/64][512]
  CUtensorMap pf_tm[4];          // gate/up codes, W_down codes, x codes, h codes

  cudaEvent_t prof_start = nullptr;
  cudaEvent_t prof_stop = nullptr;

  // debugging (moe_set_debug): flags, logits of the last routing
  int debug_flags = 0;
  float* dbg_logits = nullptr;   // [max_tokens][E]
  int last_route_T = 0;          // tokens of the last routing
  int last_route_b1 = 0;         // 1 when it was the batch-1 path (logits in `logits`)
  int last_route_kept = 0;       // 1 when its logits were kept
};

namespace nvmoe {

// Where the top-k kernels store the logits they ranked: the context's debug
// buffer while MOE_DEBUG_KEEP_LOGITS is set, otherwise nowhere.
inline float* debug_logits(const moe_ctx* c) {
  return (c->debug_flags & MOE_DEBUG_KEEP_LOGITS) ? c->dbg_logits : nullptr;
}
cudaError_t launch_wait_selftest(int* status, uint32_t spin_limit, cudaStream_t s);
// Every device allocation of the library goes through here (moe_debug_fail_alloc can fail it).
cudaError_t device_alloc(void** p, size_t bytes);
cudaError_t launch_router(const moe_ctx* c, const __nv_bfloat16* x, int T, cudaStream_t s);
cudaError_t launch_bucket(const moe_ctx* c, int T, cudaStream_t s);
int bucket_kernel_count(int T);   // kernels launch_bucket() issues for T tokens
cudaError_t prepare_bucket_kernel();
cudaError_t launch_gateup_decode(const moe_ctx* c, const __nv_bfloat16* x, int T, cudaStream_t s);
cudaError_t launch_down_decode(const moe_ctx* c, int T, cudaStream_t s);
cudaError_t launch_combine(const moe_ctx* c, const __nv_bfloat16* x, int T, __nv_bfloat16* y,
                           int residual, cudaStream_t s);
cudaError_t launch_quantize_nvfp4(const float* w, int n, int rows, int K, uint8_t* codes,
                                  uint8_t* scales, float* ts, cudaStream_t s);
int router_chunks(int d, int T);
cudaError_t launch_router_topk(const float* part, const float* bias, int has_bias, int T, int E, int K, int nkc,
                               int32_t* idx, float* w, int* status, float* logits_out, cudaStream_t s);
constexpr int kRTcChunks = 4;   // K chunks of the tensor-core router
constexpr int kRTcMinTokens = 256;
int router_tc_padded_experts(const moe_config& c);
bool router_tc_supported(const moe_config& c);
cudaError_t router_tc_prepare(moe_ctx* c);
cudaError_t launch_router_tc(const moe_ctx* c, const __nv_bfloat16* x, int T, cudaStream_t s);
cudaError_t prepare_router_kernels();
// Allocation-free router (split-K partials in a static device array, see router.cu).
size_t router_static_capacity();
cudaError_t launch_router_static(const __nv_bfloat16* x, int T, const float* wr, const float* bias, int d,
                                 int E, int K, int32_t* idx, float* w, cudaStream_t s);
cudaError_t prepare_decode_kernels(const moe_ctx* c);
bool mma_decode_supported(const moe_config& c);
cudaError_t prepare_mma_decode(const moe_ctx* c);
cudaError_t launch_mma_decode(const moe_ctx* c, const __nv_bfloat16* x, int T, cudaStream_t s);
// 2-D byte tensor map [rows][row_bytes] with boxes of box_bytes x box_rows (prefill.cu)
bool make_tmap_u8(CUtensorMap* m, const void* base, uint64_t rows, uint64_t row_bytes, uint32_t box_bytes,
                  uint32_t box_rows, bool swizzle128);
bool prefill_supported(const moe_config& c);
bool prefill_accumulates(const moe_config& c, int T);
size_t prefill_max_rows(const moe_config& c);
cudaError_t prefill_prepare(moe_ctx* c);
cudaError_t launch_prefill_experts(const moe_ctx* c, const __nv_bfloat16* x, int T, cudaStream_t s);
cudaError_t launch_gather_prefill_h(const moe_ctx* c, int T, uint8_t* codes, uint8_t* sf, cudaStream_t s);
cudaError_t launch_prefill_finish(const moe_ctx* c, const __nv_bfloat16* x, int T, __nv_bfloat16* y, int residual,
                                  cudaStream_t s);
bool b1_supported(const moe_config& c);
bool b1_plan(const moe_config& c, int sm_count, int ctas_per_sm, int* grid, int* rmax, int* nbmax, size_t* smem);
size_t b1_row_bytes(int d);
cudaError_t prepare_b1_kernels(const moe_ctx* c);
cudaError_t repack_b1_layouts(moe_ctx* c);
cudaError_t launch_router_b1(const moe_ctx* c, const __nv_bfloat16* x, cudaStream_t s);
cudaError_t launch_experts_b1(const moe_ctx* c, const __nv_bfloat16* x, __nv_bfloat16* y, int residual,
                              cudaStream_t s);

}  // namespace nvmoe
