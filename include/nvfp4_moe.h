/*
 * nvfp4_moe.h -- C ABI of the NVFP4 sparse mixture-of-experts FFN layer (sm_103a).
 *
 * What the layer computes.  The Flint 40B-A2.5B pages ("Recursive Flint
 * 40B-A2.5B：まず速さを第一に考えて作られたコーディングモデル", OrcaRouter blog,
 * section "このアーキテクチャはメモリ帯域幅に関する主張である") give each MoE layer
 * 256 routed experts, 6 of them chosen per token, plus one always-on shared
 * expert, and ship the weights in NVFP4 (same page, section
 * "量子化のレシピは最も転用しやすい部分です").  Everything else is a stated
 * reading, identical in the library and its test oracle:
 *
 *   logits[t,e] = sum_k x[t,k] * W_r[k,e] (+ bias[e])            fp32
 *   idx[t,:]    = the top_k largest logits, descending, ties -> lower e
 *   w[t,j]      = softmax of the chosen logits (== full softmax renormalised)
 *   expert_e(x) = W_down,e (silu(W_gate,e x) * W_up,e x)          SwiGLU, no bias
 *   y[t]        = sum_j w[t,j] expert_{idx[t,j]}(x_t) + sum_s shared_s(x_t)
 *
 * NVFP4 tensor of R rows and K columns (K % 16 == 0), "canonical" layout:
 *   codes  uint8 [R][K/2]   E2M1 codes, two per byte, even k in the low nibble
 *   scales uint8 [R][K/16]  E4M3 (OCP E4M3FN) scale of each 16-element run along K
 *   ts     fp32             one scale per tensor;  value = e2m1 * e4m3 * ts
 * gate and up are [d_ff][d_model] (K = d_model), down is [d_model][d_ff].
 * Arrays of several experts are stacked on the first index.
 *
 * Conventions for every call:
 *   - Every pointer argument is a device pointer unless marked "host or
 *     device"; activations are bf16 row-major [T][d_model].
 *   - Argument errors are detected on the host before any work is queued and
 *     returned as MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED; nothing is launched
 *     then.  CUDA launch failures return MOE_ERR_CUDA.
 *   - Forward calls are asynchronous on `stream` (NULL = legacy default
 *     stream) and allocate nothing; all scratch is allocated by moe_init for
 *     config.max_tokens.  Conditions found on the device are latched in a
 *     device status word and reported by moe_get_device_status; no kernel
 *     ever traps.
 *   - A context is not thread-safe and its forward calls must not overlap on
 *     the GPU (they share the context's scratch).
 */
#ifndef NVFP4_MOE_H
#define NVFP4_MOE_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct moe_ctx moe_ctx; /* opaque, owned by the library */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,   /* NULL pointer, size out of range, misaligned pointer */
  MOE_ERR_UNSUPPORTED = 2,   /* valid but not implemented shape/format */
  MOE_ERR_OOM = 3,           /* cudaMalloc failed in moe_init */
  MOE_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed */
  MOE_ERR_TIMEOUT = 5,       /* a bounded device-side wait gave up */
  MOE_ERR_DEVICE_CHECK = 6   /* a device-side consistency check failed */
} moe_status;

typedef enum { MOE_W_NVFP4 = 0, MOE_W_BF16 = 1 } moe_weight_format;

/* Debug flags of moe_set_debug. */
enum {
  MOE_DEBUG_KEEP_LOGITS = 1,   /* routing stores the fp32 logits it ranked (moe_debug_logits) */
  MOE_DEBUG_FORCE_TIMEOUT = 2  /* kernels with bounded waits report MOE_ERR_TIMEOUT after their
                                  waits have completed normally (tests the status plumbing) */
};

typedef struct {
  int d_model;        /* hidden size: 256, 512, 1024, 2048 or 4096               */
  int n_experts;      /* routed experts, 1..256                                  */
  int top_k;          /* experts chosen per token, 1..min(8, n_experts)          */
  int d_ff;           /* expert width: 128, 256, 512 or 1024                     */
  int n_shared;       /* always-on shared experts, 0..2                          */
  int d_ff_shared;    /* width of the shared experts; must equal d_ff            */
  int max_tokens;     /* largest T any forward call will pass, 1..65536          */
  int weight_format;  /* moe_weight_format                                       */
} moe_config;

/* One weight matrix of a stack of experts (n = n_experts or n_shared).
 * NVFP4: codes/scales/tensor_scale as described above, bf16 NULL.
 * BF16:  bf16 = [n][rows][K] row-major bf16 values, the other three NULL.
 * Pointers may be host or device; they are read during moe_init only. */
typedef struct {
  const uint8_t* codes;
  const uint8_t* scales;
  const float* tensor_scale;
  const void* bf16;
} moe_matrix;

typedef struct {
  const float* router;       /* [d_model][n_experts] fp32, host or device        */
  const float* router_bias;  /* [n_experts] fp32 or NULL, host or device         */
  moe_matrix gate, up, down; /* routed experts                                   */
  moe_matrix shared_gate, shared_up, shared_down; /* shared experts (n_shared)   */
} moe_weights;

/* Validate the config, allocate the device arena on `device`, copy and
 * repack the weights into the library's device layouts, allocate scratch for
 * max_tokens.  On success *out owns all of it until moe_destroy.
 * Pages: the layer's shape (256 routed experts, 6 per token, one shared
 * expert, NVFP4 weights) is the OrcaRouter page's, sections
 * "このアーキテクチャはメモリ帯域幅に関する主張である" and
 * "量子化のレシピは最も転用しやすい部分です"; sizes are configurable.
 * Errors: MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED on the host before any
 * allocation, MOE_ERR_OOM when the arena cannot be allocated (nothing is
 * left allocated), MOE_ERR_CUDA if a copy or set-up kernel fails. */
MOE_API moe_status moe_init(const moe_config* cfg, const moe_weights* weights, int device,
                    moe_ctx** out);

/* Router only: logits, top-k, combine weights and per-expert token counts.
 * x [T][d_model] bf16 -> idx [T][top_k] int32, w [T][top_k] fp32,
 * counts [n_experts] int32 (any of the three outputs may be NULL), all
 * device pointers owned by the caller.  0 <= T <= max_tokens.
 * Pages: "6 of 256 experts per token" (OrcaRouter page, section
 * "このアーキテクチャはメモリ帯域幅に関する主張である"); the scoring function
 * (fp32 logits, top-k with ties to the lower expert, softmax renormalised over
 * the chosen k) is this library's reading, stated at the top of this file. */
MOE_API moe_status moe_route(moe_ctx* ctx, const void* x_bf16, int T, int32_t* idx, float* w,
                     int32_t* counts, cudaStream_t stream);

/* Router without a context and without any allocation.  The Flint pages have
 * no counterpart: it exists for callers that must not allocate device memory
 * (for example a scheduler embedded in a runtime that owns every byte of the
 * device through its own pool, which wants to know where tokens go -- to plan
 * expert placement or prefetch -- before or without creating a layer context).
 * Computes the same idx / w as moe_route, with the same kernels and the same
 * summation order, so the two agree bit for bit on the same inputs.
 *
 *   x_bf16      [T][d_model] bf16, device
 *   router      [d_model][n_experts] fp32, device;  router_bias [n_experts] fp32
 *               device, or NULL for none
 *   idx, w      [T][top_k] int32 / fp32 outputs, device, both required
 *   d_model a multiple of 256 in 256..4096, 1 <= n_experts <= 256,
 *   1 <= top_k <= min(8, n_experts); T == 0 does nothing.  A pointer the GPU
 *   cannot dereference (plain pageable host memory) is MOE_ERR_INVALID_ARG.
 *
 * Scratch: the split-K partial logits live in one fixed device array of
 * 1,048,576 fp32 (4 MiB) per device, inside the library's module.  A call needs
 * nkc * T * n_experts elements of it, where nkc (1..64) is the router's K split
 * for T; at n_experts = 256 every T up to 4096 fits.  A call that does not fit
 * returns MOE_ERR_UNSUPPORTED before anything is queued.  Nothing in the array
 * has to start at zero: each call writes every element it later reads.
 * On the first call on each device (with that device current) the array's
 * device address is looked up (cudaGetSymbolAddress) and the router kernel's
 * shared-memory limit is raised (cudaFuncSetAttribute); make that first call
 * outside any stream capture.  Calls are asynchronous on `stream`; two calls that can
 * run on the GPU at the same time (different streams, different host threads)
 * share the one array and race -- order them on one stream or with events.
 * Having no context, it has no device status word either: the device-side
 * consistency checks that moe_route reports through moe_get_device_status
 * are not reported by this entry point. */
MOE_API moe_status moe_route_noalloc(const void* x_bf16, int T, const float* router,
                             const float* router_bias, int d_model, int n_experts, int top_k,
                             int32_t* idx, float* w, cudaStream_t stream);

/* Decode form of the layer: activations stay exact (bf16 -> fp32), the NVFP4
 * weights are dequantised on the fly.  y [T][d_model] bf16 (may not alias x).
 * If `residual` is non-zero, y = bf16(x + layer(x)) (the stack's residual).
 * x and y are caller-owned device buffers, 16-byte aligned.
 * Pages: decode as moving each chosen weight from memory to the ALUs
 * (OrcaRouter page, section "このアーキテクチャはメモリ帯域幅に関する主張である"). */
MOE_API moe_status moe_forward_decode(moe_ctx* ctx, const void* x_bf16, int T, void* y_bf16,
                              int residual, cudaStream_t stream);

/* Prefill form: x and the SwiGLU output h are quantised to NVFP4 (16-element
 * E4M3 block scales, tensor scale 1) and every expert product runs as a
 * block-scaled FP4 x FP4 tensor-core GEMM.  NVFP4 weights only
 * (MOE_ERR_UNSUPPORTED otherwise).  Buffers as for moe_forward_decode.
 * Pages: the vendor lists "prompt processing" kernels among its custom
 * kernels (OrcaRouter page, section "量子化のレシピは最も転用しやすい部分です"). */
MOE_API moe_status moe_forward_prefill(moe_ctx* ctx, const void* x_bf16, int T, void* y_bf16,
                               int residual, cudaStream_t stream);

/* Pages: weights ship as NVFP4 (OrcaRouter page, section
 * "量子化のレシピは最も転用しやすい部分です"); the rules below are this
 * library's reading of the format.
 * Quantise n fp32 tensors w [n][rows][K] to canonical NVFP4 on the device:
 * codes [n][rows][K/2], scales [n][rows][K/16], ts [n].  Rules (all fp32,
 * round-to-nearest-even):  ts = amax/2688;  s = E4M3(amax_16 / (6*ts));
 * q = E2M1(v / (e4m3(s)*ts)); zero tensors give ts = 0 and zero codes.
 * K % 16 == 0.  Scratch-free; `w` is not modified. */
MOE_API moe_status moe_quantize_nvfp4(const float* w, int n, int rows, int K, uint8_t* codes,
                              uint8_t* scales, float* ts, cudaStream_t stream);

/* Copy the quantised SwiGLU activations h of the last prefill call to the
 * caller: h_codes [T*(top_k+n_shared)][d_ff/2], h_scales [...][d_ff/16], in
 * slot order s = t*top_k + j for routed slots, T*top_k + i*T + t for shared
 * expert i.  Asynchronous on `stream`.  For checking only. */
MOE_API moe_status moe_debug_prefill_h(moe_ctx* ctx, int T, uint8_t* h_codes, uint8_t* h_scales,
                               cudaStream_t stream);

/* Copy the routing of the last forward call (moe_forward_decode with T >= 2,
 * moe_forward_prefill, or moe_route) to the caller: idx [T][top_k] int32 and
 * w [T][top_k] fp32, device pointers.  T must be that call's T.  Prefill from
 * 256 tokens up computes its logits on the tensor cores, in another order of
 * fp32 additions than moe_route, so on a near-tie the two may pick different
 * experts; this call returns the ones prefill used.  For checking only. */
MOE_API moe_status moe_debug_routing(moe_ctx* ctx, int T, int32_t* idx, float* w, cudaStream_t stream);

/* Record `start` / `stop` (cudaEvent_t, may be NULL to disable) around the
 * expert kernels of every following forward call on its stream (for a
 * batch-1 decode: around its whole router -> experts -> down chain).  The records
 * are external event records, so inside a stream capture they become event
 * record nodes of the graph and can be timed after a replay. */
MOE_API moe_status moe_set_profile_events(moe_ctx* ctx, cudaEvent_t start, cudaEvent_t stop);

/* Debugging: set the context's debug flags (MOE_DEBUG_*; 0 clears them).
 * They apply to calls queued afterwards.  The pages have no counterpart. */
MOE_API moe_status moe_set_debug(moe_ctx* ctx, int flags);

/* Debugging: copy the fp32 logits the last routing ranked, logits
 * [T][n_experts] (device pointer), T = that call's T.  Available after a
 * batch-1 decode always, after other calls only if MOE_DEBUG_KEEP_LOGITS was
 * set when they were queued; MOE_ERR_INVALID_ARG otherwise.  Asynchronous on
 * `stream`.  The pages have no counterpart. */
MOE_API moe_status moe_debug_logits(moe_ctx* ctx, int T, float* logits, cudaStream_t stream);

/* Debugging: run the bounded device-side wait on an mbarrier that nothing
 * ever arrives on and nothing copies to, giving up after spin_limit polls
 * (>= 1).  The wait runs out and MOE_ERR_TIMEOUT is latched in the context's
 * status word, as when a product kernel's copy never lands; no asynchronous
 * operation is in flight, so the context stays usable.  The pages have no
 * counterpart. */
MOE_API moe_status moe_debug_wait_selftest(moe_ctx* ctx, int spin_limit, cudaStream_t stream);

/* Testing: make the n-th device allocation the library performs from now on
 * (the arena of a later moe_init) fail as if the device were out of memory;
 * 0 disables.  Process-wide.  The pages have no counterpart. */
MOE_API moe_status moe_debug_fail_alloc(int n);

/* ------------------------------------------------------------------------
 * Dense NVFP4 weights every token reads in full: the output layer and the
 * dense FFN layers.
 *
 * Pages: the output layer (lm_head) ships in 4 bits because, with ~2.5B
 * active parameters, it is a large share of the weights each token reads
 * (OrcaRouter page, section "量子化のレシピは最も転用しやすい部分です"); 2 of
 * the 49 layers are dense (section "このアーキテクチャはメモリ帯域幅に関する主張
 * である").  Their sizes are not on the pages; the readings taken here (vocab
 * 151,936, dense d_ff 18,432 at d_model 2048) follow from the pages' parameter
 * counts, but any size within the limits below is accepted.
 *
 * Both run as a streaming GEMV on the tensor cores with exact operands (NVFP4
 * weights and bf16 activations exact in f16, fp32 accumulation); up to 32
 * tokens share one pass over the weights, larger T takes several passes.
 * Weights are copied into a library-owned arena at init (host or device
 * pointers, canonical NVFP4 layout as above); forward calls allocate nothing,
 * are asynchronous on `stream`, and must not overlap on one context.
 * ------------------------------------------------------------------------ */
typedef struct moe_dense moe_dense; /* opaque, owned by the library */

/* lm_head: w = NVFP4 [vocab][d_model] (one tensor scale).  vocab % 16 == 0,
 * d_model a power of two in 256..4096, 1 <= max_tokens <= 4096. */
MOE_API moe_status moe_head_init(int vocab, int d_model, const moe_matrix* w, int max_tokens, int device,
                                 moe_dense** out);

/* logits [T][vocab] fp32 = x [T][d_model] bf16 . W^T; device pointers, 16-byte aligned. */
MOE_API moe_status moe_head_forward(moe_dense* head, const void* x_bf16, int T, float* logits,
                                    cudaStream_t stream);

/* Dense SwiGLU FFN: gate, up NVFP4 [d_ff][d_model], down [d_model][d_ff].
 * d_model a power of two in 256..4096; d_ff a multiple of 256 (at most 65536)
 * with a divisor K slice of at most 2304 that is a multiple of 128. */
MOE_API moe_status moe_ffn_init(int d_model, int d_ff, const moe_matrix* gate, const moe_matrix* up,
                                const moe_matrix* down, int max_tokens, int device, moe_dense** out);

/* y [T][d_model] bf16 = W_down (silu(W_gate x) * W_up x) (+ x when residual);
 * y may not alias x. */
MOE_API moe_status moe_ffn_forward(moe_dense* ffn, const void* x_bf16, int T, void* y_bf16, int residual,
                                   cudaStream_t stream);

/* Synchronise and return (then clear) the dense context's device status word. */
MOE_API moe_status moe_dense_get_device_status(moe_dense* ctx);

/* Number of kernels one moe_head_forward / moe_ffn_forward call launches for T
 * tokens (for accounting), in passes of up to 32 tokens: the output layer 2 per
 * pass; the dense FFN 5 per pass, or 4 for a one-token pass whose down
 * projection reads h itself (K slices of 2048).  0 for a NULL context or T <= 0.
 * The pages have no counterpart. */
MOE_API int moe_dense_kernels_per_forward(moe_dense* ctx, int T);

/* Free everything the dense context owns.  NULL is accepted. */
MOE_API moe_status moe_dense_destroy(moe_dense* ctx);

/* Synchronise the context's device and return the latched device status
 * (MOE_OK, MOE_ERR_TIMEOUT or MOE_ERR_DEVICE_CHECK), then clear it. */
MOE_API moe_status moe_get_device_status(moe_ctx* ctx);

/* Number of kernels one forward call launches for T tokens (for accounting):
 * 3 for batch-1 decode; otherwise the router (2), bucketing (1 kernel below
 * 1024 tokens, 3 from 1024 on) and the path's expert and combine kernels. */
MOE_API int moe_kernels_per_forward(moe_ctx* ctx, int T, int prefill);

/* Free everything the context owns.  NULL is accepted. */
MOE_API moe_status moe_destroy(moe_ctx* ctx);

/* Static description of a status code. */
MOE_API const char* moe_status_string(moe_status s);

#ifdef __cplusplus
}
#endif
#endif /* NVFP4_MOE_H */
