// Load-only model of the prefill gate/up GEMM's operand stream: does the
// layout of the weights limit how fast TMA can feed the tensor cores?
//
// One CTA per SM runs the GEMM's unit order (unit u -> 128-row token block
// u / 8, weight tile u % 8; CTA b takes units b, b + grid, ...).  Each unit
// streams K = 2048 FP4 values (1 KB per row) as 8 stages of 16 KB per operand
// through a 6-stage ring.  A producer thread issues the loads and a consumer
// thread frees each stage as soon as it lands (no MMA), so the time is that
// of the loads alone.  Weights: 257 experts x 1024 rows x 1 KB (269 MB, above
// L2); tokens: 298 blocks x 128 rows x 1 KB (39 MB, re-read by the 8 CTAs of
// a block).
//   layout "rows":  row-major [rows][1 KB]; a stage is a 2-D TMA box of
//                   128 rows x 128 bytes (rows 1 KB apart), 128-byte swizzle
//   layout "tiled": each stage's 16 KB stored contiguously; one bulk copy
// Operands: B only (the weight stream), or A + B as in the GEMM.
// Unit orders (A + B, row-major layout): round-robin over the grid one unit
// at a time (CTA b: b, b + grid, ...), in groups of 2, 4 or 8 consecutive
// units (one token block), or one contiguous run of units per CTA.
#include <cstdio>
#include <cstdint>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "../csrc/sm100.cuh"

using namespace nvmoe::sm100;

#define CK(x) do { cudaError_t err_ = (x); if (err_ != cudaSuccess) { \
  printf("CUDA error %s at %s:%d\n", cudaGetErrorString(err_), __FILE__, __LINE__); return 1; } } while (0)

constexpr int kNst = 6, kTile = 16384, kKs = 8, kNtiles = 8;
constexpr int kExperts = 257, kRowBlocks = 298;
constexpr int kUnits = kRowBlocks * kNtiles;

// j-th unit of CTA b under order g: g = 0 contiguous run, g >= 1 round-robin
// groups of g consecutive units; -1 when the CTA has no more units
__device__ __forceinline__ int unit_of(int g, int j) {
  if (g == 0) {
    const int begin = (int)(((long long)blockIdx.x * kUnits) / gridDim.x);
    const int end = (int)(((long long)(blockIdx.x + 1) * kUnits) / gridDim.x);
    return begin + j < end ? begin + j : -1;
  }
  const int u = (blockIdx.x + (j / g) * gridDim.x) * g + j % g;
  return u < kUnits ? u : -1;
}

__global__ void __launch_bounds__(64, 1) stream_kernel(const __grid_constant__ CUtensorMap tmA,
                                                       const __grid_constant__ CUtensorMap tmB,
                                                       const uint8_t* __restrict__ A, const uint8_t* __restrict__ B,
                                                       int tiled, int with_a, int order, int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t full_bar[kNst], empty_bar[kNst];
  __shared__ volatile int abort_flag;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kNst; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  const uint32_t bytes = with_a ? 2 * kTile : kTile;
  if (threadIdx.x == 0) {
    int stage = 0;
    uint32_t phase = 0;
    for (int j = 0; !abort_flag; ++j) {
      const int u = unit_of(order, j);
      if (u < 0) break;
      const int tb = u / kNtiles, nt = u % kNtiles;
      const int e = tb < kExperts - 1 ? tb : kExperts - 1;   // the last blocks share one expert
      for (int ks = 0; ks < kKs; ++ks) {
        if (!wait_parity(&empty_bar[stage], phase ^ 1)) { abort_flag = 1; atomicExch(err, 1); break; }
        mbar_arrive_expect_tx(&full_bar[stage], bytes);
        uint8_t* sa = smem + stage * 2 * kTile;
        uint8_t* sb = sa + kTile;
        if (tiled) {
          if (with_a) bulk_load(sa, A + ((size_t)tb * kKs + ks) * kTile, kTile, &full_bar[stage]);
          bulk_load(sb, B + (((size_t)e * kNtiles + nt) * kKs + ks) * kTile, kTile, &full_bar[stage]);
        } else {
          if (with_a) tma_load_2d(sa, &tmA, ks * 128, tb * 128, &full_bar[stage]);
          tma_load_2d(sb, &tmB, ks * 128, e * 1024 + nt * 128, &full_bar[stage]);
        }
        if (++stage == kNst) { stage = 0; phase ^= 1; }
      }
    }
  } else if (threadIdx.x == 32) {
    int stage = 0;
    uint32_t phase = 0;
    for (int j = 0; !abort_flag && unit_of(order, j) >= 0; ++j) {
      for (int ks = 0; ks < kKs; ++ks) {
        if (!wait_parity(&full_bar[stage], phase)) { abort_flag = 1; atomicExch(err, 2); break; }
        mbar_arrive(&empty_bar[stage]);
        if (++stage == kNst) { stage = 0; phase ^= 1; }
      }
    }
  }
  __syncthreads();
}

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
}

static bool make_tmap(CUtensorMap* m, const void* base, uint64_t rows, CUtensorMapL2promotion promo) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {1024, rows};
  const cuuint64_t strides[1] = {1024};
  const cuuint32_t box[2] = {128, 128};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, promo, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

int main() {
  int nsm = 0;
  CK(cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, 0));
  const size_t bbytes = (size_t)kExperts * 1024 * 1024, abytes = (size_t)kRowBlocks * 128 * 1024;
  uint8_t *A, *B;
  int* err;
  CK(cudaMalloc(&A, abytes));
  CK(cudaMalloc(&B, bbytes));
  CK(cudaMalloc(&err, sizeof(int)));
  CK(cudaMemset(A, 0x11, abytes));
  CK(cudaMemset(B, 0x22, bbytes));
  CK(cudaMemset(err, 0, sizeof(int)));
  const int smem = kNst * 2 * kTile + 1024;
  CK(cudaFuncSetAttribute(stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
  cudaEvent_t a, b;
  CK(cudaEventCreate(&a));
  CK(cudaEventCreate(&b));
  const CUtensorMapL2promotion promos[] = {CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_L2_PROMOTION_NONE};
  const char* pnames[] = {"L2 promotion 256B", "no L2 promotion"};
  for (int with_a = 0; with_a < 2; ++with_a) {
    for (int cfg = 0; cfg < 3; ++cfg) {
      const int tiled = cfg == 2;
      CUtensorMap ta, tb;
      const CUtensorMapL2promotion pr = promos[cfg == 1];
      if (!make_tmap(&ta, A, (uint64_t)kRowBlocks * 128, pr) || !make_tmap(&tb, B, (uint64_t)kExperts * 1024, pr)) {
        printf("tensor map encode failed\n");
        return 1;
      }
      stream_kernel<<<nsm, 64, smem>>>(ta, tb, A, B, tiled, with_a, 1, err);   // warm-up
      CK(cudaGetLastError());
      CK(cudaDeviceSynchronize());
      const int reps = 5;
      CK(cudaEventRecord(a));
      for (int r = 0; r < reps; ++r) stream_kernel<<<nsm, 64, smem>>>(ta, tb, A, B, tiled, with_a, 1, err);
      CK(cudaEventRecord(b));
      CK(cudaEventSynchronize(b));
      float ms;
      CK(cudaEventElapsedTime(&ms, a, b));
      const double us = ms * 1e3 / reps;
      const double moved = (double)kUnits * kKs * kTile * (with_a ? 2 : 1);
      printf("%-6s %-24s operands %-5s: %8.2f us per pass, %7.1f GB/s into shared memory (%.1f us per unit)\n",
             tiled ? "tiled" : "rows", tiled ? "(bulk copies)" : pnames[cfg == 1], with_a ? "A+B" : "B", us,
             moved / (us * 1e-6) / 1e9, us / ((double)kUnits / nsm));
    }
  }
  {
    CUtensorMap ta, tb;
    if (!make_tmap(&ta, A, (uint64_t)kRowBlocks * 128, promos[0]) || !make_tmap(&tb, B, (uint64_t)kExperts * 1024, promos[0]))
      return 1;
    const int orders[] = {1, 2, 4, 8, 0};
    for (int oi = 0; oi < 5; ++oi) {
      const int o = orders[oi];
      stream_kernel<<<nsm, 64, smem>>>(ta, tb, A, B, 0, 1, o, err);
      CK(cudaGetLastError());
      CK(cudaDeviceSynchronize());
      const int reps = 5;
      CK(cudaEventRecord(a));
      for (int r = 0; r < reps; ++r) stream_kernel<<<nsm, 64, smem>>>(ta, tb, A, B, 0, 1, o, err);
      CK(cudaEventRecord(b));
      CK(cudaEventSynchronize(b));
      float ms;
      CK(cudaEventElapsedTime(&ms, a, b));
      const double us = ms * 1e3 / reps;
      printf("order %-28s A+B rows: %8.2f us per pass, %7.1f GB/s into shared memory\n",
             o == 0 ? "contiguous run per CTA" : o == 1 ? "round-robin, 1 unit" : o == 2 ? "round-robin, groups of 2" :
             o == 4 ? "round-robin, groups of 4" : "round-robin, groups of 8",
             us, (double)kUnits * kKs * kTile * 2 / (us * 1e-6) / 1e9);
    }
  }
  int e;
  CK(cudaMemcpy(&e, err, sizeof(int), cudaMemcpyDeviceToHost));
  printf("err=%d\n", e);
  return e != 0;
}
