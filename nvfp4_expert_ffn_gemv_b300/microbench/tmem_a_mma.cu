// Layout check of tcgen05.mma kind::f16 with the A operand in tensor memory:
// D[128 x 16] = A[128 x 64] * B[16 x 64]^T, f16 inputs, fp32 accumulation.
//   A: written by 4 warps with tcgen05.st 32x32b (lane = row of A, 32-bit
//      column j = elements 2j, 2j+1 of the row), 32 columns = K 64;
//   B: 16 rows x 128 bytes in shared memory, K-major, 128-byte swizzle
//      (16-byte granule g of row r stored at granule g ^ (r % 8));
//   4 MMAs of K = 16: A columns advance by 8, the B descriptor by 32 bytes.
// Values are small integers, so the product is exact and compared bit for bit
// with the host's.  Then the same MMA chain is timed with A rewritten in TMEM
// before every K = 64 step, as a dequantising GEMV would do, and the issue
// rate of back-to-back MMAs (M = 128, K = 16, A in TMEM) is measured for
// N = 16 and N = 128: the per-instruction cost that bounds a decode GEMV whose
// weights are dequantised into TMEM (K = 16 per instruction, few tokens).
#include <cstdio>
#include <cstdint>
#include <cstring>
#include <vector>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "../csrc/sm100.cuh"

using namespace nvmoe::sm100;

#define CK(x) do { cudaError_t err_ = (x); if (err_ != cudaSuccess) { \
  printf("CUDA error %s at %s:%d\n", cudaGetErrorString(err_), __FILE__, __LINE__); return 1; } } while (0)

constexpr int kM = 128, kN = 16, kK = 64;

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0],"
      " {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
      :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
         "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
         "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
         "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N) {
  return (1u << 4)                          // D format: F32
         | (0u << 7)                        // A format: F16
         | (0u << 10)                       // B format: F16
         | ((uint32_t)(N >> 3) << 17)
         | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_f16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                           bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
      :: "r"(d_tmem), "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"((uint32_t)accumulate)
      : "memory");
}

// A [128][64] f16 and B [16][64] f16 row-major in global; D [128][16] fp32 out.
// reps > 1: the timed variant (A rewritten before every K step, D accumulated).
__global__ void __launch_bounds__(128, 1) tmem_a_kernel(const __half* __restrict__ A, const __half* __restrict__ B,
                                                        float* __restrict__ D, int reps, unsigned long long* cyc,
                                                        int* err) {
  __shared__ __align__(1024) uint8_t sb[kN * 128];
  __shared__ __align__(8) uint64_t bar;
  __shared__ __align__(8) uint64_t abar;
  __shared__ uint32_t tmem_base_s;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // B -> shared memory, 128-byte swizzle
  for (int i = threadIdx.x; i < kN * 8; i += blockDim.x) {
    const int r = i / 8, g = i % 8;
    *reinterpret_cast<uint4*>(sb + r * 128 + ((g ^ (r % 8)) * 16)) =
        *reinterpret_cast<const uint4*>(reinterpret_cast<const uint8_t*>(B) + r * 128 + g * 16);
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    mbar_init(&abar, 4);
    fence_barrier_init();
  }
  if (warp == 0) tmem_alloc(&tmem_base_s, 64);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;
  const uint32_t d_t = tmem, a_t = tmem + 32;   // D: columns 0..15, A: columns 32..63
  // this thread's row of A as 32 packed f16 pairs
  uint32_t ar[32];
  const int row = warp * 32 + lane;
#pragma unroll
  for (int j = 0; j < 32; ++j) ar[j] = reinterpret_cast<const uint32_t*>(A + row * kK)[j];
  const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
  const uint32_t idesc = idesc_f16_f32(kM, kN);
  const uint64_t bdesc = desc_kmajor_sw128(smem_u32(sb));
  unsigned long long t0 = 0;
  for (int it = 0; it < reps; ++it) {
    tmem_st32(a_t + lane_base, ar);
    tmem_wait_st();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&abar);
    if (threadIdx.x == 0) {
      if (!wait_parity(&abar, it & 1)) { atomicExch(err, 1); }
      tc_fence_after();
      if (it == 0) t0 = clock64();
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        mma_f16_ta(d_t, a_t + kk * 8, bdesc + (uint64_t)(kk * 2), idesc, it > 0 || kk > 0);
      tc_commit(&bar);
      // the next rewrite of A waits for these MMAs
      if (!wait_parity(&bar, it & 1)) atomicExch(err, 2);
    }
    __syncthreads();
    tc_fence_after();
  }
  if (threadIdx.x == 0) cyc[0] = clock64() - t0;
  uint32_t dv[32];
  tmem_ld32(d_t + lane_base, dv);
  if (reps == 1)
    for (int j = 0; j < kN; ++j) D[row * kN + j] = __uint_as_float(dv[j]);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 64);
  }
}

// 1024 back-to-back MMAs of 128 x N x 16 (A in TMEM, B in shared memory), one
// CTA per SM; cycles from the first issue to the completion of the last.
__global__ void __launch_bounds__(128, 1) tmem_a_rate_kernel(int N, unsigned long long* cyc, int* err) {
  __shared__ __align__(1024) uint8_t sb[256 * 128];   // B: up to 256 rows of 128 bytes
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t tmem_base_s;
  const int warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < 256 * 128 / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(sb)[i] = make_uint4(0x3C003C00u, 0x3C003C00u, 0u, 0u);
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  if (warp == 0) tmem_alloc(&tmem_base_s, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;
  if (threadIdx.x == 0) {
    const uint32_t idesc = idesc_f16_f32(kM, N);
    const uint64_t bdesc = desc_kmajor_sw128(smem_u32(sb));
    const uint32_t a_t = tmem + 384;   // A: columns 384..391 (contents arbitrary); D: 0..N-1
    const unsigned long long t0 = clock64();
    for (int i = 0; i < 1024; ++i) mma_f16_ta(tmem, a_t, bdesc + (uint64_t)((i & 3) * 2), idesc, i > 0);
    tc_commit(&bar);
    if (!wait_parity(&bar, 0)) atomicExch(err, 1);
    cyc[blockIdx.x] = clock64() - t0;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

int main() {
  std::vector<__half> a(kM * kK), b(kN * kK);
  std::vector<float> fa(kM * kK), fb(kN * kK);
  uint32_t s = 12345;
  auto rnd = [&]() { s = s * 1664525u + 1013904223u; return (int)((s >> 24) % 7) - 3; };
  for (int i = 0; i < kM * kK; ++i) { fa[i] = (float)rnd(); a[i] = __float2half(fa[i]); }
  for (int i = 0; i < kN * kK; ++i) { fb[i] = (float)rnd(); b[i] = __float2half(fb[i]); }
  __half *dA, *dB;
  float* dD;
  unsigned long long* cyc;
  int* err;
  CK(cudaMalloc(&dA, a.size() * 2));
  CK(cudaMalloc(&dB, b.size() * 2));
  CK(cudaMalloc(&dD, kM * kN * 4));
  CK(cudaMalloc(&cyc, 8));
  CK(cudaMalloc(&err, 4));
  CK(cudaMemset(err, 0, 4));
  CK(cudaMemset(dD, 0, kM * kN * 4));
  CK(cudaMemcpy(dA, a.data(), a.size() * 2, cudaMemcpyHostToDevice));
  CK(cudaMemcpy(dB, b.data(), b.size() * 2, cudaMemcpyHostToDevice));
  tmem_a_kernel<<<1, 128>>>(dA, dB, dD, 1, cyc, err);
  CK(cudaGetLastError());
  CK(cudaDeviceSynchronize());
  std::vector<float> d(kM * kN);
  CK(cudaMemcpy(d.data(), dD, d.size() * 4, cudaMemcpyDeviceToHost));
  int bad = 0;
  for (int m = 0; m < kM; ++m)
    for (int n = 0; n < kN; ++n) {
      float ref = 0.f;
      for (int k = 0; k < kK; ++k) ref += fa[m * kK + k] * fb[n * kK + k];
      if (ref != d[m * kN + n]) {
        if (bad < 5) printf("  mismatch D[%d][%d] = %g, want %g\n", m, n, d[m * kN + n], ref);
        ++bad;
      }
    }
  printf("A in TMEM, B swizzled in shared memory: %d of %d outputs differ\n", bad, kM * kN);
  const int reps = 1000;
  tmem_a_kernel<<<1, 128>>>(dA, dB, dD, reps, cyc, err);
  CK(cudaDeviceSynchronize());
  unsigned long long c;
  CK(cudaMemcpy(&c, cyc, 8, cudaMemcpyDeviceToHost));
  int e;
  CK(cudaMemcpy(&e, err, 4, cudaMemcpyDeviceToHost));
  printf("rewrite A (128 x 64 f16) + 4 MMAs + wait, serialised: %.1f cycles per K=64 step (err=%d)\n",
         (double)c / reps, e);
  int nsm = 0;
  CK(cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, 0));
  unsigned long long* cycs;
  CK(cudaMalloc(&cycs, nsm * 8));
  std::vector<unsigned long long> hc(nsm);
  for (int N : {16, 64, 128, 256}) {
    tmem_a_rate_kernel<<<nsm, 128>>>(N, cycs, err);
    tmem_a_rate_kernel<<<nsm, 128>>>(N, cycs, err);
    CK(cudaDeviceSynchronize());
    CK(cudaMemcpy(hc.data(), cycs, nsm * 8, cudaMemcpyDeviceToHost));
    double mean = 0;
    for (int b = 0; b < nsm; ++b) mean += (double)hc[b];
    mean /= nsm;
    printf("back-to-back kind::f16 MMA 128 x %3d x 16, A in TMEM: %.1f cycles per instruction (%.0f FLOP/cycle/SM)\n",
           N, mean / 1024, 2.0 * 128 * N * 16 / (mean / 1024));
  }
  CK(cudaMemcpy(&e, err, 4, cudaMemcpyDeviceToHost));
  return bad != 0 || e != 0;
}
