// Layout check of the block-scaled FP4 MMA (tcgen05.mma kind::mxf4nvf4,
// scale_vec::4X) at N = 256: D[128 x N] = A[128 x 256] * B[N x 256]^T with
// E2M1 codes and one E4M3 scale per 16 values, as the prefill GEMM uses it.
//   A, B: K-major, 128 bytes (256 values) per row, 128-byte swizzle;
//   scales: 512-byte atoms of 128 rows x 4 blocks (row r, block j at byte
//     (r % 32) * 16 + (r / 32) * 4 + j), copied into TMEM with
//     tcgen05.cp 32x128b.warpx4 (4 columns per atom);
//   4 MMAs of K = 64 (one atom per operand and k-step, 128 rows of B each).
// For N = 256 the B scales of rows 128..255 need a TMEM place; two layouts
// are tried: (a) per k-step, rows 0..127 in 4 columns and rows 128..255 in
// the next 4 (8 columns per k-step); (b) rows 128..255 after all 4 k-steps of
// rows 0..127 (+16 columns).  N = 128 is the control.  Codes and scales are
// small, so the products and sums are exact and compared bit for bit.
#include <cstdio>
#include <cstdint>
#include <cstring>
#include <vector>
#include <cuda_runtime.h>

#include "../csrc/sm100.cuh"

using namespace nvmoe::sm100;

#define CK(x) do { cudaError_t err_ = (x); if (err_ != cudaSuccess) { \
  printf("CUDA error %s at %s:%d\n", cudaGetErrorString(err_), __FILE__, __LINE__); return 1; } } while (0)

constexpr int kM = 128, kNmax = 256, kK = 256;
constexpr int kOffA = 0, kOffB = kM * 128, kOffSFA = kOffB + kNmax * 128, kOffSFB = kOffSFA + 4 * 512;
constexpr int kSmem = kOffSFB + 8 * 512 + 1024;

// A codes [128][128 B], B codes [N][128 B], SFA [4 k-steps][512 B], SFB [4][2][512 B] (atoms as in smem);
// D out [128][N] fp32.  layout: 0 = (a), 1 = (b).
__global__ void __launch_bounds__(128, 1) mxf4_kernel(const uint8_t* __restrict__ A, const uint8_t* __restrict__ B,
                                                      const uint8_t* __restrict__ SFA, const uint8_t* __restrict__ SFB,
                                                      int N, int layout, float* __restrict__ D, int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t tmem_base_s;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // operands -> shared memory: codes with the 128-byte swizzle, scale atoms as they are
  for (int i = threadIdx.x; i < (kM + N) * 8; i += blockDim.x) {
    const int r = i / 8, g = i % 8;
    const uint8_t* src = r < kM ? A + r * 128 + g * 16 : B + (r - kM) * 128 + g * 16;
    uint8_t* dst = sm + (r < kM ? kOffA + r * 128 : kOffB + (r - kM) * 128) + ((g ^ (r % 8)) * 16);
    *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(src);
  }
  for (int i = threadIdx.x; i < 4 * 512 / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(sm + kOffSFA)[i] = reinterpret_cast<const uint4*>(SFA)[i];
  for (int i = threadIdx.x; i < 8 * 512 / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(sm + kOffSFB)[i] = reinterpret_cast<const uint4*>(SFB)[i];
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
  const uint32_t sfa = tmem + 256, sfb = tmem + 256 + 16;   // SFA 16 columns, SFB up to 32
  if (threadIdx.x == 0) {
    for (int kk = 0; kk < 4; ++kk) {
      tmem_cp_sf_atom(sfa + kk * 4, desc_sf_atom(smem_u32(sm + kOffSFA + kk * 512)));
      for (int h = 0; h < N / 128; ++h) {
        const uint32_t col = N == 128 ? sfb + kk * 4 : (layout == 0 ? sfb + kk * 8 + h * 4 : sfb + h * 16 + kk * 4);
        tmem_cp_sf_atom(col, desc_sf_atom(smem_u32(sm + kOffSFB + (kk * 2 + h) * 512)));
      }
    }
    const uint32_t idesc = idesc_mxf4nvf4(kM, N);
    const uint64_t adesc = desc_kmajor_sw128(smem_u32(sm + kOffA));
    const uint64_t bdesc = desc_kmajor_sw128(smem_u32(sm + kOffB));
    for (int kk = 0; kk < 4; ++kk) {
      const uint32_t sfb_k = N == 128 ? sfb + kk * 4 : (layout == 0 ? sfb + kk * 8 : sfb + kk * 4);
      mma_mxf4nvf4(tmem, adesc + (uint64_t)(kk * 2), bdesc + (uint64_t)(kk * 2), idesc, sfa + kk * 4, sfb_k, kk > 0);
    }
    tc_commit(&bar);
    if (!wait_parity(&bar, 0)) atomicExch(err, 1);
  }
  __syncthreads();
  tc_fence_after();
  for (int c0 = 0; c0 < N; c0 += 32) {
    uint32_t v[32];
    tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + c0, v);
    for (int j = 0; j < 32; ++j) D[(warp * 32 + lane) * N + c0 + j] = __uint_as_float(v[j]);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

static const float kE2M1[16] = {0.f, 0.5f, 1.f, 1.5f, 2.f, 3.f, 4.f, 6.f, -0.f, -0.5f, -1.f, -1.5f, -2.f, -3.f, -4.f, -6.f};

int main() {
  // codes: element k of row r in byte k / 2 (low nibble: even k); scales: E4M3 0x30 (0.5), 0x38 (1), 0x40 (2)
  uint32_t s = 777;
  auto rnd = [&]() { s = s * 1664525u + 1013904223u; return s >> 8; };
  std::vector<uint8_t> A(kM * 128), B(kNmax * 128), SFA(4 * 512), SFB(8 * 512);
  std::vector<uint8_t> sa(kM * 16), sb(kNmax * 16);   // scale of (row, block 0..15)
  const uint8_t sc3[3] = {0x30, 0x38, 0x40};
  const float scv[3] = {0.5f, 1.f, 2.f};
  std::vector<float> fsa(kM * 16), fsb(kNmax * 16);
  for (auto& b : A) b = (uint8_t)(rnd() & 0xFF);
  for (auto& b : B) b = (uint8_t)(rnd() & 0xFF);
  for (int r = 0; r < kM; ++r)
    for (int j = 0; j < 16; ++j) { const int q = rnd() % 3; sa[r * 16 + j] = sc3[q]; fsa[r * 16 + j] = scv[q]; }
  for (int r = 0; r < kNmax; ++r)
    for (int j = 0; j < 16; ++j) { const int q = rnd() % 3; sb[r * 16 + j] = sc3[q]; fsb[r * 16 + j] = scv[q]; }
  // atoms: k-step kk holds blocks 4kk..4kk+3
  for (int kk = 0; kk < 4; ++kk)
    for (int r = 0; r < kM; ++r)
      for (int j = 0; j < 4; ++j) SFA[kk * 512 + (r % 32) * 16 + (r / 32) * 4 + j] = sa[r * 16 + kk * 4 + j];
  for (int kk = 0; kk < 4; ++kk)
    for (int h = 0; h < 2; ++h)
      for (int r = 0; r < 128; ++r)
        for (int j = 0; j < 4; ++j)
          SFB[(kk * 2 + h) * 512 + (r % 32) * 16 + (r / 32) * 4 + j] = sb[(h * 128 + r) * 16 + kk * 4 + j];
  auto val = [&](const std::vector<uint8_t>& c, int r, int k) {
    const uint8_t b = c[r * 128 + k / 2];
    return kE2M1[(k & 1) ? (b >> 4) : (b & 15)];
  };
  uint8_t *dA, *dB, *dSA, *dSB;
  float* dD;
  int* err;
  CK(cudaMalloc(&dA, A.size()));
  CK(cudaMalloc(&dB, B.size()));
  CK(cudaMalloc(&dSA, SFA.size()));
  CK(cudaMalloc(&dSB, SFB.size()));
  CK(cudaMalloc(&dD, kM * kNmax * 4));
  CK(cudaMalloc(&err, 4));
  CK(cudaMemset(err, 0, 4));
  CK(cudaMemcpy(dA, A.data(), A.size(), cudaMemcpyHostToDevice));
  CK(cudaMemcpy(dB, B.data(), B.size(), cudaMemcpyHostToDevice));
  CK(cudaMemcpy(dSA, SFA.data(), SFA.size(), cudaMemcpyHostToDevice));
  CK(cudaMemcpy(dSB, SFB.data(), SFB.size(), cudaMemcpyHostToDevice));
  CK(cudaFuncSetAttribute(mxf4_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem));
  const int cases[3][2] = {{128, 0}, {256, 0}, {256, 1}};
  const char* names[3] = {"N=128 (control)", "N=256, layout (a)", "N=256, layout (b)"};
  int rc = 0;
  for (int ci = 0; ci < 3; ++ci) {
    const int N = cases[ci][0], layout = cases[ci][1];
    CK(cudaMemset(dD, 0, kM * kNmax * 4));
    mxf4_kernel<<<1, 128, kSmem>>>(dA, dB, dSA, dSB, N, layout, dD, err);
    CK(cudaGetLastError());
    CK(cudaDeviceSynchronize());
    std::vector<float> D(kM * N);
    CK(cudaMemcpy(D.data(), dD, D.size() * 4, cudaMemcpyDeviceToHost));
    int bad = 0, bad_lo = 0, bad_hi = 0;
    for (int m = 0; m < kM; ++m)
      for (int n = 0; n < N; ++n) {
        double ref = 0;
        for (int k = 0; k < kK; ++k)
          ref += (double)val(A, m, k) * fsa[m * 16 + k / 16] * val(B, n, k) * fsb[n * 16 + k / 16];
        if ((float)ref != D[m * N + n]) {
          ++bad;
          (n < 128 ? bad_lo : bad_hi)++;
        }
      }
    printf("%-20s %6d of %6d outputs differ (columns 0..127: %d, 128..255: %d)\n", names[ci], bad, kM * N, bad_lo,
           bad_hi);
    if (ci == 0 && bad) rc = 1;
  }
  int e;
  CK(cudaMemcpy(&e, err, 4, cudaMemcpyDeviceToHost));
  printf("err=%d\n", e);
  return rc || e;
}
