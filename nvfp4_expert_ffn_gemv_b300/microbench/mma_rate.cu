// Issue rate of the block-scaled FP4 tensor-core path on one SM: how long a
// K = 256 stage of tcgen05.mma kind::mxf4nvf4 (4 MMAs of K = 64) and its
// scale-factor copies (tcgen05.cp 32x128b.warpx4, one per 512-byte atom) take
// when issued back to back by one thread, operands resident in shared memory.
//   mma N=128 / N=256      4 MMAs per stage, M = 128
//   cp x8                  the 8 scale-factor copies of a 128 x 128 stage alone
//   cp x8 + mma N=128      the prefill GEMM's stage (A and B scales per k-step)
//   cp x12 + mma N=256     a 128 x 256 stage (B scales for 256 rows)
//   cp x4 + mma N=128      B scales only (A scales kept in TMEM)
//   cp x8 + mma N=256      B scales only, 128 x 256
//   (valid scales) mma     MMAs only, with every scale column written once
//                          before the timed loop (the variants above without
//                          copies read scale columns that were never written)
//   ... + TMA 32 KB/stage  the same, while a second thread streams 32 KB bulk
//                          copies from an L2-resident buffer into other shared
//                          memory (a 4-slot ring) for the whole loop, as the
//                          GEMM's operand loads do
//   ... + TMEM reads       the same, while warps 1-3 keep reading the other
//                          accumulator's columns (tcgen05.ld 32x32b.x32), as
//                          the GEMM's epilogue does
//   cp 128x256b / 128x128b the cost of the other tcgen05.cp shapes (no
//                          multicast: 128 lanes x 32 or 16 bytes, 4 KB or 2 KB
//                          into TMEM per copy) against 32x128b.warpx4 (512 B
//                          read, written to all four lane quarters: 2 KB);
//                          sources are arbitrary shared-memory bytes
//   2 threads: ...         the scale copies issued by a second thread (warp 1)
//                          into a 4-slot ring of TMEM scale columns: it
//                          commits each stage's copies to an mbarrier that the
//                          MMA thread waits on, and the MMA thread's commit
//                          frees the slot again
// Every CTA (one per SM) runs 256 stages; the time is from the first issue to
// the completion of the last operation (tcgen05.commit), in SM cycles.
// Operand values are arbitrary: only the rate is measured.
#include <cstdio>
#include <cstdint>
#include <cuda_runtime.h>

#include "../csrc/sm100.cuh"

using namespace nvmoe::sm100;

#define CK(x) do { cudaError_t err_ = (x); if (err_ != cudaSuccess) { \
  printf("CUDA error %s at %s:%d\n", cudaGetErrorString(err_), __FILE__, __LINE__); return 1; } } while (0)

constexpr int kStages = 256;
constexpr int kOffA = 0, kOffB = 16384, kOffSF = 49152, kUsed = kOffSF + 12 * 512;
constexpr int kOffRing = 57344, kSlot = 32768, kSlots = 4;
constexpr int kSmem = kOffRing + kSlots * kSlot + 1024;   // 189 KB: one CTA per SM
constexpr size_t kSrcBytes = (size_t)32 << 20;           // L2-resident source of the stream

struct Variant {
  int n;        // MMA N (0: no MMA)
  int ncp;      // scale-factor copies per stage
  int pre;      // write all scale columns once before timing
  int stream;   // concurrent TMA stream into shared memory
  int tld;      // concurrent TMEM loads by warps 1-3
  int split;    // scale copies issued by a second thread
  int shape;    // copy shape: 0 = 32x128b.warpx4, 1 = 128x256b, 2 = 128x128b
};

__device__ __forceinline__ void tmem_cp_128x256b(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.128x256b [%0], %1;" :: "r"(taddr), "l"(sdesc) : "memory");
}
__device__ __forceinline__ void tmem_cp_128x128b(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.128x128b [%0], %1;" :: "r"(taddr), "l"(sdesc) : "memory");
}

constexpr int kSfSlots = 4, kSfSlotCols = 48;   // ring of scale columns at 256 .. 447

__global__ void __launch_bounds__(128, 1) rate_kernel(Variant v, const uint8_t* __restrict__ src,
                                                      unsigned long long* cycles, int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t done_bar, stage_bar, ring_bar[kSlots], sf_full[kSfSlots], sf_empty[kSfSlots];
  __shared__ volatile int mma_done;
  __shared__ uint32_t tmem_base_s;
  for (int i = threadIdx.x; i < kUsed / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(smem)[i] = make_uint4(0x22222222u, 0x22222222u, 0x38383838u, 0x38383838u);
  if (threadIdx.x == 0) {
    mbar_init(&done_bar, 1);
    mbar_init(&stage_bar, 1);
    for (int k = 0; k < kSlots; ++k) mbar_init(&ring_bar[k], 1);
    for (int k = 0; k < kSfSlots; ++k) {
      mbar_init(&sf_full[k], 1);
      mbar_init(&sf_empty[k], 1);
    }
    mma_done = 0;
    fence_barrier_init();
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  if (threadIdx.x < 32) tmem_alloc(&tmem_base_s, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;
  if (v.split) {
    const uint32_t idesc = idesc_mxf4nvf4(128, v.n);
    const uint64_t adesc = desc_kmajor_sw128(smem_u32(smem + kOffA));
    const uint64_t bdesc = desc_kmajor_sw128(smem_u32(smem + kOffB));
    if (threadIdx.x == 0) {
      const unsigned long long t0 = clock64();
      bool ok = true;
      for (int s = 0; s < kStages && ok; ++s) {
        const int slot = s % kSfSlots;
        if (!wait_parity(&sf_full[slot], (uint32_t)(s / kSfSlots) & 1u)) { atomicExch(err, 4); ok = false; break; }
        tc_fence_after();
        const uint32_t base = tmem + 256 + slot * kSfSlotCols;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_mxf4nvf4(tmem, adesc + (uint64_t)(kk * 2), bdesc + (uint64_t)(kk * 2), idesc, base + kk * 4,
                       base + 16 + kk * 8, s > 0 || kk > 0);
        tc_commit(&sf_empty[slot]);
      }
      tc_commit(&done_bar);
      ok = wait_parity(&done_bar, 0) && ok;
      const unsigned long long t1 = clock64();
      if (!ok) atomicExch(err, 1);
      cycles[blockIdx.x] = t1 - t0;
    } else if (threadIdx.x == 32) {
      for (int s = 0; s < kStages; ++s) {
        const int slot = s % kSfSlots;
        if (!wait_parity(&sf_empty[slot], ((uint32_t)(s / kSfSlots) & 1u) ^ 1u)) { atomicExch(err, 5); break; }
        tc_fence_after();
        const uint32_t base = tmem + 256 + slot * kSfSlotCols;
        for (int c = 0; c < v.ncp; ++c)
          tmem_cp_sf_atom(base + 4 * c, desc_sf_atom(smem_u32(smem + kOffSF + 512 * c)));
        tc_commit(&sf_full[slot]);
      }
      // the last stages' slots: wait until the MMA thread has consumed them
      for (int s = kStages; s < kStages + kSfSlots; ++s) {
        const int slot = s % kSfSlots;
        if (!wait_parity(&sf_empty[slot], ((uint32_t)(s / kSfSlots) & 1u) ^ 1u)) { atomicExch(err, 6); break; }
      }
    }
  } else if (threadIdx.x == 0) {
    const uint32_t idesc = idesc_mxf4nvf4(128, v.n > 0 ? v.n : 128);
    const uint64_t adesc = desc_kmajor_sw128(smem_u32(smem + kOffA));
    const uint64_t bdesc = desc_kmajor_sw128(smem_u32(smem + kOffB));
    const uint32_t sfa = tmem + 256, sfb = tmem + 256 + 16;    // columns 256..271 (A), 272..319 (B)
    if (v.pre) {
      for (int c = 0; c < 12; ++c)
        tmem_cp_sf_atom(tmem + 256 + 4 * c, desc_sf_atom(smem_u32(smem + kOffSF + 512 * c)));
      tc_commit(&done_bar);
      if (!wait_parity(&done_bar, 0)) atomicExch(err, 1);
    }
    const unsigned long long t0 = clock64();
    for (int s = 0; s < kStages; ++s) {
      if (v.shape == 1) {
        // 128 rows x 32 bytes from the A region: 16 row groups of two 128-byte core matrices
        for (int c = 0; c < v.ncp; ++c)
          tmem_cp_128x256b(tmem + 256 + 8 * c, smem_desc(smem_u32(smem + kOffA), 128, 256, kLayoutNone));
      } else if (v.shape == 2) {
        // 128 rows x 16 bytes: 16 row groups of one 128-byte core matrix
        for (int c = 0; c < v.ncp; ++c)
          tmem_cp_128x128b(tmem + 256 + 4 * c, smem_desc(smem_u32(smem + kOffA), 128, 128, kLayoutNone));
      } else {
        for (int c = 0; c < v.ncp; ++c)
          tmem_cp_sf_atom(tmem + 256 + 4 * c, desc_sf_atom(smem_u32(smem + kOffSF + 512 * c)));
      }
      if (v.n > 0) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_mxf4nvf4(tmem, adesc + (uint64_t)(kk * 2), bdesc + (uint64_t)(kk * 2), idesc, sfa + kk * 4,
                       sfb + kk * 8, s > 0 || kk > 0);
      }
      tc_commit(&stage_bar);       // as the GEMM's per-stage release (nobody waits on it)
    }
    tc_commit(&done_bar);
    const bool ok = wait_parity(&done_bar, v.pre ? 1 : 0);
    const unsigned long long t1 = clock64();
    if (!ok) atomicExch(err, 1);
    cycles[blockIdx.x] = t1 - t0;
    mma_done = 1;
  } else if (threadIdx.x >= 32 && v.tld) {
    // warps 1-3: read columns 128..255 of their lane quarter until the MMAs
    // end (the exit test is warp-uniform: tcgen05.ld is a warp-wide instruction)
    const int q = (threadIdx.x >> 5) & 3;
    uint32_t acc = 0;
    for (int it = 0; it < (1 << 20); ++it) {
      if (__any_sync(0xffffffffu, mma_done != 0)) break;
      uint32_t r[32];
      tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + 128 + (it & 3) * 32, r);
#pragma unroll
      for (int j = 0; j < 32; ++j) acc += r[j];
    }
    if (acc == 0x12345678u) atomicExch(err, 3);   // keeps the loads
  } else if (threadIdx.x == 32 && v.stream) {
    // keep kSlots bulk copies in flight until the MMA thread has finished,
    // then wait for the ones still in flight
    const size_t nsrc = kSrcBytes / kSlot;
    uint32_t phase[kSlots] = {0, 0, 0, 0};
    bool inflight[kSlots];
    size_t n = blockIdx.x * 97;
    for (int k = 0; k < kSlots; ++k, ++n) {
      mbar_arrive_expect_tx(&ring_bar[k], kSlot);
      bulk_load(smem + kOffRing + k * kSlot, src + (n % nsrc) * kSlot, kSlot, &ring_bar[k]);
      inflight[k] = true;
    }
    for (bool any = true; any;) {
      any = false;
      for (int k = 0; k < kSlots; ++k) {
        if (!inflight[k]) continue;
        if (!wait_parity(&ring_bar[k], phase[k])) atomicExch(err, 2);   // gives up: the copy may still land
        phase[k] ^= 1;
        inflight[k] = false;
        if (!mma_done) {
          mbar_arrive_expect_tx(&ring_bar[k], kSlot);
          bulk_load(smem + kOffRing + k * kSlot, src + (n++ % nsrc) * kSlot, kSlot, &ring_bar[k]);
          inflight[k] = true;
        }
        any = any || inflight[k];
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x < 32) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

int main() {
  int nsm = 0;
  CK(cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, 0));
  unsigned long long* cyc;
  int* err;
  CK(cudaMalloc(&cyc, nsm * sizeof(unsigned long long)));
  CK(cudaMalloc(&err, sizeof(int)));
  CK(cudaMemset(err, 0, sizeof(int)));
  CK(cudaFuncSetAttribute(rate_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem));
  uint8_t* src;
  CK(cudaMalloc(&src, kSrcBytes));
  CK(cudaMemset(src, 0x33, kSrcBytes));
  const Variant vs[] = {{128, 0, 0, 0}, {256, 0, 0, 0}, {0, 8, 0, 0}, {128, 8, 0, 0}, {256, 12, 0, 0},
                        {128, 4, 0, 0}, {256, 8, 0, 0}, {128, 0, 1, 0}, {256, 0, 1, 0},
                        {128, 0, 1, 1}, {256, 0, 1, 1}, {128, 8, 0, 1}, {256, 12, 0, 1},
                        {128, 0, 1, 0, 1}, {128, 8, 0, 0, 1}, {256, 12, 0, 0, 0, 1}, {128, 8, 0, 0, 0, 1},
                        {0, 6, 0, 0, 0, 0, 1}, {0, 12, 0, 0, 0, 0, 2}, {256, 6, 0, 0, 0, 0, 1}};
  const char* names[] = {"mma N=128", "mma N=256", "cp x8", "cp x8 + mma N=128", "cp x12 + mma N=256",
                         "cp x4 + mma N=128", "cp x8 + mma N=256", "(valid scales) mma N=128",
                         "(valid scales) mma N=256", "mma N=128 + TMA stream", "mma N=256 + TMA stream",
                         "cp x8 + mma N=128 + TMA", "cp x12 + mma N=256 + TMA", "mma N=128 + TMEM reads",
                         "cp x8 + mma N=128 + TMEM reads", "2 threads: cp x12 + mma N=256",
                         "2 threads: cp x8 + mma N=128", "cp 128x256b x6", "cp 128x128b x12",
                         "cp 128x256b x6 + mma N=256"};
  unsigned long long h[1024];
  if (nsm > 1024) return 1;
  for (int i = 0; i < 20; ++i) {
    rate_kernel<<<nsm, 128, kSmem>>>(vs[i], src, cyc, err);   // warm-up
    CK(cudaGetLastError());
    rate_kernel<<<nsm, 128, kSmem>>>(vs[i], src, cyc, err);
    CK(cudaDeviceSynchronize());
    CK(cudaMemcpy(h, cyc, nsm * sizeof(unsigned long long), cudaMemcpyDeviceToHost));
    double mean = 0;
    for (int b = 0; b < nsm; ++b) mean += (double)h[b];
    mean /= nsm;
    const double per = mean / kStages;
    const double flop = vs[i].n > 0 ? 2.0 * 128 * vs[i].n * 256 : 0;
    printf("%-26s %8.1f cycles per K=256 stage  %8.0f FLOP/cycle/SM  (%.2f PFLOP/s at 148 SMs x 2.032 GHz)\n",
           names[i], per, flop / per, flop / per * 148 * 2.032e9 / 1e15);
  }
  int e;
  CK(cudaMemcpy(&e, err, sizeof(int), cudaMemcpyDeviceToHost));
  printf("err=%d\n", e);
  return e != 0;
}
