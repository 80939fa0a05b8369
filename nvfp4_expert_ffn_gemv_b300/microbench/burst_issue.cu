// Microbenchmark: a cold ~10.9 MB burst pulled by 148 SMs (72 KB each) with
// five issue strategies -- one thread of 16 KB bulk copies, 32 or 128 threads
// of smaller bulk copies, 512 threads of 16-byte loads, 512 threads of
// cp.async -- timed from the first issue to the last landed byte.  Every wait
// is bounded.  Build and run with microbench/run.py.
#include <cstdio>
#include <cstdint>
#include <cuda_runtime.h>

#define CK(x) do { cudaError_t e_ = (x); if (e_ != cudaSuccess) { printf("CUDA %s at %d\n", cudaGetErrorString(e_), __LINE__); return 1; } } while (0)

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ unsigned long long gtime() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

constexpr uint32_t kPer = 73728;   // 72 KB per CTA

__global__ void __launch_bounds__(512) burst_kernel(const uint8_t* src, int mode, unsigned long long* ts, int* err) {
  extern __shared__ __align__(128) uint8_t sm[];
  __shared__ __align__(8) uint64_t bar;
  __shared__ unsigned long long t_first;
  const uint8_t* s = src + (size_t)blockIdx.x * kPer;
  if (threadIdx.x == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" :: "r"(smem_u32(&bar)));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (threadIdx.x == 0) t_first = gtime();
  __syncthreads();
  if (mode <= 2) {
    const int nthr = mode == 0 ? 1 : (mode == 1 ? 32 : 128);
    const uint32_t chunk = mode == 0 ? 16384u : kPer / nthr;
    if (threadIdx.x == 0)
      asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}"
                   :: "r"(smem_u32(&bar)), "r"(kPer) : "memory");
    __syncthreads();
    if ((int)threadIdx.x < nthr) {
      for (uint32_t off = threadIdx.x * (mode == 0 ? 0 : chunk); off < (mode == 0 ? kPer : (threadIdx.x + 1) * chunk);
           off += (mode == 0 ? 16384u : chunk)) {
        const uint32_t len = min(mode == 0 ? 16384u : chunk, kPer - off);
        asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                     :: "r"(smem_u32(sm + off)), "l"(s + off), "r"(len), "r"(smem_u32(&bar)) : "memory");
      }
    }
    if (threadIdx.x == 0) {
      uint32_t ok = 0;
      for (long i = 0; i < (1L << 24) && !ok; ++i)
        asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], 0;\n\tselp.u32 %0, 1, 0, p;\n\t}"
                     : "=r"(ok) : "r"(smem_u32(&bar)) : "memory");
      if (!ok) atomicExch(err, 1);
    }
  } else if (mode == 3) {
    uint4 v[9];
#pragma unroll
    for (int i = 0; i < 9; ++i)
      v[i] = __ldcs(reinterpret_cast<const uint4*>(s) + threadIdx.x + 512 * i);
#pragma unroll
    for (int i = 0; i < 9; ++i) reinterpret_cast<uint4*>(sm)[threadIdx.x + 512 * i] = v[i];
  } else {
#pragma unroll
    for (int i = 0; i < 9; ++i) {
      const uint32_t o = (threadIdx.x + 512 * i) * 16;
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" :: "r"(smem_u32(sm + o)), "l"(s + o) : "memory");
    }
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    ts[blockIdx.x * 2] = t_first;
    ts[blockIdx.x * 2 + 1] = gtime();
  }
}

int main() {
  int nsm = 0;
  CK(cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, 0));
  if (nsm > 1024) return 1;
  cudaStream_t st;
  CK(cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking));
  int* err;
  CK(cudaMalloc(&err, sizeof(int)));
  CK(cudaMemset(err, 0, sizeof(int)));
  const size_t big = (size_t)4 << 30;
  uint8_t* buf;
  CK(cudaMalloc(&buf, big));
  CK(cudaMemset(buf, 1, big));
  unsigned long long* ts;
  CK(cudaMalloc(&ts, 1024 * 2 * sizeof(unsigned long long)));
  CK(cudaFuncSetAttribute(burst_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPer));
  static unsigned long long h[1024 * 2];
  const char* names[] = {"1 thread, 16 KB bulk copies", "32 lanes, 2304 B bulk copies", "128 threads, 576 B bulk copies",
                         "512 threads, ld.global.v4 x9", "512 threads, cp.async 16 B x9"};
  for (int rep = 0; rep < 2; ++rep)
    for (int mode = 0; mode < 5; ++mode) {
      double span = 0;
      const int reps = 30;
      for (int r = 0; r < reps; ++r) {
        const size_t off = ((size_t)(r + 1 + mode * reps + rep * 500) * 113ull * (1 << 20)) % (big - (size_t)nsm * kPer);
        burst_kernel<<<nsm, 512, kPer, st>>>(buf + (off & ~(size_t)4095), mode, ts, err);
        CK(cudaStreamSynchronize(st));
        CK(cudaMemcpy(h, ts, nsm * 2 * sizeof(unsigned long long), cudaMemcpyDeviceToHost));
        unsigned long long first = ~0ull, last = 0;
        for (int i = 0; i < nsm; ++i) {
          first = h[i * 2] < first ? h[i * 2] : first;
          last = h[i * 2 + 1] > last ? h[i * 2 + 1] : last;
        }
        span += (double)(last - first);
      }
      printf("%-34s cold %.1f MB: first issue -> last landed %.3f us (%.0f GB/s)\n", names[mode], nsm * kPer / 1e6,
             span / reps / 1e3, nsm * kPer / (span / reps));
    }
  int e;
  CK(cudaMemcpy(&e, err, 4, cudaMemcpyDeviceToHost));
  printf("err=%d\n", e);
  return 0;
}
