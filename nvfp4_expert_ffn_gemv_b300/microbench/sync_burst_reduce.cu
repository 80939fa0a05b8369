// Microbenchmark behind the batch-1 and prefill design decisions (one B300):
//   1. the cost of a kernel boundary in a chain of 2000 kernels of 148 CTAs,
//      with and without programmatic dependent launch (PDL);
//   2. a grid-wide barrier inside one persistent cooperative kernel
//      (release add + acquire poll on one counter);
//   3. the time 148 SMs need to pull ~10.9 MB (72 KB each, bulk copies) cold
//      from HBM, and after an L2 prefetch issued 1-3 us earlier;
//   4. the throughput of red.global.add.v4.f32 against plain 16-byte stores
//      into a 32 MB buffer (L2-resident).
// Every wait is bounded.  Build and run with microbench/run.py.
#include <cstdio>
#include <cstdint>
#include <cuda_runtime.h>

#define CK(x) do { cudaError_t e_ = (x); if (e_ != cudaSuccess) { printf("CUDA %s at %d\n", cudaGetErrorString(e_), __LINE__); return 1; } } while (0)

__device__ __forceinline__ void gd_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void gd_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// chain kernel: each CTA reads word[blockIdx.x] (written by the previous kernel), writes word[...] + 1
__global__ void chain_kernel(int* words, int n) {
  gd_launch();
  gd_wait();
  if (threadIdx.x == 0) {
    int v = __ldcg(words + (blockIdx.x + 1) % n);
    words[blockIdx.x] = v + 1;
  }
}

// persistent: iters grid barriers; flat counter, bounded spin
__global__ void barrier_kernel(unsigned* counter, int iters, int* err, unsigned long long* t_out) {
  unsigned long long t0;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  for (int i = 0; i < iters; ++i) {
    __syncthreads();
    if (threadIdx.x == 0) {
      const unsigned target = (unsigned)(i + 1) * gridDim.x;
      asm volatile("red.release.gpu.global.add.u32 [%0], 1;" :: "l"(counter) : "memory");
      unsigned v = 0;
      long spins = 0;
      do {
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(counter) : "memory");
        if (++spins > (1L << 24)) { atomicExch(err, 1); break; }
      } while (v < target);
    }
    __syncthreads();
  }
  unsigned long long t1;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t1));
  if (threadIdx.x == 0 && blockIdx.x == 0) *t_out = t1 - t0;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

// burst: each CTA bulk-copies `bytes` from src + blockIdx.x * bytes into smem (in 16 KB pieces)
// and records globaltimer at issue and at completion.  Optional L2 prefetch of the same range
// `pre` ns before (issued by the same CTA, then spin on globaltimer).
__global__ void burst_kernel(const uint8_t* src, uint32_t bytes, long long pre_ns, unsigned long long* tstamp,
                             int* err) {
  extern __shared__ __align__(128) uint8_t sm[];
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" :: "r"(smem_u32(&bar)));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const uint8_t* s = src + (size_t)blockIdx.x * bytes;
  unsigned long long t0 = 0, t1 = 0, tp = 0;
  if (threadIdx.x == 0) {
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(tp));
    if (pre_ns > 0) {
      for (uint32_t off = 0; off < bytes; off += 16384)
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(s + off), "r"(min(16384u, bytes - off)) : "memory");
      unsigned long long now;
      do { asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(now)); } while ((long long)(now - tp) < pre_ns);
    }
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}"
                 :: "r"(smem_u32(&bar)), "r"(bytes) : "memory");
    for (uint32_t off = 0; off < bytes; off += 16384)
      asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                   :: "r"(smem_u32(sm + off)), "l"(s + off), "r"(min(16384u, bytes - off)), "r"(smem_u32(&bar)) : "memory");
    uint32_t ok = 0;
    for (long i = 0; i < (1L << 24) && !ok; ++i)
      asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], 0;\n\tselp.u32 %0, 1, 0, p;\n\t}"
                   : "=r"(ok) : "r"(smem_u32(&bar)) : "memory");
    if (!ok) atomicExch(err, 1);
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t1));
    tstamp[blockIdx.x * 3 + 0] = tp;
    tstamp[blockIdx.x * 3 + 1] = t0;
    tstamp[blockIdx.x * 3 + 2] = t1;
  }
  __syncthreads();
}


// red.global.add.v4.f32 throughput into a buffer of n16 16-byte slots (L2-resident at 32 MB):
// thread i of the grid adds to slots (i * 7919 + r * 104729) mod n16 for r < reps
__global__ void red_kernel(float* buf, size_t n16, int reps, int mode) {
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (int r = 0; r < reps; ++r) {
    const size_t slot = (i * 4 + (size_t)r * 104729ull * 4) % n16;   // neighbouring threads: neighbouring slots
    float* p = buf + slot * 4;
    if (mode == 0) {
      asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" :: "l"(p), "f"(1.f), "f"(2.f), "f"(3.f), "f"(4.f) : "memory");
    } else if (mode == 1) {
      *reinterpret_cast<float4*>(p) = make_float4(1.f, 2.f, 3.f, 4.f);
    } else {
      atomicAdd(p, 1.f);
    }
  }
}

int main() {
  int nsm = 0;
  CK(cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, 0));
  printf("SMs %d\n", nsm);
  cudaStream_t st;
  CK(cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking));
  int* words;
  CK(cudaMalloc(&words, 4096 * sizeof(int)));
  CK(cudaMemset(words, 0, 4096 * sizeof(int)));
  int* err;
  CK(cudaMalloc(&err, sizeof(int)));
  CK(cudaMemset(err, 0, sizeof(int)));
  cudaEvent_t a, b;
  CK(cudaEventCreate(&a));
  CK(cudaEventCreate(&b));

  // ---- 1. PDL chain of N kernels (148 CTAs x 128) in a graph
  for (int pdl = 0; pdl < 2; ++pdl) {
    const int N = 2000;
    cudaGraph_t g;
    cudaGraphExec_t ge;
    CK(cudaStreamBeginCapture(st, cudaStreamCaptureModeGlobal));
    for (int i = 0; i < N; ++i) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(nsm);
      cfg.blockDim = dim3(128);
      cfg.stream = st;
      cudaLaunchAttribute at[1];
      at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      at[0].val.programmaticStreamSerializationAllowed = pdl;
      cfg.attrs = at;
      cfg.numAttrs = 1;
      CK(cudaLaunchKernelEx(&cfg, chain_kernel, words, nsm));
    }
    CK(cudaStreamEndCapture(st, &g));
    CK(cudaGraphInstantiate(&ge, g, 0));
    CK(cudaGraphLaunch(ge, st));
    CK(cudaGraphLaunch(ge, st));
    CK(cudaEventRecord(a, st));
    CK(cudaGraphLaunch(ge, st));
    CK(cudaEventRecord(b, st));
    CK(cudaStreamSynchronize(st));
    float ms;
    CK(cudaEventElapsedTime(&ms, a, b));
    printf("chain pdl=%d: %.3f us per kernel boundary\n", pdl, ms * 1e3 / N);
  }

  // ---- 2. persistent grid barrier
  unsigned* counter;
  unsigned long long* tout;
  CK(cudaMalloc(&counter, sizeof(unsigned)));
  CK(cudaMalloc(&tout, sizeof(unsigned long long)));
  for (int rep = 0; rep < 3; ++rep) {
    CK(cudaMemset(counter, 0, sizeof(unsigned)));
    const int iters = 2000;
    void* args[] = {&counter, (void*)&iters, &err, &tout};
    CK(cudaLaunchCooperativeKernel((void*)barrier_kernel, dim3(nsm), dim3(128), args, 0, st));
    CK(cudaStreamSynchronize(st));
    unsigned long long t;
    CK(cudaMemcpy(&t, tout, 8, cudaMemcpyDeviceToHost));
    int e;
    CK(cudaMemcpy(&e, err, 4, cudaMemcpyDeviceToHost));
    printf("grid barrier (flat, %d CTAs): %.3f us per barrier (err=%d)\n", nsm, t / 1e3 / iters, e);
  }

  // ---- 3. cold burst: 148 CTAs x 72 KB from a 4 GB buffer, rotating regions
  const size_t big = (size_t)4 << 30;
  uint8_t* buf;
  CK(cudaMalloc(&buf, big));
  CK(cudaMemset(buf, 1, big));
  const uint32_t per = 73728;   // 72 KB per CTA -> 10.9 MB
  unsigned long long* ts;
  CK(cudaMalloc(&ts, nsm * 3 * sizeof(unsigned long long)));
  CK(cudaFuncSetAttribute(burst_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)per));
  unsigned long long h[1024 * 3];
  if (nsm > 1024) return 1;
  const long long pres[] = {0, 0, 1000, 2000, 3000};
  for (int pi = 0; pi < 5; ++pi) {
    double sum_span = 0, sum_max = 0;
    const int reps = 20;
    for (int r = 0; r < reps; ++r) {
      const size_t off = ((size_t)(r + 1 + pi * reps) * 97ull * (1 << 20)) % (big - (size_t)nsm * per);
      burst_kernel<<<nsm, 128, per, st>>>(buf + (off & ~(size_t)4095), per, pres[pi], ts, err);
      CK(cudaStreamSynchronize(st));
      CK(cudaMemcpy(h, ts, nsm * 3 * sizeof(unsigned long long), cudaMemcpyDeviceToHost));
      unsigned long long first = ~0ull, last = 0, maxd = 0;
      for (int i = 0; i < nsm; ++i) {
        first = h[i * 3 + 1] < first ? h[i * 3 + 1] : first;
        last = h[i * 3 + 2] > last ? h[i * 3 + 2] : last;
        const unsigned long long dd = h[i * 3 + 2] - h[i * 3 + 1];
        maxd = dd > maxd ? dd : maxd;
      }
      sum_span += (double)(last - first);
      sum_max += (double)maxd;
    }
    printf("burst %.1f MB, L2 prefetch %lld ns before: first-issue->last-land %.3f us, max per-CTA %.3f us\n",
           nsm * per / 1e6, pres[pi], sum_span / reps / 1e3, sum_max / reps / 1e3);
  }
  // ---- 4. vector fp32 reductions into a 32 MB buffer
  {
    const size_t n16 = (32u << 20) / 16;
    float* rb;
    CK(cudaMalloc(&rb, n16 * 16));
    CK(cudaMemset(rb, 0, n16 * 16));
    const int reps = 64, blocks = nsm * 8, threads = 256;
    const char* names[] = {"red.global.add.v4.f32", "st.global.v4 (plain store)", "atomicAdd f32 (scalar)"};
    for (int mode = 0; mode < 3; ++mode) {
      red_kernel<<<blocks, threads, 0, st>>>(rb, n16, 4, mode);
      CK(cudaEventRecord(a, st));
      red_kernel<<<blocks, threads, 0, st>>>(rb, n16, reps, mode);
      CK(cudaEventRecord(b, st));
      CK(cudaStreamSynchronize(st));
      float ms;
      CK(cudaEventElapsedTime(&ms, a, b));
      const double ops = (double)blocks * threads * reps;
      printf("%s: %.1f G ops/s (%.1f GB/s of payload) over 32 MB\n", names[mode], ops / (ms * 1e-3) / 1e9,
             ops * (mode == 2 ? 4 : 16) / (ms * 1e-3) / 1e9);
    }
  }
  int e;
  CK(cudaMemcpy(&e, err, 4, cudaMemcpyDeviceToHost));
  printf("err=%d\n", e);
  return 0;
}
