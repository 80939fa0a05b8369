// Microbenchmark: PDL boundary cost against grid size, a flag hand-off
// between PDL-chained kernels (release counter / acquire poll instead of
// griddepcontrol.wait), and a cluster-hierarchical grid barrier.  Every wait
// is bounded.  Build and run with microbench/run.py.
#include <cstdio>
#include <cstdint>
#include <cuda_runtime.h>
#include <cooperative_groups.h>

namespace cg = cooperative_groups;

#define CK(x) do { cudaError_t e_ = (x); if (e_ != cudaSuccess) { printf("CUDA %s at %d\n", cudaGetErrorString(e_), __LINE__); return 1; } } while (0)

__device__ __forceinline__ void gd_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void gd_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__global__ void chain_kernel(int* words, int n) {
  gd_launch();
  gd_wait();
  if (threadIdx.x == 0) {
    int v = __ldcg(words + (blockIdx.x + 1) % n);
    words[blockIdx.x] = v + 1;
  }
}

// Flag hand-off: kernel number `gen` (1, 2, ...) waits until counter >= (gen - 1) * grid (every CTA
// of the previous kernel has published), reads the previous kernel's words, writes its own and
// publishes with a release add.  No griddepcontrol.wait: the kernel launches as soon as every CTA of
// the previous one has run griddepcontrol.launch_dependents, so the previous one is entirely resident.
__global__ void flag_kernel(int* words, int n, unsigned* counter, unsigned gen, int* err) {
  gd_launch();
  if (threadIdx.x == 0) {
    const unsigned target = (gen - 1) * gridDim.x;
    unsigned v = 0;
    long spins = 0;
    do {
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(counter) : "memory");
      if (++spins > (1L << 22)) { atomicExch(err, 1); break; }
    } while (v < target);
    const int x = __ldcg(words + (blockIdx.x + 1) % n);
    words[blockIdx.x] = x + 1;
    asm volatile("red.release.gpu.global.add.u32 [%0], 1;" :: "l"(counter) : "memory");
  }
}

// hierarchical barrier: cluster barrier, then one atomic per cluster, then cluster barrier
__global__ void __cluster_dims__(4, 1, 1) hbar_kernel(unsigned* counter, int iters, int* err, unsigned long long* t_out) {
  cg::cluster_group cl = cg::this_cluster();
  const unsigned nclusters = gridDim.x / 4;
  unsigned long long t0;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  for (int i = 0; i < iters; ++i) {
    cl.sync();
    if (cl.block_rank() == 0 && threadIdx.x == 0) {
      const unsigned target = (unsigned)(i + 1) * nclusters;
      asm volatile("red.release.gpu.global.add.u32 [%0], 1;" :: "l"(counter) : "memory");
      unsigned v = 0;
      long spins = 0;
      do {
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(counter) : "memory");
        if (++spins > (1L << 24)) { atomicExch(err, 1); break; }
      } while (v < target);
    }
    cl.sync();
  }
  unsigned long long t1;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t1));
  if (threadIdx.x == 0 && blockIdx.x == 0) *t_out = t1 - t0;
}

int main() {
  int nsm = 0;
  CK(cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, 0));
  cudaStream_t st;
  CK(cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking));
  int* words;
  CK(cudaMalloc(&words, 4096 * sizeof(int)));
  CK(cudaMemset(words, 0, 4096 * sizeof(int)));
  int* err;
  CK(cudaMalloc(&err, sizeof(int)));
  CK(cudaMemset(err, 0, sizeof(int)));
  unsigned* counter;
  CK(cudaMalloc(&counter, sizeof(unsigned)));
  cudaEvent_t a, b;
  CK(cudaEventCreate(&a));
  CK(cudaEventCreate(&b));
  const int N = 1000;

  // ---- 1. PDL chain vs grid size
  const int grids[] = {16, 64, 128, nsm, 2 * nsm};
  for (int gi = 0; gi < 5; ++gi) {
    const int G = grids[gi];
    cudaGraph_t g;
    cudaGraphExec_t ge;
    CK(cudaStreamBeginCapture(st, cudaStreamCaptureModeGlobal));
    for (int i = 0; i < N; ++i) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(G);
      cfg.blockDim = dim3(128);
      cfg.stream = st;
      cudaLaunchAttribute at[1];
      at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      at[0].val.programmaticStreamSerializationAllowed = 1;
      cfg.attrs = at;
      cfg.numAttrs = 1;
      CK(cudaLaunchKernelEx(&cfg, chain_kernel, words, G));
    }
    CK(cudaStreamEndCapture(st, &g));
    CK(cudaGraphInstantiate(&ge, g, 0));
    CK(cudaGraphLaunch(ge, st));
    CK(cudaEventRecord(a, st));
    CK(cudaGraphLaunch(ge, st));
    CK(cudaEventRecord(b, st));
    CK(cudaStreamSynchronize(st));
    float ms;
    CK(cudaEventElapsedTime(&ms, a, b));
    printf("PDL chain, grid %d: %.3f us per boundary\n", G, ms * 1e3 / N);
  }

  // ---- 2. flag hand-off chain (graph of N kernels, counter reset before each replay)
  for (int gi = 0; gi < 3; ++gi) {
    const int G = gi == 0 ? 64 : (gi == 1 ? nsm : 2 * nsm);
    cudaGraph_t g;
    cudaGraphExec_t ge;
    CK(cudaStreamBeginCapture(st, cudaStreamCaptureModeGlobal));
    CK(cudaMemsetAsync(counter, 0, sizeof(unsigned), st));
    for (int i = 0; i < N; ++i) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(G);
      cfg.blockDim = dim3(128);
      cfg.stream = st;
      cudaLaunchAttribute at[1];
      at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      at[0].val.programmaticStreamSerializationAllowed = 1;
      cfg.attrs = at;
      cfg.numAttrs = 1;
      CK(cudaLaunchKernelEx(&cfg, flag_kernel, words, G, counter, (unsigned)(i + 1), err));
    }
    CK(cudaStreamEndCapture(st, &g));
    CK(cudaGraphInstantiate(&ge, g, 0));
    CK(cudaGraphLaunch(ge, st));
    CK(cudaEventRecord(a, st));
    CK(cudaGraphLaunch(ge, st));
    CK(cudaEventRecord(b, st));
    CK(cudaStreamSynchronize(st));
    float ms;
    CK(cudaEventElapsedTime(&ms, a, b));
    int e;
    CK(cudaMemcpy(&e, err, 4, cudaMemcpyDeviceToHost));
    printf("flag hand-off chain, grid %d: %.3f us per hand-off (err=%d)\n", G, ms * 1e3 / N, e);
  }

  // ---- 3. hierarchical barrier (clusters of 4)
  unsigned long long* tout;
  CK(cudaMalloc(&tout, sizeof(unsigned long long)));
  for (int rep = 0; rep < 2; ++rep) {
    CK(cudaMemset(counter, 0, sizeof(unsigned)));
    const int iters = 2000;
    const int G = (nsm / 4) * 4;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(G);
    cfg.blockDim = dim3(128);
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeCooperative;
    at[0].val.cooperative = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    CK(cudaLaunchKernelEx(&cfg, hbar_kernel, counter, iters, err, tout));
    CK(cudaStreamSynchronize(st));
    unsigned long long t;
    CK(cudaMemcpy(&t, tout, 8, cudaMemcpyDeviceToHost));
    int e;
    CK(cudaMemcpy(&e, err, 4, cudaMemcpyDeviceToHost));
    printf("hierarchical barrier (clusters of 4, %d CTAs): %.3f us per barrier (err=%d)\n", G, t / 1e3 / iters, e);
  }
  return 0;
}
