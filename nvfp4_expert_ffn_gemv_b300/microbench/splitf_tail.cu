// What a split-F batch-1 decode would pay after h, against what the
// three-kernel chain pays.
//
// In a split-F layer every CTA owns a slice of the k + S experts' hidden
// rows and applies W_down to it, so each CTA ends with a partial y of all
// d = 2048 outputs.  The partials must be summed across the grid before the
// bf16 y (+ residual) exists.  Two ways are timed here, inside one
// persistent cooperative kernel (every CTA resident, one per SM):
//   mode 0: every CTA adds its 2048 partials into an fp32 accumulator with
//           red.global.add.v4.f32 (one 16-byte reduction per thread), then
//           counts itself done (fence + atomic); the last CTA reads the
//           accumulator, writes bf16 y and clears the accumulator;
//   mode 1: clusters of 4 CTAs first sum their partials through distributed
//           shared memory, so each address takes a quarter of the
//           reductions, then the same count and last-CTA finish.
// The chain being replaced:
//   mode 2: every CTA stores its h values, a grid-wide barrier stands in for
//           the kernel boundary (a PDL boundary costs the same ~1.1 us), then
//           every CTA reads the 7 x 512 fp32 of h from L2 and writes its 16
//           bf16 outputs.
// Each iteration starts after a grid barrier; the time is from CTA 0 leaving
// it to the last bf16 store (max over CTAs).  Every wait is bounded.
#include <cstdio>
#include <algorithm>
#include <cstdint>
#include <vector>
#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace cg = cooperative_groups;

#define CK(x) do { cudaError_t e_ = (x); if (e_ != cudaSuccess) { \
  printf("CUDA error %s at %s:%d\n", cudaGetErrorString(e_), __FILE__, __LINE__); return 1; } } while (0)

constexpr int kThreads = 512, kD = 2048, kH = 7 * 512;

__device__ __forceinline__ unsigned long long gtimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// flat grid barrier: release add, acquire poll, bounded; false (for every
// thread of the CTA) when the poll gave up
__device__ bool grid_barrier(unsigned* counter, unsigned target, int* err) {
  __shared__ int ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    asm volatile("red.release.gpu.global.add.u32 [%0], 1;" :: "l"(counter) : "memory");
    unsigned v = 0;
    long spins = 0;
    ok = 1;
    do {
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(counter) : "memory");
      if (++spins > (1L << 20)) { atomicExch(err, 1); ok = 0; break; }
    } while (v < target);
  }
  __syncthreads();
  return ok != 0;
}

struct Args {
  unsigned* bar;                 // grid barrier counter
  unsigned* done;                // CTAs finished with their reductions (reset by the last)
  float* acc;                    // [kD] fp32 accumulator
  float* h;                      // [kH] fp32
  const __nv_bfloat16* x;        // [kD] residual
  __nv_bfloat16* y;              // [kD]
  unsigned long long* tstart;    // [iters] CTA 0 leaving the barrier
  unsigned long long* tend;      // [iters] max over CTAs of the last bf16 store
  int iters, mode;
  int* err;
};

__global__ void __launch_bounds__(kThreads, 1) tail_kernel(Args a) {
  __shared__ float4 part[kThreads];
  __shared__ float wsum[kThreads / 32];
  __shared__ int is_last;
  const int t = threadIdx.x, G = gridDim.x;
  unsigned epoch = 0;
  for (int it = 0; it < a.iters; ++it) {
    if (!grid_barrier(a.bar, ++epoch * (unsigned)G, a.err)) return;
    const unsigned long long t0 = gtimer();
    if (blockIdx.x == 0 && t == 0) a.tstart[it] = t0;
    if (a.mode <= 1) {
      const float4 p = make_float4(1.f, 1.f, 1.f, 1.f);   // this CTA's partial of outputs 4t .. 4t+3
      if (a.mode == 0) {
        asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};"
                     :: "l"(a.acc + 4 * t), "f"(p.x), "f"(p.y), "f"(p.z), "f"(p.w) : "memory");
      } else {
        cg::cluster_group cl = cg::this_cluster();
        part[t] = p;
        cl.sync();
        const int r = (int)cl.block_rank();
        if (t < kThreads / 4) {
          const int col = r * (kThreads / 4) + t;          // float4 column this CTA sums
          float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float4 v = *cl.map_shared_rank(&part[col], q);
            s.x += v.x; s.y += v.y; s.z += v.z; s.w += v.w;
          }
          asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};"
                       :: "l"(a.acc + 4 * col), "f"(s.x), "f"(s.y), "f"(s.z), "f"(s.w) : "memory");
        }
        cl.sync();   // peers have read this CTA's partials
      }
      __syncthreads();
      if (t == 0) {
        __threadfence();
        const unsigned old = atomicAdd(a.done, 1u);
        is_last = old == (unsigned)G - 1;
      }
      __syncthreads();
      if (is_last) {
        __threadfence();
        const float4 v = __ldcg(reinterpret_cast<const float4*>(a.acc) + t);
        const uint2 xv = __ldcg(reinterpret_cast<const uint2*>(a.x) + t);
        const float x0 = __uint_as_float(xv.x << 16), x1 = __uint_as_float(xv.x & 0xFFFF0000u);
        const float x2 = __uint_as_float(xv.y << 16), x3 = __uint_as_float(xv.y & 0xFFFF0000u);
        __nv_bfloat162 y01 = __floats2bfloat162_rn(x0 + v.x, x1 + v.y), y23 = __floats2bfloat162_rn(x2 + v.z, x3 + v.w);
        uint2 yo;
        yo.x = *reinterpret_cast<uint32_t*>(&y01);
        yo.y = *reinterpret_cast<uint32_t*>(&y23);
        reinterpret_cast<uint2*>(a.y)[t] = yo;
        __stcg(reinterpret_cast<float4*>(a.acc) + t, make_float4(0.f, 0.f, 0.f, 0.f));
        __syncthreads();
        if (t == 0) {
          *a.done = 0u;
          atomicMax(a.tend + it, gtimer());
        }
      }
    } else {
      // the chain: this CTA's ~25 h values, the boundary, then all of h back from L2
      const int per = (kH + G - 1) / G;
      if (t < per && blockIdx.x * per + t < kH) a.h[blockIdx.x * per + t] = 1.f + (float)it;
      if (!grid_barrier(a.bar, ++epoch * (unsigned)G, a.err)) return;
      float s = 0.f;
      for (int i = t; i < kH / 4; i += kThreads) {
        const float4 v = __ldcg(reinterpret_cast<const float4*>(a.h) + i);
        s += (v.x + v.y) + (v.z + v.w);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
      if ((t & 31) == 0) wsum[t >> 5] = s;
      __syncthreads();
      if (t < 16) {
        float v = 0.f;
        for (int w = 0; w < kThreads / 32; ++w) v += wsum[w];
        a.y[(blockIdx.x * 16 + t) % kD] = __float2bfloat16_rn(v * 1e-6f);
      }
      __syncthreads();
      if (t == 0) atomicMax(a.tend + it, gtimer());
    }
  }
}

int main() {
  int nsm = 0;
  CK(cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, 0));
  const int iters = 400;
  unsigned *bar, *done;
  float *acc, *h;
  __nv_bfloat16 *x, *y;
  unsigned long long *ts, *te;
  int* err;
  CK(cudaMalloc(&bar, 4));
  CK(cudaMalloc(&done, 4));
  CK(cudaMalloc(&acc, kD * 4));
  CK(cudaMalloc(&h, kH * 4));
  CK(cudaMalloc(&x, kD * 2));
  CK(cudaMalloc(&y, kD * 2));
  CK(cudaMalloc(&ts, iters * 8));
  CK(cudaMalloc(&te, iters * 8));
  CK(cudaMalloc(&err, 4));
  CK(cudaMemset(x, 0, kD * 2));
  CK(cudaMemset(err, 0, 4));
  const char* names[3] = {"split-F: red.v4 from every CTA + last-CTA finish",
                          "split-F: cluster-of-4 DSMEM sum, red.v4 + last-CTA finish",
                          "chain: store h, boundary (grid barrier), read h, store y"};
  int rc = 0;
  for (int mode = 0; mode < 3; ++mode) {
    int G = nsm;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    int na = 0;
    attr[na].id = cudaLaunchAttributeCooperative;
    attr[na].val.cooperative = 1;
    ++na;
    if (mode == 1) {
      attr[na].id = cudaLaunchAttributeClusterDimension;
      attr[na].val.clusterDim.x = 4;
      attr[na].val.clusterDim.y = 1;
      attr[na].val.clusterDim.z = 1;
      ++na;
      cudaLaunchConfig_t q = {};
      q.gridDim = dim3(nsm / 4 * 4);
      q.blockDim = dim3(kThreads);
      q.attrs = attr + 1;
      q.numAttrs = 1;
      int ncl = 0;
      CK(cudaOccupancyMaxActiveClusters(&ncl, tail_kernel, &q));
      G = (ncl < nsm / 4 ? ncl : nsm / 4) * 4;
    }
    cfg.gridDim = dim3(G);
    cfg.blockDim = dim3(kThreads);
    cfg.attrs = attr;
    cfg.numAttrs = na;
    CK(cudaMemset(bar, 0, 4));
    CK(cudaMemset(done, 0, 4));
    CK(cudaMemset(acc, 0, kD * 4));
    CK(cudaMemset(te, 0, iters * 8));
    Args a{bar, done, acc, h, x, y, ts, te, iters, mode, err};
    CK(cudaLaunchKernelEx(&cfg, tail_kernel, a));
    CK(cudaGetLastError());
    CK(cudaDeviceSynchronize());
    std::vector<unsigned long long> s(iters), e(iters);
    CK(cudaMemcpy(s.data(), ts, iters * 8, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(e.data(), te, iters * 8, cudaMemcpyDeviceToHost));
    double sum = 0;
    int n = 0;
    std::vector<double> d;
    for (int i = 10; i < iters; ++i) {   // skip the first iterations
      d.push_back((double)(long long)(e[i] - s[i]));
      sum += d.back();
      ++n;
    }
    std::vector<double> sorted = d;
    std::sort(sorted.begin(), sorted.end());
    std::vector<__nv_bfloat16> yh(kD);
    CK(cudaMemcpy(yh.data(), y, kD * 2, cudaMemcpyDeviceToHost));
    const float y0 = __bfloat162float(yh[0]);
    printf("%-60s %3d CTAs: mean %.3f us, median %.3f us%s\n", names[mode], G, sum / n / 1e3, sorted[n / 2] / 1e3,
           mode <= 1 ? (y0 == (float)G ? "  (sums ok)" : "  (SUMS WRONG)") : "");
    if (mode <= 1 && y0 != (float)G) rc = 1;
  }
  int ev;
  CK(cudaMemcpy(&ev, err, 4, cudaMemcpyDeviceToHost));
  printf("err=%d\n", ev);
  return rc || ev;
}
