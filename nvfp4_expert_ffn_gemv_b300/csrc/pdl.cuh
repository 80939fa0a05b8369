// Programmatic dependent launch (PDL) for the kernels of a forward pass.
//
// A kernel launched with PDL (launch_maybe_pdl) may begin while the kernel before it
// in the stream is still running.  It must call pdl_wait() before it reads or
// writes anything an earlier kernel of the stream touches; what it does before
// that may only read data written before the forward began (the weights), or
// its own shared memory.  Data an earlier kernel wrote must not be read
// through the non-coherent path (__ldg, or a const __restrict__ pointer the
// compiler may turn into one) even after pdl_wait(): that path assumes the
// data is fixed for the kernel's whole life, and this kernel was alive while
// it was written.  Such reads use __ldcg or plain loads.  pdl_trigger() lets the next kernel be scheduled;
// every CTA calls it at its start, and a CTA that exits counts as triggered.
// A kernel launched this way after one that never triggers simply starts when
// that one ends, so foreign kernels in the stream keep their full ordering.
#pragma once

#include <cuda_runtime.h>

namespace nvmoe {

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Launch with PDL when `pdl` is set, as a plain stream-ordered launch
// otherwise (the kernel's pdl_wait / pdl_trigger then do nothing).
template <typename... KArgs, typename... Args>
cudaError_t launch_maybe_pdl(bool pdl, void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                             Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// The decode-sized batches chain their kernels with PDL; for prefill batches
// the measured step was faster with plain launches (its kernels are long, and
// the early-resident waiting CTAs of the next kernel gain nothing).
constexpr int kPdlMaxTokens = 256;
inline bool use_pdl(int T) { return T < kPdlMaxTokens; }

}  // namespace nvmoe
