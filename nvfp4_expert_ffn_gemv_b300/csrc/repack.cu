// Init-time repacking of weights into the batch-1 decode layouts.
//
//   router_t   [E][d] fp32      W_r transposed, one contiguous row per expert
//   b1_rows    [n][f] gate/up records, record j of an expert:
//                gate row j codes (d/2) | up row j codes (d/2) |
//                gate row j scales (d/16) | up row j scales (d/16)
//              so a CTA that owns hidden rows [j0, j0+len) of an expert fetches
//              them with one bulk copy.  Gate/up scales are lane-ordered: lane
//              l of a warp finds the scales of its chunks c = l + 32q
//              (q < d/1024) in 2*d/1024 consecutive bytes.
#include "internal.h"

namespace nvmoe {

namespace {

__global__ void transpose_f32_kernel(const float* __restrict__ src, float* __restrict__ dst, int rows,
                                     int cols) {
  __shared__ float tile[32][33];
  const int c0 = blockIdx.x * 32, r0 = blockIdx.y * 32;
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int r = r0 + i, c = c0 + threadIdx.x;
    if (r < rows && c < cols) tile[i][threadIdx.x] = src[(size_t)r * cols + c];
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int c = c0 + i, r = r0 + threadIdx.x;
    if (r < rows && c < cols) dst[(size_t)c * rows + r] = tile[threadIdx.x][i];
  }
}

// one thread per output byte
__global__ void gu_scale_perm_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst,
                                     size_t n_rows, int d) {
  const int per_row = d / 16;
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n_rows * per_row) return;
  const size_t row = i / per_row;
  const int o = (int)(i % per_row);
  const int cpl = d / 1024;
  const int lane = o / (2 * cpl), rem = o % (2 * cpl);
  const int q = rem / 2, b = rem % 2;
  const int c = lane + 32 * q;
  dst[i] = src[row * per_row + 2 * c + b];
}

// one block per (hidden row j, expert e): gather the gate/up record from the
// tile-interleaved gate/up arrays and the lane-ordered scales
__global__ void assemble_rows_kernel(const uint8_t* __restrict__ gu_codes, const uint8_t* __restrict__ sperm,
                                     uint8_t* __restrict__ rows, int d, int f) {
  const int j = blockIdx.x, e = blockIdx.y;
  const size_t gub = (size_t)d + d / 8;
  uint8_t* rec = rows + ((size_t)e * f + j) * gub;
  const size_t grow = (size_t)e * 2 * f + gu_row_of_gate(j), urow = (size_t)e * 2 * f + gu_row_of_up(j);
  const uint4* srcs[4] = {reinterpret_cast<const uint4*>(gu_codes + grow * (d / 2)),
                          reinterpret_cast<const uint4*>(gu_codes + urow * (d / 2)),
                          reinterpret_cast<const uint4*>(sperm + grow * (d / 16)),
                          reinterpret_cast<const uint4*>(sperm + urow * (d / 16))};
  uint8_t* dsts[4] = {rec, rec + d / 2, rec + d, rec + d + d / 16};
  const int len16[4] = {d / 32, d / 32, d / 256, d / 256};
  for (int p = 0; p < 4; ++p)
    for (int i = threadIdx.x; i < len16[p]; i += blockDim.x) reinterpret_cast<uint4*>(dsts[p])[i] = srcs[p][i];
}

}  // namespace

cudaError_t repack_b1_layouts(moe_ctx* c) {
  const int d = c->cfg.d_model, f = c->cfg.d_ff, E = c->cfg.n_experts, n = c->n_all;
  transpose_f32_kernel<<<dim3((E + 31) / 32, (d + 31) / 32), dim3(32, 8)>>>(c->router, c->router_t, d, E);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  uint8_t* sperm = nullptr;
  const size_t gu_rows = (size_t)n * 2 * f;
  if ((e = device_alloc(reinterpret_cast<void**>(&sperm), gu_rows * (d / 16))) != cudaSuccess) return e;
  const size_t tot = gu_rows * (d / 16);
  gu_scale_perm_kernel<<<(unsigned)((tot + 255) / 256), 256>>>(c->gu_scales, sperm, gu_rows, d);
  assemble_rows_kernel<<<dim3(f, n), 128>>>(c->gu_codes, sperm, c->b1_rows, d, f);
  e = cudaGetLastError();
  cudaError_t e2 = cudaDeviceSynchronize();
  cudaFree(sperm);
  return e != cudaSuccess ? e : e2;
}

}  // namespace nvmoe
