// Ways to add 128 x 128 fp32 tiles into scattered token rows of an L2-resident
// fp32 accumulator, the write pattern of prefill's down-GEMM epilogue (each of
// the tile's 128 rows belongs to a different token; 16 column tiles cover
// d = 2048).  Four warps per CTA, one CTA per SM, thread m owns row m of the
// tile as the TMEM lane layout gives it, values in registers:
//   0. per-thread red.global.add.v4.f32 into its own row (32 rows per instruction)
//   1. staged through shared memory, then red.v4 with 8 lanes per row (4 rows per instruction)
//   2. staged through shared memory, then one 512-byte bulk reduce per row
//      (cp.reduce.async.bulk .add.f32, issued by the row's own thread)
//   3. as 2, in 128-byte bulk reduces per 32-column chunk
//   4. as 1, plain 16-byte stores (the write ceiling of the pattern)
// Every variant adds the same values to the same places, so the accumulators
// of variants 0-3 must agree exactly (all values are small integers).
#include <cstdio>
#include <cstdint>
#include <cstring>
#include <vector>
#include <cuda_runtime.h>

#define CK(x) do { cudaError_t err_ = (x); if (err_ != cudaSuccess) { \
  printf("CUDA error %s at %s:%d\n", cudaGetErrorString(err_), __FILE__, __LINE__); return 1; } } while (0)

constexpr int kT = 4096, kD = 2048, kRowsPerTok = 7;
constexpr int kTiles = kT * kRowsPerTok / 128 * (kD / 128);    // 3584 tiles, 235 MB of adds
constexpr int kStride512 = 528, kStride128 = 144;               // padded smem row strides (bytes)

__device__ __forceinline__ int tile_token(int tile, int r) {
  const uint32_t row = (uint32_t)(tile / (kD / 128)) * 128u + (uint32_t)r;
  return (int)((row * 2654435761u) % (uint32_t)kT);
}
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__global__ void __launch_bounds__(128) reduce_kernel(float* __restrict__ acc, int mode) {
  extern __shared__ __align__(128) uint8_t sm[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m = threadIdx.x;
  for (int tile = blockIdx.x; tile < kTiles; tile += gridDim.x) {
    const int nt = tile % (kD / 128);
    const int tok = tile_token(tile, m);
    float* dst = acc + (size_t)tok * kD + nt * 128;
    float v[128];
#pragma unroll
    for (int j = 0; j < 128; ++j) v[j] = (float)((m + j + tile) & 3);
    if (mode == 0) {
#pragma unroll
      for (int j = 0; j < 128; j += 4)
        asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst + j), "f"(v[j]), "f"(v[j + 1]),
                     "f"(v[j + 2]), "f"(v[j + 3]) : "memory");
    } else if (mode == 1 || mode == 4) {
      // 32 rows x 32 columns per warp at a time, staged with a 144-byte row stride
      uint8_t* ws = sm + warp * 32 * kStride128;
      __shared__ int toks[128];
      toks[m] = tok;
#pragma unroll
      for (int c = 0; c < 128; c += 32) {
        __syncwarp();
#pragma unroll
        for (int j = 0; j < 32; j += 4)
          *reinterpret_cast<float4*>(ws + lane * kStride128 + j * 4) = make_float4(v[c + j], v[c + j + 1], v[c + j + 2], v[c + j + 3]);
        __syncwarp();
#pragma unroll
        for (int rr = 0; rr < 32; rr += 4) {
          const int row = rr + (lane >> 3), q = lane & 7;
          const float4 x = *reinterpret_cast<const float4*>(ws + row * kStride128 + q * 16);
          float* p = acc + (size_t)toks[warp * 32 + row] * kD + nt * 128 + c + q * 4;
          if (mode == 1)
            asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(x.x), "f"(x.y), "f"(x.z), "f"(x.w) : "memory");
          else
            *reinterpret_cast<float4*>(p) = x;
        }
      }
      __syncwarp();   // every lane has read toks before the next tile rewrites it
    } else if (mode == 2) {
      uint8_t* row = sm + m * kStride512;
      asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");   // previous tile's reduce has read the row
#pragma unroll
      for (int j = 0; j < 128; j += 4)
        *reinterpret_cast<float4*>(row + j * 4) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], 512;"
                   ::"l"(dst), "r"(smem_u32(row)) : "memory");
      asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    } else {
      // 128-byte reduces, four row buffers per thread (one per 32-column chunk)
      uint8_t* row = sm + m * 4 * kStride128;
      asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
#pragma unroll
      for (int c = 0; c < 4; ++c) {
#pragma unroll
        for (int j = 0; j < 32; j += 4)
          *reinterpret_cast<float4*>(row + c * kStride128 + j * 4) =
              make_float4(v[c * 32 + j], v[c * 32 + j + 1], v[c * 32 + j + 2], v[c * 32 + j + 3]);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], 128;"
                     ::"l"(dst + c * 32), "r"(smem_u32(row + c * kStride128)) : "memory");
      }
      asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    }
  }
  if (mode == 2 || mode == 3) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

int main() {
  int nsm = 0;
  CK(cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, 0));
  const size_t n = (size_t)kT * kD;
  float* acc;
  CK(cudaMalloc(&acc, n * 4));
  const int smem = 128 * kStride512 > 128 * 4 * kStride128 ? 128 * kStride512 : 128 * 4 * kStride128;
  CK(cudaFuncSetAttribute(reduce_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
  cudaEvent_t a, b;
  CK(cudaEventCreate(&a));
  CK(cudaEventCreate(&b));
  const char* names[] = {"red.v4, 32 rows per instruction", "smem + red.v4, 4 rows per instruction",
                         "smem + 512-B bulk reduce per row", "smem + 128-B bulk reduce per chunk",
                         "smem + st.v4, 4 rows per instruction (ceiling)"};
  std::vector<float> ref(n), got(n);
  const int reps = 10;
  const double bytes = (double)kTiles * 128 * 128 * 4;
  for (int mode = 0; mode < 5; ++mode) {
    CK(cudaMemset(acc, 0, n * 4));
    reduce_kernel<<<nsm, 128, smem>>>(acc, mode);   // one pass: the accumulator to compare
    CK(cudaGetLastError());
    CK(cudaDeviceSynchronize());
    if (mode < 4) {
      CK(cudaMemcpy(mode == 0 ? ref.data() : got.data(), acc, n * 4, cudaMemcpyDeviceToHost));
      if (mode > 0) printf("  mode %d matches mode 0: %s\n", mode, memcmp(ref.data(), got.data(), n * 4) == 0 ? "yes" : "NO");
    }
    CK(cudaEventRecord(a));
    for (int r = 0; r < reps; ++r) reduce_kernel<<<nsm, 128, smem>>>(acc, mode);
    CK(cudaEventRecord(b));
    CK(cudaEventSynchronize(b));
    float ms;
    CK(cudaEventElapsedTime(&ms, a, b));
    printf("%-48s %8.2f us per 235 MB pass  %7.1f GB/s\n", names[mode], ms * 1e3 / reps, bytes * reps / (ms * 1e-3) / 1e9);
  }
  return 0;
}
