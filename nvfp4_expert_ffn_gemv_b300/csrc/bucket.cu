// Token -> expert bucketing: counts, exclusive offsets and a stable scatter.
//
// Not on the pages; it is the bookkeeping any batched MoE needs once the
// router has chosen k experts per token.  Positions p order the (token,
// expert) pairs by expert, token-major inside an expert; shared expert s
// follows at T*k + s*T + t.  Up to 1023 tokens, one block of 1024 threads:
//   A. each warp takes chunks of 32 tokens; a per-warp bitmask per expert
//      (atomicOr of 1 << lane) gives every pair its rank among the chunk's
//      tokens that chose the same expert (popc of the lower lanes) and the
//      chunk's count per expert;
//   B. thread e turns its column of chunk counts into an exclusive prefix;
//   C. warp 0 scans the per-expert totals into offsets and compacts the
//      active experts (count > 0), shared experts appended;
//   D. every pair lands at offsets[e] + prefix[chunk][e] + rank.
// All sums are integer, so the result is exact and deterministic.  When they
// fit, the per-chunk counts, ranks and chosen experts stay in shared memory;
// otherwise they go through global scratch.  From 1024 tokens on, the same
// phases run as three grids (see below), so A and D use every SM.
#include "internal.h"

namespace nvmoe {

namespace {

constexpr int kBucketThreads = 1024;
constexpr int kMaxE = 256;

// C. per-expert offsets and the active-expert list from the per-expert totals
// cnt[0..E) (one warp, 8 experts per lane; off gets E + 1 entries)
__device__ __forceinline__ void offsets_and_active(const Routing& r, const int* cnt, int* off, int T, int k, int E,
                                                   int S, int* status) {
  const int lane = threadIdx.x & 31;
  int local[8], lsum = 0, lact = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = lane * 8 + i;
    local[i] = (e < E) ? cnt[e] : 0;
    lsum += local[i];
    lact += local[i] > 0;
  }
  int incl = lsum, aincl = lact;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    const int a = __shfl_up_sync(0xffffffffu, aincl, o);
    if (lane >= o) { incl += v; aincl += a; }
  }
  int run = incl - lsum, a = aincl - lact;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = lane * 8 + i;
    if (e < E) {
      off[e] = run;
      r.offsets[e] = run;
      r.counts[e] = local[i];
      if (local[i] > 0) {
        r.act_e[a] = e;
        r.act_pos[a] = run;
        r.act_n[a] = local[i];
        ++a;
      }
    }
    run += local[i];
  }
  const int total = __shfl_sync(0xffffffffu, incl, 31);
  const int nact = __shfl_sync(0xffffffffu, aincl, 31);
  if (lane == 0) {
    off[E] = total;
    r.offsets[E] = total;
    int na = nact;
    if (T > 0) {
      for (int s = 0; s < S; ++s) {
        r.act_e[na] = E + s;
        r.act_pos[na] = T * k + s * T;
        r.act_n[na] = T;
        ++na;
      }
    }
    *r.n_active = na;
    if (total != T * k) latch_status(status, MOE_ERR_DEVICE_CHECK);
  }
  // padded 128-row blocks of the active experts (prefill's GEMM tiles) and
  // the active expert of every block, in the same compaction order
  int pl = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) pl += (local[i] + 127) >> 7;
  int pincl = pl;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, pincl, o);
    if (lane >= o) pincl += v;
  }
  int blk = pincl - pl, a2 = aincl - lact;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    if (local[i] > 0) {
      const int nb = (local[i] + 127) >> 7;
      r.act_ppos[a2] = blk * 128;
      for (int b = 0; b < nb; ++b) r.blk_a[blk + b] = a2;
      blk += nb;
      ++a2;
    }
  }
  const int rblocks = __shfl_sync(0xffffffffu, pincl, 31);
  const int nact2 = __shfl_sync(0xffffffffu, aincl, 31);
  int sblk = rblocks;
  const int snb = (T + 127) >> 7;
  for (int s2 = 0; s2 < (T > 0 ? S : 0); ++s2) {
    if (lane == 0) r.act_ppos[nact2 + s2] = sblk * 128;
    for (int b = lane; b < snb; b += 32) r.blk_a[sblk + b] = nact2 + s2;
    sblk += snb;
  }
  if (lane == 0) r.act_ppos[nact2 + (T > 0 ? S : 0)] = sblk * 128;
}

template <bool kSmem>
__global__ void __launch_bounds__(kBucketThreads) bucket_kernel(Routing r, int T, int k, int E,
                                                                int S, int* status) {
  extern __shared__ __align__(16) uint8_t bsm[];
  // shared-memory variant: pre [nchunks][E] uint16, then chosen expert and rank per pair (uint8)
  uint16_t* pre = reinterpret_cast<uint16_t*>(bsm);
  __shared__ uint32_t mask[kBucketThreads / 32][kMaxE];
  __shared__ int cnt[kMaxE];
  __shared__ int off[kMaxE + 1];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = blockDim.x >> 5;
  const int nchunks = (T + 31) / 32;
  uint8_t* ej_s = bsm + (size_t)nchunks * E * 2;
  uint8_t* rank_s = ej_s + (size_t)T * k;

  // A. per-chunk ranks and counts
  for (int c = warp; c < nchunks; c += nwarps) {
    for (int e = lane; e < E; e += 32) mask[warp][e] = 0u;
    __syncwarp();
    const int t = c * 32 + lane;
    const bool valid = t < T;
    int ej[8];
    if (valid) {
      for (int j = 0; j < k; ++j) {
        int e = r.idx[(size_t)t * k + j];
        if (e < 0 || e >= E) { latch_status(status, MOE_ERR_DEVICE_CHECK); e = 0; }
        ej[j] = e;
        atomicOr(&mask[warp][e], 1u << lane);
      }
    }
    __syncwarp();
    if (valid) {
      const uint32_t lower = (1u << lane) - 1u;
      for (int j = 0; j < k; ++j) {
        const int rk = __popc(mask[warp][ej[j]] & lower);
        if (kSmem) {
          rank_s[(size_t)t * k + j] = static_cast<uint8_t>(rk);
          ej_s[(size_t)t * k + j] = static_cast<uint8_t>(ej[j]);
        } else {
          r.rank[(size_t)t * k + j] = rk;
        }
      }
    }
    for (int e = lane; e < E; e += 32) {
      const int v = __popc(mask[warp][e]);
      if (kSmem) pre[(size_t)c * E + e] = static_cast<uint16_t>(v);
      else r.chunk_cnt[(size_t)c * E + e] = v;
    }
    __syncwarp();
  }
  __syncthreads();

  // B. exclusive prefix of each expert's chunk counts
  if (threadIdx.x < E) {
    const int e = threadIdx.x;
    int run = 0;
    if (kSmem) {
      for (int c = 0; c < nchunks; ++c) {
        const int v = pre[(size_t)c * E + e];
        pre[(size_t)c * E + e] = static_cast<uint16_t>(run);
        run += v;
      }
    } else {
      // 32 loads in flight per batch (the stores of a batch follow all its loads)
      for (int c0 = 0; c0 < nchunks; c0 += 32) {
        int v[32];
#pragma unroll
        for (int q = 0; q < 32; ++q) v[q] = c0 + q < nchunks ? __ldcg(r.chunk_cnt + (size_t)(c0 + q) * E + e) : 0;
#pragma unroll
        for (int q = 0; q < 32; ++q) {
          if (c0 + q < nchunks) r.chunk_cnt[(size_t)(c0 + q) * E + e] = run;
          run += v[q];
        }
      }
    }
    cnt[e] = run;
  }
  __syncthreads();

  if (warp == 0) offsets_and_active(r, cnt, off, T, k, E, S, status);
  __syncthreads();

  // D. stable scatter
  for (int s = threadIdx.x; s < T * k; s += blockDim.x) {
    const int t = s / k;
    int p;
    if (kSmem) {
      const int e = ej_s[s];
      p = off[e] + pre[(size_t)(t >> 5) * E + e] + rank_s[s];
    } else {
      int e = r.idx[s];
      if (e < 0 || e >= E) e = 0;
      p = off[e] + r.chunk_cnt[(size_t)(t >> 5) * E + e] + r.rank[s];
    }
    r.slot_pos[s] = p;
    r.pos_tok[p] = t;
    r.pos_w[p] = r.w[s];
  }
  for (int q = threadIdx.x; q < S * T; q += blockDim.x) {
    r.pos_tok[T * k + q] = q % T;
    r.pos_w[T * k + q] = 1.f;
  }
}

// ---------------------------------------------------------------------------
// Large batches: the same four phases as three grids, so that phases A and D
// run on every SM instead of one.  Chunks of 32 tokens are grouped by 8
// (256 tokens):
//   count:   one block per group, one warp per chunk (phase A) -> rank; the
//            block also prefixes its 8 chunk counts per expert (chunk_cnt,
//            relative to the group) and writes the group totals (group_cnt)
//   scan:    one block; four threads per expert prefix the group totals
//            (phase B), then warp 0 runs phase C
//   scatter: one thread per (token, choice) pair (phase D)
// ---------------------------------------------------------------------------
constexpr int kGroupChunks = 8;                      // chunks per group = warps per count block
constexpr int kScanThreads = 1024;
constexpr int kScanParts = kScanThreads / kMaxE;   // threads per expert
constexpr int kScanBatch = 32;                       // loads in flight per thread

__global__ void __launch_bounds__(kGroupChunks * 32) bucket_count_kernel(Routing r, int T, int k, int E,
                                                                         int* status) {
  __shared__ uint32_t mask[kGroupChunks][kMaxE];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nchunks = (T + 31) / 32;
  const int g = blockIdx.x, c = g * kGroupChunks + warp;
  for (int e = lane; e < E; e += 32) mask[warp][e] = 0u;
  __syncwarp();
  if (c < nchunks) {
    const int t = c * 32 + lane;
    const bool valid = t < T;
    int ej[8];
    if (valid) {
      for (int j = 0; j < k; ++j) {
        int e = __ldg(r.idx + (size_t)t * k + j);
        if (e < 0 || e >= E) { latch_status(status, MOE_ERR_DEVICE_CHECK); e = 0; }
        ej[j] = e;
        atomicOr(&mask[warp][e], 1u << lane);
      }
    }
    __syncwarp();
    if (valid) {
      const uint32_t lower = (1u << lane) - 1u;
      for (int j = 0; j < k; ++j) r.rank[(size_t)t * k + j] = __popc(mask[warp][ej[j]] & lower);
    }
  }
  __syncthreads();
  // per expert: each chunk's count prefix inside the group, and the group total
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = 0;
    for (int w = 0; w < kGroupChunks; ++w) {
      const int cc = g * kGroupChunks + w;
      if (cc >= nchunks) break;
      r.chunk_cnt[(size_t)cc * E + e] = run;
      run += __popc(mask[w][e]);
    }
    r.group_cnt[(size_t)g * E + e] = run;
  }
}

__global__ void __launch_bounds__(kScanThreads) bucket_scan_kernel(Routing r, int T, int k, int E, int S,
                                                                   int* status) {
  __shared__ int part[kScanParts][kMaxE];
  __shared__ int cnt[kMaxE];
  __shared__ int off[kMaxE + 1];
  const int e = threadIdx.x % kMaxE, q = threadIdx.x / kMaxE;
  const int ngroups = ((T + 31) / 32 + kGroupChunks - 1) / kGroupChunks;
  const int per = (ngroups + kScanParts - 1) / kScanParts;
  const int g0 = min(ngroups, q * per), g1 = min(ngroups, g0 + per);
  // B1. this thread's share of expert e's group totals
  int sum = 0;
  if (e < E) {
    for (int gb = g0; gb < g1; gb += kScanBatch) {
      int v[kScanBatch];
#pragma unroll
      for (int i = 0; i < kScanBatch; ++i) v[i] = gb + i < g1 ? __ldcg(r.group_cnt + (size_t)(gb + i) * E + e) : 0;
#pragma unroll
      for (int i = 0; i < kScanBatch; ++i) sum += v[i];
    }
  }
  part[q][e] = sum;
  __syncthreads();
  // B2. exclusive prefix over the groups, in group order
  if (e < E) {
    int run = 0;
    for (int qq = 0; qq < q; ++qq) run += part[qq][e];
    for (int gb = g0; gb < g1; gb += kScanBatch) {
      int v[kScanBatch];
#pragma unroll
      for (int i = 0; i < kScanBatch; ++i) v[i] = gb + i < g1 ? __ldcg(r.group_cnt + (size_t)(gb + i) * E + e) : 0;
#pragma unroll
      for (int i = 0; i < kScanBatch; ++i) {
        if (gb + i < g1) r.group_cnt[(size_t)(gb + i) * E + e] = run;
        run += v[i];
      }
    }
    if (q == kScanParts - 1) cnt[e] = run;
  }
  __syncthreads();
  if (threadIdx.x < 32) offsets_and_active(r, cnt, off, T, k, E, S, status);
}

__global__ void __launch_bounds__(256) bucket_scatter_kernel(Routing r, int T, int k, int E, int S) {
  const int s = blockIdx.x * blockDim.x + threadIdx.x;
  if (s < T * k) {
    const int t = s / k;
    int e = __ldg(r.idx + s);
    if (e < 0 || e >= E) e = 0;   // reported by the count kernel
    const int p = __ldg(r.offsets + e) + __ldg(r.group_cnt + (size_t)(t >> 8) * E + e) +
                  __ldg(r.chunk_cnt + (size_t)(t >> 5) * E + e) + __ldg(r.rank + s);
    r.slot_pos[s] = p;
    r.pos_tok[p] = t;
    r.pos_w[p] = __ldg(r.w + s);
  } else if (s < T * k + S * T) {
    const int q = s - T * k;
    r.pos_tok[T * k + q] = q % T;
    r.pos_w[T * k + q] = 1.f;
  }
}

}  // namespace

size_t bucket_smem_bytes(int T, int k, int E) { return (size_t)((T + 31) / 32) * E * 2 + (size_t)2 * T * k; }

constexpr size_t kBucketSmemMax = 180 * 1024;

cudaError_t prepare_bucket_kernel() {
  return cudaFuncSetAttribute(bucket_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kBucketSmemMax);
}

// Batches of at least this many tokens take the three-grid path.
constexpr int kBucketGridTokens = 1024;

int bucket_kernel_count(int T) { return T >= kBucketGridTokens ? 3 : 1; }

cudaError_t launch_bucket(const moe_ctx* c, int T, cudaStream_t s) {
  const int k = c->cfg.top_k, E = c->cfg.n_experts, S = c->cfg.n_shared;
  if (T >= kBucketGridTokens) {
    const int ngroups = (T + 32 * kGroupChunks - 1) / (32 * kGroupChunks);
    bucket_count_kernel<<<ngroups, kGroupChunks * 32, 0, s>>>(c->r, T, k, E, c->status);
    bucket_scan_kernel<<<1, kScanThreads, 0, s>>>(c->r, T, k, E, S, c->status);
    const int n = T * k + S * T;
    bucket_scatter_kernel<<<(n + 255) / 256, 256, 0, s>>>(c->r, T, k, E, S);
    return cudaGetLastError();
  }
  const size_t smem = bucket_smem_bytes(T, k, E);
  if (smem <= kBucketSmemMax)
    bucket_kernel<true><<<1, kBucketThreads, smem, s>>>(c->r, T, k, E, S, c->status);
  else
    bucket_kernel<false><<<1, kBucketThreads, 0, s>>>(c->r, T, k, E, S, c->status);
  return cudaGetLastError();
}

}  // namespace nvmoe
