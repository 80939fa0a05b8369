// Plain C++ CPU oracle of the NVFP4 sparse mixture-of-experts FFN layer.
//
// TEST INFRASTRUCTURE ONLY.  This file exists to check the CUDA library and
// shares nothing with it: no header, no table, no helper.  Only the test
// suite, the smoke check and the benchmark's CPU-baseline / reference arm load
// it (through oracle/cpp.py).  The product path never calls it.
//
// What it computes, and where each step comes from:
//
//   * 256 routed experts per MoE layer, 6 chosen per token, one always-on
//     shared expert: "Recursive Flint 40B-A2.5B：まず速さを第一に考えて作られた
//     コーディングモデル" (OrcaRouter blog), section "このアーキテクチャはメモリ帯域
//     幅に関する主張である"; the 648news page "Recursiveのコードエージェント向けMoE
//     モデルFlintがGGUF版で公開された", section "398億パラメータのMoE構造と推奨設定".
//   * weights shipped in NVFP4: the OrcaRouter page, section
//     "量子化のレシピは最も転用しやすい部分です" (the format is named, not defined).
//
// The pages print no formula.  Readings taken (the plainest ones, identical to
// the numpy oracle next to this file):
//
//   NVFP4 value   = e2m1(code) * e4m3(block scale) * ts; E2M1 = sign, 2
//                   exponent bits (bias 1), 1 mantissa bit; E4M3 = OCP E4M3FN
//                   (bias 7, subnormals, no infinity, 0x7F / 0xFF are NaN);
//                   one scale per 16 consecutive elements along K, one fp32 ts
//                   per (expert, matrix); two codes per byte, even K index in
//                   the low nibble.
//   quantiser     ts = amax/2688; s = E4M3_rne_sat(amax16 / (6 ts));
//                   q = E2M1_rne_sat(v / (e4m3(s) ts)); each step one IEEE fp32
//                   operation; zero codes canonical (never -0); activations
//                   (prefill) use the block step with ts = 1.
//   router        l[t,e] = sum_k x[t,k] W_r[k,e] (+ bias[e]);
//                   the k largest logits, descending; equal logits (+0 equals
//                   -0) go to the lower expert index; NaN ranks below every
//                   number;
//                   w = softmax over the chosen k (the full softmax renormalised).
//   expert        y_e = W_down (silu(W_gate x) * W_up x), silu(z) = z/(1+e^-z).
//   combine       y = sum_j w_j y_{idx_j} + sum_s shared_s(x).
//   prefill       x and h are quantised to NVFP4 (ts = 1) before their products.
//   output layer  logits = W_head x with the 4-bit (NVFP4) head the OrcaRouter
//                 page describes (section "量子化のレシピは最も転用しやすい部分です").
//   dense layers  2 of the 49 layers are dense (section "このアーキテクチャは
//                 メモリ帯域幅に関する主張である"); read as one SwiGLU FFN of
//                 width d_ff in NVFP4, y = W_down (silu(W_gate x) * W_up x).
//
// Precision.  NVFP4 is dequantised to FP32 (e2m1*e4m3 is exact in fp32, the
// multiplication by ts rounds once) and every value the layer passes from
// step to step is an FP32 number: x, W, logits, the combine weights, g, u, h,
// each expert's output and y.  Inside each dot product the fp32 operands are
// multiplied and summed in FP64 in index order and the sum is rounded once to
// FP32, so every step's result is independent of any summation order a
// faster implementation might choose.  silu and the softmax are evaluated in
// FP64 and rounded to FP32.
//
// Threads.  Each output element is computed by exactly one thread with the
// same operations whatever the thread count, so results do not depend on it.
#include <stdint.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <functional>
#include <thread>
#include <vector>

// One NVFP4 weight stack in canonical layout: codes [n][rows][K/2],
// scales [n][rows][K/16], ts [n].
struct OrMatrix {
  const uint8_t* codes;
  const uint8_t* scales;
  const float* ts;
};

// One layer: experts 0..E-1 routed, E..E+S-1 shared; gate/up [n][f][d],
// down [n][d][f]; router [d][E] fp32; bias [E] fp32 or NULL.  The configuration
// of the task's tiny layer has bf16 weights: those come as dense fp32 arrays.
struct OrLayer {
  int d, E, k, f, S;
  const float* router;
  const float* bias;
  OrMatrix gate, up, down;
  // bf16-valued weights (the tiny configuration's format): fp32 arrays
  // gate/up [n][f][d], down [n][d][f]; when set they replace the NVFP4 stacks
  const float* dense_gate;
  const float* dense_up;
  const float* dense_down;
};

namespace {

// --------------------------------------------------------------------------
// minifloat definitions
// --------------------------------------------------------------------------
double e2m1_value(int code) {
  const int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
  const double mag = e == 0 ? 0.5 * m : std::ldexp(1.0 + 0.5 * m, e - 1);
  return s ? -mag : mag;
}

double e4m3_value(int code) {
  const int s = (code >> 7) & 1, e = (code >> 3) & 15, m = code & 7;
  if (e == 15 && m == 7) return std::nan("");
  const double mag = e == 0 ? std::ldexp(m / 8.0, -6) : std::ldexp(1.0 + m / 8.0, e - 7);
  return s ? -mag : mag;
}

struct Tables {
  double e2m1[16];
  double e4m3[256];
  Tables() {
    for (int c = 0; c < 16; ++c) e2m1[c] = e2m1_value(c);
    for (int c = 0; c < 256; ++c) e4m3[c] = e4m3_value(c);
  }
};
const Tables& tables() {
  static const Tables t;
  return t;
}

// Index of the grid point nearest to v >= 0 on a strictly increasing grid of
// n non-negative values; a value halfway between two points goes to the even
// index (the code whose mantissa LSB is 0); at or above the last point it
// saturates there.
int rne_on_grid(double v, const double* grid, int n) {
  if (!(v < grid[n - 1])) return n - 1;
  const int lo = int(std::upper_bound(grid, grid + n, v) - grid) - 1;   // grid[lo] <= v < grid[lo+1]
  const int hi = lo + 1;
  const double mid = 0.5 * (grid[lo] + grid[hi]);
  if (v > mid) return hi;
  if (v < mid) return lo;
  return (hi % 2 == 0) ? hi : lo;
}

// E4M3 code of a non-negative fp32 value (saturating at 448, code 0x7E).
int e4m3_encode(float v) { return rne_on_grid(v, tables().e4m3, 0x7F); }

// E2M1 code of an fp32 value (saturating at +-6); zero is never negative.
int e2m1_encode(float v) {
  const int mag = rne_on_grid(std::fabs((double)v), tables().e2m1, 8);
  return (v < 0.f && mag != 0) ? (mag | 8) : mag;
}

// --------------------------------------------------------------------------
// threads
// --------------------------------------------------------------------------
int thread_count(int requested) {
  if (requested > 0) return requested;
  const unsigned hc = std::thread::hardware_concurrency();
  return hc ? (int)hc : 1;
}

// fn(i) for i in [0, n), item i on thread i % nt.
void parallel_for(long n, int nthreads, const std::function<void(long)>& fn) {
  const int nt = (int)std::min<long>(thread_count(nthreads), std::max<long>(n, 1));
  if (nt <= 1) {
    for (long i = 0; i < n; ++i) fn(i);
    return;
  }
  std::vector<std::thread> pool;
  for (int p = 0; p < nt; ++p)
    pool.emplace_back([&, p] {
      for (long i = p; i < n; i += nt) fn(i);
    });
  for (auto& th : pool) th.join();
}

// --------------------------------------------------------------------------
// quantiser and dequantiser (one tensor of `rows` rows of K elements)
// --------------------------------------------------------------------------
void quantize_blocks(const float* w, int rows, int K, float ts, uint8_t* codes, uint8_t* scales) {
  const int nb = K / 16;
  if (ts == 0.f) {
    std::memset(codes, 0, (size_t)rows * K / 2);
    std::memset(scales, 0, (size_t)rows * nb);
    return;
  }
  const float six_ts = 6.0f * ts;
  for (int r = 0; r < rows; ++r) {
    for (int b = 0; b < nb; ++b) {
      const float* v = w + (size_t)r * K + 16 * b;
      float amax = 0.f;
      for (int i = 0; i < 16; ++i) amax = std::max(amax, std::fabs(v[i]));
      const int s = e4m3_encode(amax / six_ts);
      const float dq = (float)tables().e4m3[s] * ts;
      scales[(size_t)r * nb + b] = (uint8_t)s;
      for (int i = 0; i < 16; i += 2) {
        const int c0 = dq > 0.f ? e2m1_encode(v[i] / dq) : 0;
        const int c1 = dq > 0.f ? e2m1_encode(v[i + 1] / dq) : 0;
        codes[(size_t)r * (K / 2) + 8 * b + i / 2] = (uint8_t)(c0 | (c1 << 4));
      }
    }
  }
}

// fp32 values of an NVFP4 tensor: (e2m1 * e4m3) exactly, then * ts rounded once.
void dequantize(const uint8_t* codes, const uint8_t* scales, float ts, int rows, int K, float* out) {
  const Tables& tb = tables();
  for (int r = 0; r < rows; ++r)
    for (int k = 0; k < K; ++k) {
      const uint8_t byte = codes[(size_t)r * (K / 2) + k / 2];
      const int c = (k & 1) ? (byte >> 4) : (byte & 15);
      const float q = (float)(tb.e2m1[c] * tb.e4m3[scales[(size_t)r * (K / 16) + k / 16]]);
      out[(size_t)r * K + k] = q * ts;
    }
}

// sum_i a[i] * b[i * stride] in fp64, rounded to fp32
inline float dot(const float* a, const float* b, int n, size_t stride = 1) {
  double acc = 0.0;
  for (int i = 0; i < n; ++i) acc += (double)a[i] * (double)b[(size_t)i * stride];
  return (float)acc;
}

inline double silu(double z) { return z / (1.0 + std::exp(-z)); }

// logit a ranks before logit b (larger first; equal values, +0 and -0 included,
// go to the lower index; NaN below every number)
inline bool ranks_before(float la, int a, float lb, int b) {
  const bool na = la != la, nb = lb != lb;
  if (na != nb) return nb;
  if (!na && la != lb) return la > lb;
  return a < b;
}

// --------------------------------------------------------------------------
// experts
// --------------------------------------------------------------------------
// Dequantised fp32 weights of one expert.
struct ExpertF32 {
  int e = -1;
  std::vector<float> wg, wu, wd;
  void load(const OrLayer* L, int ex) {
    if (ex == e) return;
    const int d = L->d, f = L->f;
    wg.resize((size_t)f * d);
    wu.resize((size_t)f * d);
    wd.resize((size_t)d * f);
    if (L->dense_gate) {
      const size_t m = (size_t)f * d;
      std::copy(L->dense_gate + ex * m, L->dense_gate + (ex + 1) * m, wg.begin());
      std::copy(L->dense_up + ex * m, L->dense_up + (ex + 1) * m, wu.begin());
      std::copy(L->dense_down + ex * m, L->dense_down + (ex + 1) * m, wd.begin());
      e = ex;
      return;
    }
    dequantize(L->gate.codes + (size_t)ex * f * d / 2, L->gate.scales + (size_t)ex * f * d / 16, L->gate.ts[ex], f,
               d, wg.data());
    dequantize(L->up.codes + (size_t)ex * f * d / 2, L->up.scales + (size_t)ex * f * d / 16, L->up.ts[ex], f, d,
               wu.data());
    dequantize(L->down.codes + (size_t)ex * d * f / 2, L->down.scales + (size_t)ex * d * f / 16, L->down.ts[ex], d,
               f, wd.data());
    e = ex;
  }
};

// SwiGLU expert on one token row: h (fp32, before any activation
// quantisation) and y; prefill quantises x and h to NVFP4 (ts = 1) first.
void expert_row(const ExpertF32& W, int d, int f, const float* x, int prefill, float* h_out, float* y_out) {
  std::vector<float> xv(x, x + d), h(f), hq;
  std::vector<uint8_t> c(std::max(d, f) / 2), s(std::max(d, f) / 16);
  if (prefill) {
    quantize_blocks(xv.data(), 1, d, 1.0f, c.data(), s.data());
    dequantize(c.data(), s.data(), 1.0f, 1, d, xv.data());
  }
  for (int j = 0; j < f; ++j) {
    const float g = dot(W.wg.data() + (size_t)j * d, xv.data(), d);
    const float u = dot(W.wu.data() + (size_t)j * d, xv.data(), d);
    h[j] = (float)(silu((double)g) * (double)u);
  }
  if (h_out) std::copy(h.begin(), h.end(), h_out);
  hq = h;
  if (prefill) {
    quantize_blocks(h.data(), 1, f, 1.0f, c.data(), s.data());
    dequantize(c.data(), s.data(), 1.0f, 1, f, hq.data());
  }
  if (y_out)
    for (int r = 0; r < d; ++r) y_out[r] = dot(W.wd.data() + (size_t)r * f, hq.data(), f);
}

// A list of (expert, token row) pairs sorted by expert, cut into one
// contiguous run per thread; a thread dequantises an expert when its run
// reaches it.  Output i of the list goes to h_out / y_out row i.
void run_pairs(const OrLayer* L, const std::vector<std::pair<int, long>>& pairs, const float* x, int prefill,
               float* h_out, float* y_out, int nthreads) {
  const long n = (long)pairs.size();
  const int nt = (int)std::min<long>(thread_count(nthreads), std::max<long>(n, 1));
  parallel_for(nt, nt, [&](long p) {
    ExpertF32 W;
    for (long i = n * p / nt; i < n * (p + 1) / nt; ++i) {
      W.load(L, pairs[i].first);
      expert_row(W, L->d, L->f, x + (size_t)pairs[i].second * L->d, prefill,
                 h_out ? h_out + (size_t)i * L->f : nullptr, y_out ? y_out + (size_t)i * L->d : nullptr);
    }
  });
}

}  // namespace

extern "C" {

void or_tables(double* e2m1_out, double* e4m3_out) {
  std::memcpy(e2m1_out, tables().e2m1, sizeof(tables().e2m1));
  std::memcpy(e4m3_out, tables().e4m3, sizeof(tables().e4m3));
}

void or_e4m3_encode(const float* v, long n, uint8_t* out) {
  for (long i = 0; i < n; ++i) out[i] = (uint8_t)e4m3_encode(v[i]);
}

void or_e2m1_encode(const float* v, long n, uint8_t* out) {
  for (long i = 0; i < n; ++i) out[i] = (uint8_t)e2m1_encode(v[i]);
}

// Weight quantiser: n tensors w [n][rows][K] -> codes, scales, ts.
void or_quantize(const float* w, int n, int rows, int K, uint8_t* codes, uint8_t* scales, float* ts,
                 int nthreads) {
  const size_t per = (size_t)rows * K;
  for (int e = 0; e < n; ++e) {
    // amax over the tensor (a maximum does not depend on the order), then rows in parallel
    const float* we = w + e * per;
    const long nchunk = std::min<long>(rows, 256);
    std::vector<float> part(nchunk, 0.f);
    parallel_for(nchunk, nthreads, [&](long c) {
      const size_t r0 = (size_t)rows * c / nchunk, r1 = (size_t)rows * (c + 1) / nchunk;
      float m = 0.f;
      for (size_t i = r0 * K; i < r1 * K; ++i) m = std::max(m, std::fabs(we[i]));
      part[c] = m;
    });
    float amax = 0.f;
    for (long c = 0; c < nchunk; ++c) amax = std::max(amax, part[c]);
    ts[e] = amax / 2688.0f;
    parallel_for(rows, nthreads, [&](long r) {
      quantize_blocks(we + (size_t)r * K, 1, K, ts[e], codes + e * per / 2 + (size_t)r * K / 2,
                      scales + e * per / 16 + (size_t)r * K / 16);
    });
  }
}

// Activation quantiser (tensor scale 1): a [rows][K] -> codes, scales.
void or_quantize_act(const float* a, int rows, int K, uint8_t* codes, uint8_t* scales) {
  quantize_blocks(a, rows, K, 1.0f, codes, scales);
}

void or_dequantize(const uint8_t* codes, const uint8_t* scales, float ts, int rows, int K, float* out) {
  dequantize(codes, scales, ts, rows, K, out);
}

// bf16 value nearest to each fp32 value (ties to even), returned as fp32.
void or_bf16_rne(const float* in, long n, float* out) {
  for (long i = 0; i < n; ++i) {
    uint32_t u;
    std::memcpy(&u, in + i, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) {
      out[i] = in[i];   // NaN stays NaN
      continue;
    }
    u += 0x7FFFu + ((u >> 16) & 1u);
    u &= 0xFFFF0000u;
    std::memcpy(out + i, &u, 4);
  }
}

// logits [T][E] = x [T][d] . W_r [d][E] (+ bias)
void or_router_logits(const float* x, int T, int d, const float* wr, const float* bias, int E, float* logits,
                      int nthreads) {
  parallel_for((long)T * E, nthreads, [&](long i) {
    const long t = i / E, e = i % E;
    double acc = 0.0;
    for (int kk = 0; kk < d; ++kk) acc += (double)x[t * d + kk] * (double)wr[(size_t)kk * E + e];
    if (bias) acc += (double)bias[e];
    logits[i] = (float)acc;
  });
}

// idx [T][k]: the k best logits per token, in rank order.
void or_top_k(const float* logits, int T, int E, int k, int32_t* idx) {
  std::vector<int> order(E);
  for (int t = 0; t < T; ++t) {
    const float* l = logits + (size_t)t * E;
    for (int e = 0; e < E; ++e) order[e] = e;
    std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return ranks_before(l[a], a, l[b], b); });
    for (int j = 0; j < k; ++j) idx[(size_t)t * k + j] = order[j];
  }
}

// w [T][k] = exp(l_j - l_max) / sum over the chosen k (fp64, rounded to fp32)
void or_combine_weights(const float* logits, const int32_t* idx, int T, int E, int k, float* w) {
  for (int t = 0; t < T; ++t) {
    double m = -INFINITY, s = 0.0;
    std::vector<double> z(k);
    for (int j = 0; j < k; ++j) m = std::max(m, (double)logits[(size_t)t * E + idx[(size_t)t * k + j]]);
    for (int j = 0; j < k; ++j) {
      const double l = logits[(size_t)t * E + idx[(size_t)t * k + j]];
      z[j] = std::exp(l - m);
      s += z[j];
    }
    if (m != m) s = NAN;
    for (int j = 0; j < k; ++j) w[(size_t)t * k + j] = (float)(z[j] / s);
  }
}

// counts [E], offsets [E+1], perm [T*k]: slots t*k+j grouped by expert, token-major.
void or_bucket(const int32_t* idx, int T, int k, int E, int32_t* counts, int32_t* offsets, int32_t* perm) {
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (long s = 0; s < (long)T * k; ++s) counts[idx[s]]++;
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  std::vector<int32_t> fill(offsets, offsets + E);
  for (long s = 0; s < (long)T * k; ++s) perm[fill[idx[s]]++] = (int32_t)s;
}

// One expert on T token rows x [T][d]: h [T][f] (fp32 SwiGLU output before
// any activation quantisation) and y [T][d]; either output may be NULL.
void or_expert(const OrLayer* L, int e, const float* x, int T, int prefill, float* h_out, float* y_out,
               int nthreads) {
  std::vector<std::pair<int, long>> pairs;
  for (long t = 0; t < T; ++t) pairs.emplace_back(e, t);
  run_pairs(L, pairs, x, prefill, h_out, y_out, nthreads);
}

// The layer on T tokens.  force_idx (or NULL) replaces the selection; logits,
// idx, w, counts may be NULL.  y [T][d] fp32.
void or_moe_layer(const OrLayer* L, const float* x, int T, int prefill, const int32_t* force_idx, float* y,
                  float* logits_out, int32_t* idx_out, float* w_out, int32_t* counts_out, int nthreads) {
  const int d = L->d, E = L->E, k = L->k, S = L->S;
  std::vector<float> logits((size_t)T * E), w((size_t)T * k);
  std::vector<int32_t> idx((size_t)T * k);
  or_router_logits(x, T, d, L->router, L->bias, E, logits.data(), nthreads);
  if (force_idx)
    std::copy(force_idx, force_idx + (size_t)T * k, idx.begin());
  else
    or_top_k(logits.data(), T, E, k, idx.data());
  or_combine_weights(logits.data(), idx.data(), T, E, k, w.data());
  // (expert, token) pairs: routed choice j of token t is slot t*k + j, shared
  // expert s of token t is slot T*k + s*T + t
  std::vector<std::pair<int, long>> pairs;
  std::vector<long> slot_of;
  for (int e = 0; e < E + S; ++e) {
    if (e < E) {
      for (int t = 0; t < T; ++t)
        for (int j = 0; j < k; ++j)
          if (idx[(size_t)t * k + j] == e) {
            pairs.emplace_back(e, t);
            slot_of.push_back((long)t * k + j);
          }
    } else {
      for (int t = 0; t < T; ++t) {
        pairs.emplace_back(e, t);
        slot_of.push_back((long)T * k + (long)(e - E) * T + t);
      }
    }
  }
  std::vector<float> yp(pairs.size() * d), ys((size_t)T * (k + S) * d);
  run_pairs(L, pairs, x, prefill, nullptr, yp.data(), nthreads);
  for (size_t i = 0; i < pairs.size(); ++i)
    std::copy(yp.begin() + i * d, yp.begin() + (i + 1) * d, ys.begin() + (size_t)slot_of[i] * d);
  parallel_for(T, nthreads, [&](long t) {
    for (int r = 0; r < d; ++r) {
      double acc = 0.0;
      for (int j = 0; j < k; ++j) acc += (double)w[t * k + j] * (double)ys[(size_t)(t * k + j) * d + r];
      for (int s = 0; s < S; ++s) acc += (double)ys[(size_t)(T * k + s * T + t) * d + r];
      y[t * d + r] = (float)acc;
    }
  });
  if (logits_out) std::copy(logits.begin(), logits.end(), logits_out);
  if (idx_out) std::copy(idx.begin(), idx.end(), idx_out);
  if (w_out) std::copy(w.begin(), w.end(), w_out);
  if (counts_out) {
    std::vector<int32_t> offs(E + 1), perm((size_t)T * k);
    or_bucket(idx.data(), T, k, E, counts_out, offs.data(), perm.data());
  }
}

// Output layer: out [T][R] = x [T][K] . W^T for one NVFP4 matrix W [R][K].
void or_gemv(const uint8_t* codes, const uint8_t* scales, float ts, int R, int K, const float* x, int T, float* out,
             int nthreads) {
  parallel_for(R, nthreads, [&](long r) {
    std::vector<float> w(K);
    dequantize(codes + (size_t)r * K / 2, scales + (size_t)r * K / 16, ts, 1, K, w.data());
    for (int t = 0; t < T; ++t) out[(size_t)t * R + r] = dot(w.data(), x + (size_t)t * K, K);
  });
}

// Dense SwiGLU FFN (one NVFP4 expert of width f, weight 1): y [T][d] fp32.
void or_dense_ffn(OrMatrix gate, OrMatrix up, OrMatrix down, int d, int f, const float* x, int T, float* y,
                  int nthreads) {
  OrLayer L{};
  L.d = d;
  L.E = 1;
  L.k = 1;
  L.f = f;
  L.S = 0;
  L.gate = gate;
  L.up = up;
  L.down = down;
  std::vector<std::pair<int, long>> pairs;
  for (long t = 0; t < T; ++t) pairs.emplace_back(0, t);
  run_pairs(&L, pairs, x, 0, nullptr, y, nthreads);
}

}  // extern "C"
