"""The MoE FFN layer, step by step, in fp64 (oracle side).

Steps and where they come from:

* router scores over the routed experts, top-6 selection, always-on shared
  expert -- "Recursive Flint 40B-A2.5B：まず速さを第一に考えて作られたコーディング
  モデル" (OrcaRouter blog), section "このアーキテクチャはメモリ帯域幅に関する主張
  である", sparsity bullet; "Recursiveのコードエージェント向けMoEモデルFlintが
  GGUF版で公開された" (648news), section "398億パラメータのMoE構造と推奨設定".
* the pages do not give the router function, the expert MLP or the combine.
  Readings taken: fp32 logits l = x W_r (+ bias); the k largest logits win,
  ties to the lower expert index; weights are the softmax over all experts
  renormalised over the chosen k, which equals the softmax over the chosen
  k alone; experts are SwiGLU without biases, y_e = W_down (silu(W_gate x) *
  W_up x); the shared expert adds with weight 1; y = sum_j w_j y_{e_j} + y_sh.
* decode keeps activations exact (bf16 input, fp64 here).  Prefill feeds the
  block-scaled FP4 product, so x and h are quantised to NVFP4 (tensor scale 1)
  before their matrix products; h is rounded to fp32 before its quantisation,
  the precision in which the GPU takes the same decision.
"""
from __future__ import annotations

import dataclasses

import numpy as np

from . import nvfp4

F32 = np.float32


# --------------------------------------------------------------------------
# weights
# --------------------------------------------------------------------------
@dataclasses.dataclass
class NVFP4Tensor:
    codes: np.ndarray    # uint8 [n, rows, K/2]
    scales: np.ndarray   # uint8 [n, rows, K/16]
    ts: np.ndarray       # fp32  [n]

    def dense(self, e: int) -> np.ndarray:
        """fp64 [rows, K] real values of expert e."""
        return nvfp4.dequantize(self.codes[e], self.scales[e], self.ts[e])


@dataclasses.dataclass
class LayerWeights:
    """One MoE layer.  Experts 0..E-1 are routed, E..E+S-1 are shared.

    Either NVFP4 tensors (gate, up, down) or bf16-valued fp64 dense arrays.
    """
    router: np.ndarray                   # fp32 [d, E]
    bias: np.ndarray | None              # fp32 [E] or None
    gate: NVFP4Tensor | None = None      # [n, f, d]
    up: NVFP4Tensor | None = None        # [n, f, d]
    down: NVFP4Tensor | None = None      # [n, d, f]
    dense_gate: np.ndarray | None = None  # fp64 [n, f, d]   (bf16 weight format)
    dense_up: np.ndarray | None = None
    dense_down: np.ndarray | None = None  # fp64 [n, d, f]

    @property
    def n_experts(self) -> int:
        return self.router.shape[1]

    def expert(self, e: int):
        if self.gate is not None:
            return self.gate.dense(e), self.up.dense(e), self.down.dense(e)
        return self.dense_gate[e], self.dense_up[e], self.dense_down[e]


def quantize_layer(w_gate, w_up, w_down, router, bias=None, experts=None) -> LayerWeights:
    """NVFP4-quantise fp32 expert weights [n, f, d] / [n, d, f] with the oracle quantiser.

    ``experts`` restricts the work to a subset (other experts are left zero):
    a full 257-expert layer takes a while on the CPU and the checks only need
    the experts that tokens actually chose.
    """
    n = w_gate.shape[0]
    sel = range(n) if experts is None else sorted(set(int(e) for e in experts))

    def q(w):
        n_, rows, K = w.shape
        codes = np.zeros((n_, rows, K // 2), np.uint8)
        scales = np.zeros((n_, rows, K // 16), np.uint8)
        ts = np.zeros((n_,), F32)
        for e in sel:
            codes[e], scales[e], ts[e] = nvfp4.quantize(np.asarray(w[e], dtype=F32))
        return NVFP4Tensor(codes, scales, ts)

    return LayerWeights(router=np.asarray(router, F32),
                        bias=None if bias is None else np.asarray(bias, F32),
                        gate=q(w_gate), up=q(w_up), down=q(w_down))


# --------------------------------------------------------------------------
# router
# --------------------------------------------------------------------------
def router_logits(x: np.ndarray, router: np.ndarray, bias=None) -> np.ndarray:
    """l[t, e] = sum_k x[t, k] W_r[k, e] (+ bias_e), accumulated in fp64, stored fp32."""
    l = np.asarray(x, np.float64) @ np.asarray(router, np.float64)
    if bias is not None:
        l = l + np.asarray(bias, np.float64)[None, :]
    return l.astype(F32)


def _rank_key(value: float, e: int):
    """Sort key of expert e's logit: larger values first, equal values (+0 and -0
    included) to the lower index, NaN after every number."""
    if value != value:
        return (1, 0.0, e)
    return (0, -value, e)


def top_k(logits: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest logits per row, descending; ties to the lower index; NaN last."""
    logits = np.asarray(logits, F32)
    T, E = logits.shape
    out = np.empty((T, k), np.int32)
    for t in range(T):
        order = sorted(range(E), key=lambda e: _rank_key(float(logits[t, e]), e))
        out[t] = order[:k]
    return out


def combine_weights(logits: np.ndarray, idx: np.ndarray) -> np.ndarray:
    """w[t, j] = exp(l_j - l_max) / sum_i exp(l_i - l_max) over the chosen k (fp64)."""
    sel = np.take_along_axis(np.asarray(logits, np.float64), idx.astype(np.int64), axis=1)
    z = np.exp(sel - sel.max(axis=1, keepdims=True))
    return z / z.sum(axis=1, keepdims=True)


def near_ties(logits: np.ndarray, k: int, gap: float = 1e-6) -> np.ndarray:
    """Per token: True where two adjacent logits among the top k+1 differ by < gap.

    On such a token another selection (or order) is equally valid.
    """
    s = -np.sort(-np.asarray(logits, np.float64), axis=1)[:, : k + 1]
    return np.any(np.abs(np.diff(s, axis=1)) < gap, axis=1)


# --------------------------------------------------------------------------
# bucketing
# --------------------------------------------------------------------------
def bucket(idx: np.ndarray, n_experts: int):
    """counts[e], exclusive offsets[E+1] and perm: (t*k + j) grouped by expert, token-major."""
    T, k = idx.shape
    counts = np.zeros(n_experts, np.int32)
    for t in range(T):
        for j in range(k):
            counts[idx[t, j]] += 1
    offsets = np.zeros(n_experts + 1, np.int32)
    offsets[1:] = np.cumsum(counts)
    perm = np.empty(T * k, np.int32)
    fill = offsets[:-1].copy()
    for t in range(T):
        for j in range(k):
            e = idx[t, j]
            perm[fill[e]] = t * k + j
            fill[e] += 1
    return counts, offsets, perm


# --------------------------------------------------------------------------
# experts
# --------------------------------------------------------------------------
def silu(z):
    z = np.asarray(z, np.float64)
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def swiglu_expert(wg, wu, wd, x: np.ndarray, quant_act: bool = False) -> np.ndarray:
    """y = W_down (silu(W_gate x) * W_up x) for rows of x [T, d]; fp64 [T, d].

    With ``quant_act`` x and h go through the NVFP4 activation quantiser
    (tensor scale 1) before their products, as the FP4 x FP4 prefill does.
    """
    x = np.asarray(x, np.float64)
    if quant_act:
        c, s = nvfp4.quantize_activation(x.astype(F32))
        x = nvfp4.dequantize(c, s, 1.0)
    g = x @ np.asarray(wg, np.float64).T
    u = x @ np.asarray(wu, np.float64).T
    h = silu(g) * u
    if quant_act:
        c, s = nvfp4.quantize_activation(h.astype(F32))
        h = nvfp4.dequantize(c, s, 1.0)
    return h @ np.asarray(wd, np.float64).T


def expert_hidden(wg, wu, x: np.ndarray, quant_act: bool = False) -> np.ndarray:
    """h = silu(W_gate x) * W_up x (fp64 [T, f]); x quantised first when ``quant_act``."""
    x = np.asarray(x, np.float64)
    if quant_act:
        c, s = nvfp4.quantize_activation(x.astype(F32))
        x = nvfp4.dequantize(c, s, 1.0)
    return silu(x @ np.asarray(wg, np.float64).T) * (x @ np.asarray(wu, np.float64).T)


# --------------------------------------------------------------------------
# the layer
# --------------------------------------------------------------------------
@dataclasses.dataclass
class LayerResult:
    y: np.ndarray          # fp64 [T, d]
    y_bf16: np.ndarray     # fp64 [T, d], values rounded to bf16
    logits: np.ndarray     # fp32 [T, E]
    idx: np.ndarray        # int32 [T, k]
    w: np.ndarray          # fp64 [T, k]
    counts: np.ndarray     # int32 [E]
    near_tie: np.ndarray   # bool [T]


def moe_layer(lw: LayerWeights, x: np.ndarray, k: int, n_shared: int = 1,
              prefill: bool = False, force_idx: np.ndarray | None = None) -> LayerResult:
    """y[t] = sum_j w[t, j] * expert_{idx[t, j]}(x_t) + sum_s shared_s(x_t).

    ``force_idx`` replaces the selection (used where a near-tie makes another
    choice equally valid); everything else is recomputed from it.
    """
    x = np.asarray(x, np.float64)
    T, d = x.shape
    E = lw.n_experts
    logits = router_logits(x, lw.router, lw.bias)
    idx = top_k(logits, k) if force_idx is None else np.asarray(force_idx, np.int32)
    w = combine_weights(logits, idx)
    counts, _, _ = bucket(idx, E)
    y = np.zeros((T, d), np.float64)
    for e in np.unique(idx):
        rows, slots = np.nonzero(idx == e)
        wg, wu, wd = lw.expert(int(e))
        ye = swiglu_expert(wg, wu, wd, x[rows], quant_act=prefill)
        y[rows] += w[rows, slots][:, None] * ye
    for s in range(n_shared):
        wg, wu, wd = lw.expert(E + s)
        y += swiglu_expert(wg, wu, wd, x, quant_act=prefill)
    return LayerResult(y=y, y_bf16=nvfp4.bf16_rne(y), logits=logits, idx=idx, w=w,
                       counts=counts, near_tie=near_ties(logits, k))


def residual(x: np.ndarray, y: np.ndarray) -> np.ndarray:
    """Next layer input of the stack: bf16_rne(x + y)."""
    return nvfp4.bf16_rne(np.asarray(x, np.float64) + np.asarray(y, np.float64))


def moe_stack(layers, x: np.ndarray, k: int, n_shared: int = 1):
    """Chain of MoE layers with the residual add between them (attention omitted)."""
    results = []
    for lw in layers:
        r = moe_layer(lw, x, k, n_shared)
        results.append(r)
        x = residual(x, r.y)
    return x, results
