"""Test-side glue: build the same seeded layer for the CUDA library and for the oracle.

Both sides start from the same fp32 weights drawn by ``synth``; each side
quantises them with its own quantiser (the library's kernel, the C++ oracle's
code), so nothing the oracle sees comes from the CUDA path.  The reference for
every GPU parity test is the C++ oracle (``oracle/cpp.py``); the numpy oracle
is its cross-check on the CPU.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

import synth
from oracle import cpp

#: parity bar on bf16 outputs: relative L2 and max-abs relative to the output RMS
REL_L2_TOL = 1e-3
MAX_ABS_RMS_TOL = 2e-2
#: logit gap below which another selection is also correct whatever the arithmetic
NEAR_TIE = 1e-6
U32 = 2.0 ** -24


@dataclasses.dataclass
class GpuLayer:
    ctx: int
    shape: synth.MoEShape
    w_gate: torch.Tensor   # fp32 [n_all, f, d] on the device (kept for the oracle)
    w_up: torch.Tensor
    w_down: torch.Tensor
    router: torch.Tensor   # fp32 [d, E]
    bias: torch.Tensor | None
    fmt: int
    codes: dict            # the library's own quantisation (device tensors)
    cfg: dict = None       # the moe_init arguments, to create more contexts from the same weights
    weights: dict = None

    def oracle_weights(self, experts=None) -> cpp.Layer:
        """C++-oracle view of this layer: NVFP4 by the oracle's quantiser (only the listed
        experts, all when None), or the bf16-rounded dense weights for the bf16 format."""
        n = self.w_gate.shape[0]
        sel = list(range(n)) if experts is None else sorted(set(int(e) for e in experts))
        router = self.router.cpu().numpy()
        bias = None if self.bias is None else self.bias.cpu().numpy()
        s = self.shape
        if self.fmt == 1:
            bf = lambda t: t.to(torch.bfloat16).float().cpu().numpy()  # noqa: E731
            return cpp.Layer(router=router, bias=bias, gate=None, up=None, down=None, k=s.top_k, S=s.n_shared,
                             dense=(bf(self.w_gate), bf(self.w_up), bf(self.w_down)))
        f, d = s.d_ff, s.d_model
        wg = np.zeros((n, f, d), np.float32)
        wu = np.zeros((n, f, d), np.float32)
        wd = np.zeros((n, d, f), np.float32)
        idx = torch.tensor(sel, dtype=torch.long, device=self.w_gate.device)
        wg[sel] = self.w_gate[idx].cpu().numpy()
        wu[sel] = self.w_up[idx].cpu().numpy()
        wd[sel] = self.w_down[idx].cpu().numpy()
        return cpp.quantize_layer(wg, wu, wd, router, bias, k=s.top_k, S=s.n_shared, experts=sel)


def make_layer(lib, shape: synth.MoEShape, seed: int, router_seed: int, fmt: int = 0,
               max_tokens: int = 64, bias: torch.Tensor | None = None, device: str = "cuda",
               gen_device: str | None = None, router: torch.Tensor | None = None) -> GpuLayer:
    gen_device = gen_device or device
    wg, wu, wd = (t.to(device) for t in synth.expert_weights(shape, seed, device=gen_device))
    if router is None:
        router = synth.router_weight(shape, router_seed, device=gen_device)
    router = router.to(device).contiguous()
    E, S = shape.n_experts, shape.n_shared
    cfg = dict(d_model=shape.d_model, n_experts=E, top_k=shape.top_k, d_ff=shape.d_ff, n_shared=S,
               d_ff_shared=shape.d_ff, max_tokens=max_tokens, weight_format=fmt)
    weights = {"router": router,
               "router_bias": None if bias is None else bias.to(device).contiguous()}
    codes = {}
    if fmt == 0:
        for name, w in (("gate", wg), ("up", wu), ("down", wd)):
            c, s, ts = lib.quantize(w)
            codes[name] = (c, s, ts)
            weights[name] = dict(codes=c[:E], scales=s[:E], tensor_scale=ts[:E])
            weights["shared_" + name] = dict(codes=c[E:], scales=s[E:], tensor_scale=ts[E:])
    else:
        for name, w in (("gate", wg), ("up", wu), ("down", wd)):
            b = w.to(torch.bfloat16).contiguous()
            codes[name] = b
            weights[name] = dict(bf16=b[:E])
            weights["shared_" + name] = dict(bf16=b[E:])
    torch.cuda.synchronize()
    ctx = lib.moe_init(cfg, weights, device=torch.device(device).index or 0)
    return GpuLayer(ctx, shape, wg, wu, wd, router, bias, fmt, codes, cfg, weights)


def compare(y_gpu_bf16, y_ref_bf16):
    """(relative L2 error, max-abs error / RMS of the reference) of bf16 outputs."""
    g = torch.as_tensor(y_gpu_bf16).float().cpu().double().numpy()
    r = np.asarray(y_ref_bf16, np.float64)
    rms = np.sqrt(np.mean(r * r))
    rel = np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-300)
    mx = np.max(np.abs(g - r)) / max(rms, 1e-300)
    return float(rel), float(mx)


def assert_close(y_gpu_bf16, y_ref_bf16, what=""):
    rel, mx = compare(y_gpu_bf16, y_ref_bf16)
    assert rel <= REL_L2_TOL and mx <= MAX_ABS_RMS_TOL, f"{what}: rel_l2={rel:.3e} max_abs/rms={mx:.3e}"
    return rel, mx


def logit_error_bound(x: np.ndarray, router: np.ndarray, bias=None) -> np.ndarray:
    """A-priori bound on |fp32 logit - exact logit| for any order of fp32 additions.

    The GPU forms x[t] . W_r[:, e] with d products, each exact or rounded once
    (an FMA, or bf16 x bf16 splits summed by the tensor cores: at most 3 d
    terms), in any summation tree; Higham's bound for such a sum is
    gamma_n * sum |terms| with gamma_n = n u / (1 - n u), u = 2^-24, n = 3 d.
    Adding the bias and the final rounding add 2 u |l| more.
    """
    x = np.asarray(x, np.float64)
    a = np.abs(x) @ np.abs(np.asarray(router, np.float64))
    n = 3 * x.shape[1]
    gamma = n * U32 / (1 - n * U32)
    exact = x @ np.asarray(router, np.float64)
    if bias is not None:
        exact = exact + np.asarray(bias, np.float64)[None, :]
    return gamma * a + 2 * U32 * np.abs(exact) + 1e-30


def check_routing(idx_gpu: np.ndarray, ref: cpp.LayerResult, logits_gpu: np.ndarray | None = None,
                  bound: np.ndarray | None = None):
    """The GPU's expert indices against the oracle's.

    * With the GPU's logits: its selection must be exactly the top-k of those
      logits under the ranking rule (larger first, equal values to the lower
      expert, NaN last), and each logit must lie within ``bound`` of the
      oracle's (when given).
    * A token may differ from the oracle's selection only where the choice is
      ambiguous: at every position that differs, the oracle's logits of the
      two experts involved are within NEAR_TIE plus twice the largest
      GPU-vs-oracle logit difference seen on that token (0 without GPU logits).
    Returns the tokens that differ (logged by the callers, not failed).
    """
    k = idx_gpu.shape[1]
    if logits_gpu is not None:
        own = cpp.top_k(logits_gpu, k)
        bad = np.nonzero(np.any(own != idx_gpu, axis=1))[0]
        assert bad.size == 0, f"selection is not the top-k of the GPU's own logits on tokens {bad[:8].tolist()}"
        if bound is not None:
            fin = np.isfinite(ref.logits) & np.isfinite(logits_gpu)
            over = fin & (np.abs(logits_gpu.astype(np.float64) - ref.logits) > bound)
            assert not over.any(), f"GPU logits outside the fp32 error bound at {np.argwhere(over)[:4].tolist()}"
    moved = []
    for t in np.nonzero(np.any(idx_gpu != ref.idx, axis=1))[0]:
        delta = 0.0
        if logits_gpu is not None:
            ex = np.union1d(idx_gpu[t], ref.idx[t])
            delta = float(np.max(np.abs(logits_gpu[t, ex].astype(np.float64) - ref.logits[t, ex])))
        for j in np.nonzero(idx_gpu[t] != ref.idx[t])[0]:
            a, b = ref.logits[t, idx_gpu[t, j]], ref.logits[t, ref.idx[t, j]]
            gap = abs(float(a) - float(b))
            assert gap <= NEAR_TIE + 2 * delta, (f"token {t}, choice {j}: GPU expert {idx_gpu[t, j]} vs oracle "
                                                 f"{ref.idx[t, j]}, oracle logit gap {gap:.3e} > {NEAR_TIE + 2 * delta:.3e}")
        moved.append(int(t))
    return moved


def check_counts(counts_gpu: np.ndarray, idx_gpu: np.ndarray, n_experts: int, ref=None, moved=()):
    """Per-expert counts: exactly the histogram of the GPU's indices, and exactly the
    oracle's when no token's selection moved."""
    hist = np.bincount(idx_gpu.ravel(), minlength=n_experts)
    assert np.array_equal(counts_gpu, hist), "counts are not the histogram of the chosen experts"
    if ref is not None and not moved:
        assert np.array_equal(counts_gpu, ref.counts), "counts differ from the oracle's"
