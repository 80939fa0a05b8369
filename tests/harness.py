"""Test-side glue: build the same seeded layer for the CUDA library and for the oracle.

Both sides start from the same fp32 weights drawn by ``synth``; each side
quantises them with its own quantiser (the library's kernel, the oracle's
numpy code), so nothing the oracle sees comes from the CUDA path.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

import synth
from oracle import moe as omoe
from oracle import nvfp4 as onv

#: parity bar on bf16 outputs: relative L2 and max-abs relative to the output RMS
REL_L2_TOL = 1e-3
MAX_ABS_RMS_TOL = 2e-2


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

    def oracle_weights(self, experts) -> omoe.LayerWeights:
        """Oracle view of this layer: NVFP4 via the oracle quantiser (chosen experts only),
        or bf16-rounded dense weights for the bf16 format."""
        sel = sorted(set(int(e) for e in experts))
        router = self.router.cpu().numpy()
        bias = None if self.bias is None else self.bias.cpu().numpy()
        n = self.w_gate.shape[0]
        if self.fmt == 1:
            bf = lambda t: t.to(torch.bfloat16).double().cpu().numpy()  # noqa: E731
            return omoe.LayerWeights(router=router, bias=bias, dense_gate=bf(self.w_gate),
                                     dense_up=bf(self.w_up), dense_down=bf(self.w_down))
        f, d = self.shape.d_ff, self.shape.d_model
        wg = np.zeros((n, f, d), np.float32)
        wu = np.zeros((n, f, d), np.float32)
        wd = np.zeros((n, d, f), np.float32)
        for e in sel:
            wg[e] = self.w_gate[e].cpu().numpy()
            wu[e] = self.w_up[e].cpu().numpy()
            wd[e] = self.w_down[e].cpu().numpy()
        return omoe.quantize_layer(wg, wu, wd, router, bias, experts=sel)


def make_layer(lib, shape: synth.MoEShape, seed: int, router_seed: int, fmt: int = 0,
               max_tokens: int = 64, bias: torch.Tensor | None = None, device: str = "cuda",
               gen_device: str | None = None) -> GpuLayer:
    gen_device = gen_device or device
    wg, wu, wd = (t.to(device) for t in synth.expert_weights(shape, seed, device=gen_device))
    router = synth.router_weight(shape, router_seed, device=gen_device).to(device)
    E, S = shape.n_experts, shape.n_shared
    cfg = dict(d_model=shape.d_model, n_experts=E, top_k=shape.top_k, d_ff=shape.d_ff, n_shared=S,
               d_ff_shared=shape.d_ff, max_tokens=max_tokens, weight_format=fmt)
    weights = {"router": router.contiguous(),
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
    return GpuLayer(ctx, shape, wg, wu, wd, router, bias, fmt, codes)


def compare(y_gpu_bf16: torch.Tensor, y_ref_bf16: np.ndarray):
    """(relative L2 error, max-abs error / RMS of the reference) of bf16 outputs."""
    g = y_gpu_bf16.float().cpu().double().numpy()
    r = np.asarray(y_ref_bf16, np.float64)
    rms = np.sqrt(np.mean(r * r))
    rel = np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-300)
    mx = np.max(np.abs(g - r)) / max(rms, 1e-300)
    return float(rel), float(mx)


def assert_close(y_gpu_bf16, y_ref_bf16, what=""):
    rel, mx = compare(y_gpu_bf16, y_ref_bf16)
    assert rel <= REL_L2_TOL and mx <= MAX_ABS_RMS_TOL, f"{what}: rel_l2={rel:.3e} max_abs/rms={mx:.3e}"
    return rel, mx


def check_routing(idx_gpu: np.ndarray, ref: omoe.LayerResult):
    """idx must match exactly except on tokens the oracle flags as near-ties."""
    bad = [t for t in range(idx_gpu.shape[0])
           if not np.array_equal(idx_gpu[t], ref.idx[t]) and not ref.near_tie[t]]
    assert not bad, f"expert indices differ on tokens {bad[:8]}"
    return [t for t in range(idx_gpu.shape[0]) if not np.array_equal(idx_gpu[t], ref.idx[t])]
