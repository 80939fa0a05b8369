"""Seeded synthetic inputs for the NVFP4 sparse-MoE FFN layer.

This module is the only code shared by the CPU oracle (``oracle/``) and the
CUDA path (``nvfp4_expert_ffn_gemv_b300``).  It draws random numbers and
nothing else: no quantisation, no routing, no matrix arithmetic of the layer.
Everything the layer computes is done independently on each side.

Workload recipe (the model facts come from the Flint 40B-A2.5B pages: 256
routed experts, 6 chosen per token, one always-on shared expert, 47 MoE
layers; hidden size 2048 and expert width 512 are the stated assumptions):

* expert weights  W_gate, W_up [f, d] and W_down [d, f], fp32 ~ N(0, 0.02),
  later quantised to NVFP4 by whichever side consumes them;
* router weight   W_r [d, E] fp32 ~ N(0, 0.02);
* tokens          x [T, d] ~ N(0, 1), rounded to bf16 (returned as the bf16
  tensor and as its exact fp32 image);
* optional router bias for the skewed batched-decode workload: every expert
  gets a Zipf rank r_e (a seeded permutation of 1..E) and the bias
  -beta * s * ln(r_e) with s = 1.1, beta = 0.1.

* the output layer W_head [vocab, d] and the dense FFN layers (W_gate, W_up
  [d_ff, d], W_down [d, d_ff]), fp32 ~ N(0, 0.02) like the experts.  Their
  sizes are not on the pages; the readings: vocab 151,936 (the ~0.3B gap
  between ~2.5B active including the output head and the ~2.2B active body,
  at d = 2048) and d_ff 18,432 for each of the 2 dense layers (what the 39.8B
  total and the ~2.2B active body leave for them).

Seeds: weights of layer l use 1000 + l, the router of layer l uses 2000 + l,
tokens of step i use 3000 + i, dense layer l 5000 + l, the output layer 6000;
the tiny workload uses seed 0 throughout.

Generation uses ``torch.Generator`` on the requested device, so the same call
on the same device always gives the same numbers.  CPU and CUDA generators
give *different* streams: a consumer that needs the values on the host copies
the generated tensor, it never regenerates it on another device.
"""
from __future__ import annotations

import dataclasses
import math

import torch

__all__ = [
    "MoEShape", "TINY", "FLINT", "layer_seed", "router_seed", "token_seed",
    "expert_weights", "expert_weights_one", "router_weight", "zipf_bias", "tokens",
    "FLINT_VOCAB", "FLINT_DENSE_FF", "dense_seed", "head_seed", "dense_ffn_weights", "head_weight",
]


@dataclasses.dataclass(frozen=True)
class MoEShape:
    d_model: int
    n_experts: int
    top_k: int
    d_ff: int
    n_shared: int = 1

    @property
    def n_all(self) -> int:
        """Routed plus shared experts."""
        return self.n_experts + self.n_shared


#: tiny CPU-checkable layer: d=256, 16 experts top-2 + 1 shared, f=128
TINY = MoEShape(d_model=256, n_experts=16, top_k=2, d_ff=128, n_shared=1)
#: Flint-shaped layer: d=2048, 256 experts top-6 + 1 shared, f=512
FLINT = MoEShape(d_model=2048, n_experts=256, top_k=6, d_ff=512, n_shared=1)


#: output-layer rows and dense-FFN width (readings of the pages' parameter counts)
FLINT_VOCAB = 151_936
FLINT_DENSE_FF = 18_432


def dense_seed(layer: int) -> int:
    return 5000 + layer


def head_seed() -> int:
    return 6000


def layer_seed(layer: int) -> int:
    return 1000 + layer


def router_seed(layer: int) -> int:
    return 2000 + layer


def token_seed(step: int) -> int:
    return 3000 + step


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def expert_weights(shape: MoEShape, seed: int, device="cpu", std: float = 0.02,
                   n: int | None = None):
    """fp32 expert weights of one layer, routed experts first then shared.

    Returns (w_gate [n, f, d], w_up [n, f, d], w_down [n, d, f]) with
    n = shape.n_all unless given.  Drawn in that order from one generator.
    """
    n = shape.n_all if n is None else n
    g = _gen(seed, device)
    f, d = shape.d_ff, shape.d_model
    w_gate = torch.randn((n, f, d), generator=g, device=device, dtype=torch.float32).mul_(std)
    w_up = torch.randn((n, f, d), generator=g, device=device, dtype=torch.float32).mul_(std)
    w_down = torch.randn((n, d, f), generator=g, device=device, dtype=torch.float32).mul_(std)
    return w_gate, w_up, w_down


def expert_weights_one(shape: MoEShape, seed: int, expert: int, device="cpu",
                       std: float = 0.02):
    """fp32 weights of a single expert, drawn from its own generator.

    Used where a workload is too large to hold every layer's fp32 weights at
    once: expert e of a layer with seed s comes from seed s * 4096 + e.
    """
    g = _gen(seed * 4096 + expert, device)
    f, d = shape.d_ff, shape.d_model
    w_gate = torch.randn((f, d), generator=g, device=device, dtype=torch.float32).mul_(std)
    w_up = torch.randn((f, d), generator=g, device=device, dtype=torch.float32).mul_(std)
    w_down = torch.randn((d, f), generator=g, device=device, dtype=torch.float32).mul_(std)
    return w_gate, w_up, w_down


def dense_ffn_weights(d_model: int, d_ff: int, seed: int, device="cpu", std: float = 0.02):
    """fp32 (W_gate [d_ff, d], W_up [d_ff, d], W_down [d, d_ff]) of one dense layer, in that order."""
    g = _gen(seed, device)
    w_gate = torch.randn((d_ff, d_model), generator=g, device=device, dtype=torch.float32).mul_(std)
    w_up = torch.randn((d_ff, d_model), generator=g, device=device, dtype=torch.float32).mul_(std)
    w_down = torch.randn((d_model, d_ff), generator=g, device=device, dtype=torch.float32).mul_(std)
    return w_gate, w_up, w_down


def head_weight(vocab: int, d_model: int, seed: int, device="cpu", std: float = 0.02):
    """fp32 output-layer weight [vocab, d]."""
    g = _gen(seed, device)
    return torch.randn((vocab, d_model), generator=g, device=device, dtype=torch.float32).mul_(std)


def router_weight(shape: MoEShape, seed: int, device="cpu", std: float = 0.02):
    """fp32 router weight [d, E] (row-major, the d index outer)."""
    g = _gen(seed, device)
    return torch.randn((shape.d_model, shape.n_experts), generator=g, device=device,
                       dtype=torch.float32).mul_(std)


def zipf_bias(shape: MoEShape, seed: int, s: float = 1.1, beta: float = 0.1):
    """Per-expert additive router bias from a seeded Zipf(s) rank (fp32 [E], CPU)."""
    g = _gen(seed, "cpu")
    ranks = torch.randperm(shape.n_experts, generator=g) + 1  # rank of expert e
    bias = [-beta * s * math.log(float(r)) for r in ranks.tolist()]
    return torch.tensor(bias, dtype=torch.float32)


def tokens(shape: MoEShape, n_tokens: int, seed: int, device="cpu"):
    """Activations x [T, d] ~ N(0, 1) as bf16; also returns their exact fp32 image."""
    g = _gen(seed, device)
    x = torch.randn((n_tokens, shape.d_model), generator=g, device=device, dtype=torch.float32)
    xb = x.to(torch.bfloat16)
    return xb, xb.float()
