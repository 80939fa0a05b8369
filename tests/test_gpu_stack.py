"""GPU parity of the layer stack: Flint-shaped layers chained with the residual add.

The chain runs as the 47-layer benchmark runs it: one token per call, batch-1
decode path, each layer's bf16 output (x + layer(x)) is the next layer's input,
all calls queued back to back on one stream (so the per-layer kernel chains
overlap through programmatic dependent launch).  Parity is checked layer by
layer along the GPU's own trajectory: the oracle gets the exact bf16 input the
GPU layer got and the experts it used, so a one-ulp difference at one layer
cannot turn into a different routing decision further down.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import cpp
from tests import harness

pytestmark = pytest.mark.gpu

N_LAYERS = 6
N_TOKENS = 3


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import nvfp4_expert_ffn_gemv_b300 as lib
    return lib


def test_stack_chain_layerwise(lib):
    s = synth.FLINT
    layers = [harness.make_layer(lib, s, seed=synth.layer_seed(l), router_seed=synth.router_seed(l), fmt=0,
                                 max_tokens=1) for l in range(N_LAYERS)]
    try:
        k = s.top_k
        for t in range(N_TOKENS):
            xb, _ = synth.tokens(s, 1, seed=synth.token_seed(100 + t))
            bufs = [xb.cuda()] + [torch.empty((1, s.d_model), dtype=torch.bfloat16, device="cuda")
                                  for _ in range(N_LAYERS)]
            idx = torch.empty((N_LAYERS, 1, k), dtype=torch.int32, device="cuda")
            w = torch.empty((N_LAYERS, 1, k), dtype=torch.float32, device="cuda")
            logits = torch.empty((N_LAYERS, 1, s.n_experts), dtype=torch.float32, device="cuda")
            for l, layer in enumerate(layers):
                lib.moe_forward_decode(layer.ctx, bufs[l], 1, bufs[l + 1], 1)
                lib.moe_debug_routing(layer.ctx, 1, idx[l], w[l])   # stream-ordered after this layer
                lib.moe_debug_logits(layer.ctx, 1, logits[l])
            torch.cuda.synchronize()
            for layer in layers:
                assert lib.moe_get_device_status(layer.ctx) == 0
            idx_h, lg_h = idx.cpu().numpy(), logits.cpu().numpy()
            for l, layer in enumerate(layers):
                x_l = bufs[l].float().cpu().numpy()              # the exact bf16 input of layer l
                used = np.concatenate([idx_h[l].ravel(), np.arange(s.n_experts, s.n_all)])
                L = layer.oracle_weights(used)
                ref = cpp.moe_layer(L, x_l)
                bound = harness.logit_error_bound(x_l, layer.router.cpu().numpy())
                if harness.check_routing(idx_h[l], ref, lg_h[l], bound):
                    L = layer.oracle_weights(np.concatenate([used, ref.idx.ravel()]))
                    ref = cpp.moe_layer(L, x_l, force_idx=idx_h[l])
                harness.assert_close(bufs[l + 1], cpp.residual(x_l, ref.y), f"token {t} layer {l}")
    finally:
        for layer in layers:
            lib.moe_destroy(layer.ctx)


N_LAYERS_BATCHED = 4
T_BATCHED = 16


def test_stack_chain_batched_layerwise(lib):
    """The batched-decode path chained the same way (16 tokens a call, 4 layers back to back on one
    stream): its kernels overlap across calls through programmatic dependent launch, so each
    layer's router may start while the previous layer's combine still runs.  Checked layer by layer
    against the oracle on the GPU's own inputs, as above."""
    s = synth.FLINT
    layers = [harness.make_layer(lib, s, seed=synth.layer_seed(10 + l), router_seed=synth.router_seed(10 + l),
                                 fmt=0, max_tokens=T_BATCHED) for l in range(N_LAYERS_BATCHED)]
    try:
        k, T = s.top_k, T_BATCHED
        xb, _ = synth.tokens(s, T, seed=synth.token_seed(200))
        bufs = [xb.cuda()] + [torch.empty((T, s.d_model), dtype=torch.bfloat16, device="cuda")
                              for _ in range(N_LAYERS_BATCHED)]
        for l, layer in enumerate(layers):
            lib.moe_forward_decode(layer.ctx, bufs[l], T, bufs[l + 1], 1)
        torch.cuda.synchronize()
        for layer in layers:
            assert lib.moe_get_device_status(layer.ctx) == 0
        for l, layer in enumerate(layers):
            x_l = bufs[l].float().cpu().numpy()
            idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
            lib.moe_route(layer.ctx, bufs[l], T, idx)        # the routing this layer's forward used
            torch.cuda.synchronize()
            idx_h = idx.cpu().numpy()
            used = np.concatenate([np.unique(idx_h.ravel()), np.arange(s.n_experts, s.n_all)])
            L = layer.oracle_weights(used)
            ref = cpp.moe_layer(L, x_l)
            if harness.check_routing(idx_h, ref):
                L = layer.oracle_weights(np.concatenate([used, ref.idx.ravel()]))
                ref = cpp.moe_layer(L, x_l, force_idx=idx_h)
            harness.assert_close(bufs[l + 1], cpp.residual(x_l, ref.y), f"batched layer {l}")
    finally:
        for layer in layers:
            lib.moe_destroy(layer.ctx)

