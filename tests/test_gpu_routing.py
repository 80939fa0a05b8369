"""GPU routing against the C++ oracle: exact ties on every selection path, and full-size batches.

The rule under test (the reading of "6 of 256 experts per token" taken here):
the k largest fp32 logits, descending, equal logits to the lower expert index.
The GPU has five places that apply it:

  * the batch-1 decode chain (each experts / down CTA selects from the logits),
  * router_topk_kernel (moe_route and batched decode, few tokens),
  * router_topk_warp_kernel (1024 tokens and more),
  * the tensor-core router of prefill (from 256 tokens),
  * moe_route_noalloc.

Exact ties are made two ways whose logits are exact on both sides: a router
whose 256 columns are 64 distinct columns repeated four times (experts e,
e + 64, e + 128, e + 192 get bit-identical logits, since every path applies
the same operations to identical columns), and a zero router with an
integer-valued bias (logits equal the bias exactly).  On those inputs the GPU's
selection must equal the oracle's exactly.

Full size: all 4096 tokens of the prefill workload, and 32768 tokens, are
routed by moe_route and by prefill's tensor-core router and compared with the
oracle token by token (harness.check_routing), with per-expert counts exact.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import cpp
from tests import harness
from tests.test_gpu_decode import last_routing, route_gpu
from tests.test_gpu_prefill import check_prefill

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import nvfp4_expert_ffn_gemv_b300 as lib
    return lib


def _tie_router(s, kind):
    if kind == "repeated_columns":
        base = synth.router_weight(s, synth.router_seed(3))
        return base[:, torch.arange(s.n_experts) % 64].contiguous(), None
    g = torch.Generator().manual_seed(5)
    bias = torch.randint(0, 4, (s.n_experts,), generator=g).float()
    return torch.zeros((s.d_model, s.n_experts), dtype=torch.float32), bias


def _assert_exact(idx, logits, ref, what):
    assert np.array_equal(idx, ref.idx), f"{what}: selection differs from the oracle on exact ties"
    if logits is not None:
        assert np.array_equal(cpp.top_k(logits, idx.shape[1]), idx), f"{what}: not the top-k of its own logits"


@pytest.mark.parametrize("kind", ["repeated_columns", "zero_router_integer_bias"])
def test_exact_ties_every_selection_path(lib, kind):
    s = synth.FLINT
    router, bias = _tie_router(s, kind)
    layer = harness.make_layer(lib, s, seed=synth.layer_seed(9), router_seed=0, fmt=0, max_tokens=1024,
                               bias=bias, router=router)
    try:
        r_np = router.numpy()
        b_np = None if bias is None else bias.numpy()
        k = s.top_k
        xb, x = synth.tokens(s, 1024, seed=synth.token_seed(50))
        xb, x = xb.cuda(), x.numpy()
        if kind == "repeated_columns":
            # the repeated columns must give bit-identical logits on the GPU too
            _, _, _, lg = route_gpu(lib, layer, xb[:64], 64)
            assert np.array_equal(lg[:, :64], lg[:, 64:128]) and np.array_equal(lg[:, :64], lg[:, 192:])
        # batch-1 chain
        for t in range(3):
            y = torch.empty((1, s.d_model), dtype=torch.bfloat16, device="cuda")
            lib.moe_forward_decode(layer.ctx, xb[t:t + 1], 1, y)
            idx, _, lg = last_routing(lib, layer, 1)
            _assert_exact(idx, lg, cpp.route(x[t:t + 1], r_np, b_np, k), "batch-1 chain")
        # router_topk_kernel (64 tokens: many K chunks) and the warp kernel (1024 tokens)
        for T in (64, 1024):
            idx, _, counts, lg = route_gpu(lib, layer, xb[:T], T)
            ref = cpp.route(x[:T], r_np, b_np, k)
            _assert_exact(idx, lg, ref, f"moe_route T={T}")
            harness.check_counts(counts, idx, s.n_experts, ref)
        # tensor-core router of prefill
        y = torch.empty((512, s.d_model), dtype=torch.bfloat16, device="cuda")
        lib.moe_set_debug(layer.ctx, lib.MOE_DEBUG_KEEP_LOGITS)
        lib.moe_forward_prefill(layer.ctx, xb[:512], 512, y)
        idx, _, lg = last_routing(lib, layer, 512)
        _assert_exact(idx, lg, cpp.route(x[:512], r_np, b_np, k), "prefill tensor-core router")
        # the allocation-free router
        idx = torch.empty((64, k), dtype=torch.int32, device="cuda")
        w = torch.empty((64, k), dtype=torch.float32, device="cuda")
        lib.moe_route_noalloc(xb[:64], 64, layer.router, None if bias is None else bias.cuda(), s.d_model,
                              s.n_experts, k, idx, w)
        torch.cuda.synchronize()
        _assert_exact(idx.cpu().numpy(), None, cpp.route(x[:64], r_np, b_np, k), "moe_route_noalloc")
        assert lib.moe_get_device_status(layer.ctx) == 0
    finally:
        lib.moe_destroy(layer.ctx)


def _full_routing(lib, layer, xb, x, T):
    """moe_route and prefill's routing of all T tokens against the oracle."""
    s = layer.shape
    router = layer.router.cpu().numpy()
    ref = cpp.route(x, router, None, s.top_k)
    bound = harness.logit_error_bound(x, router)
    idx, w, counts, logits = route_gpu(lib, layer, xb, T)
    moved = harness.check_routing(idx, ref, logits, bound)
    harness.check_counts(counts, idx, s.n_experts, ref, moved)
    y = torch.empty((T, s.d_model), dtype=torch.bfloat16, device="cuda")
    lib.moe_forward_prefill(layer.ctx, xb, T, y)
    pidx, _, plogits = last_routing(lib, layer, T)
    pmoved = harness.check_routing(pidx, ref, plogits, bound)
    assert lib.moe_get_device_status(layer.ctx) == 0
    print(f"T={T}: {len(moved)} moe_route and {len(pmoved)} prefill tokens on near-ties")
    return moved, pmoved


def test_full_routing_flint_4096(lib):
    s = synth.FLINT
    layer = harness.make_layer(lib, s, seed=synth.layer_seed(0), router_seed=synth.router_seed(0), fmt=0,
                               max_tokens=4096)
    try:
        xb, x = synth.tokens(s, 4096, seed=synth.token_seed(7))
        _full_routing(lib, layer, xb.cuda(), x.numpy(), 4096)
    finally:
        lib.moe_destroy(layer.ctx)


def test_prefill_flint_32768(lib):
    """32768 tokens (the tensor-bound prefill point): routing and counts of every token, h codes and y on
    sampled tokens."""
    s = synth.FLINT
    layer = harness.make_layer(lib, s, seed=synth.layer_seed(1), router_seed=synth.router_seed(1), fmt=0,
                               max_tokens=32768)
    try:
        T = 32768
        xb, x = synth.tokens(s, T, seed=synth.token_seed(8))
        xb, x = xb.cuda(), x.numpy()
        _full_routing(lib, layer, xb, x, T)
        sample = [0, 1, 4097, 16384, T - 1] + list(range(3000, T, 6007))
        check_prefill(lib, layer, xb, x, T, sample=sample)
    finally:
        lib.moe_destroy(layer.ctx)
