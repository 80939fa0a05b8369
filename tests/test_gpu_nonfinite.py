"""Non-finite activations on the GPU: they propagate to the outputs of their own token only,
and never raise a device error.

Decode keeps activations exact, so the rule is the oracle's: a NaN in x makes
every logit of that token NaN (ranked below every number, so the selection is
experts 0..k-1 in index order) and every output NaN; an infinite entry makes
the logits infinite (the selection follows the ranking rule) and the
combine weights NaN.  The other tokens of the batch are unaffected and match
the oracle.  Prefill quantises x to NVFP4, which has no NaN or infinity, so
there the only requirement is that the call completes without a device error.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import cpp
from tests import harness
from tests.test_gpu_decode import last_routing, route_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import nvfp4_expert_ffn_gemv_b300 as lib
    return lib


def _poison(xb, x):
    xb, x = xb.clone(), x.clone()
    xb[1, 3] = float("nan")
    x[1, 3] = float("nan")
    xb[3, 7] = float("inf")
    x[3, 7] = float("inf")
    return xb, x


def test_batched_decode_nonfinite_rows(lib):
    s = synth.TINY
    layer = harness.make_layer(lib, s, seed=0, router_seed=0, fmt=0, max_tokens=8)
    try:
        xb, x = synth.tokens(s, 5, seed=61)
        xb, x = _poison(xb, x)
        xb = xb.cuda()
        x = x.numpy()
        idx, _, _, _ = route_gpu(lib, layer, xb, 5)
        ref = cpp.route(x, layer.router.cpu().numpy(), None, s.top_k)
        assert np.array_equal(idx, ref.idx)
        assert idx[1].tolist() == list(range(s.top_k))            # all-NaN logits: index order
        y = torch.empty((5, s.d_model), dtype=torch.bfloat16, device="cuda")
        lib.moe_forward_decode(layer.ctx, xb, 5, y)
        torch.cuda.synchronize()
        assert lib.moe_get_device_status(layer.ctx) == 0
        y = y.float().cpu().numpy()
        assert np.all(np.isnan(y[1])) and not np.any(np.isfinite(y[3]))
        good = [0, 2, 4]
        L = layer.oracle_weights(np.concatenate([idx[good].ravel(), np.arange(s.n_experts, s.n_all)]))
        r = cpp.moe_layer(L, x[good])
        harness.assert_close(torch.tensor(y[good]), r.y_bf16, "finite rows of a poisoned batch")
    finally:
        lib.moe_destroy(layer.ctx)


def test_batch1_decode_nan_token(lib):
    s = synth.FLINT
    layer = harness.make_layer(lib, s, seed=synth.layer_seed(2), router_seed=synth.router_seed(2), fmt=0,
                               max_tokens=1)
    try:
        xb, _ = synth.tokens(s, 1, seed=62)
        xb = xb.cuda()
        xb[0, 100] = float("nan")
        y = torch.empty((1, s.d_model), dtype=torch.bfloat16, device="cuda")
        lib.moe_forward_decode(layer.ctx, xb, 1, y)
        idx, _, _ = last_routing(lib, layer, 1)
        assert lib.moe_get_device_status(layer.ctx) == 0
        assert idx[0].tolist() == list(range(s.top_k))
        assert torch.isnan(y.float()).all()
    finally:
        lib.moe_destroy(layer.ctx)


def test_prefill_nonfinite_completes(lib):
    s = synth.MoEShape(d_model=256, n_experts=16, top_k=2, d_ff=256, n_shared=1)
    layer = harness.make_layer(lib, s, seed=3, router_seed=4, fmt=0, max_tokens=300)
    try:
        xb, x = synth.tokens(s, 300, seed=63)
        xb, _ = _poison(xb, x)
        y = torch.empty((300, s.d_model), dtype=torch.bfloat16, device="cuda")
        lib.moe_forward_prefill(layer.ctx, xb.cuda(), 300, y)
        torch.cuda.synchronize()
        assert lib.moe_get_device_status(layer.ctx) == 0
        yf = y.float()
        assert torch.isfinite(yf[0]).all() and torch.isfinite(yf[2]).all()
    finally:
        lib.moe_destroy(layer.ctx)
