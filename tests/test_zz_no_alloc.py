"""moe_route_noalloc: the context-free router whose scratch is a fixed device array.

It runs the same kernels, in the same summation order, as moe_route, so on the
same inputs its expert indices and combine weights must equal moe_route's bit
for bit -- on every one of several calls in a row, since the fixed scratch is
reused by each call without being cleared.  This file is collected last so
that it also runs after every other GPU test in the same process.
"""
import pytest
import torch

import synth
from tests import harness

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import nvfp4_expert_ffn_gemv_b300 as lib
    return lib


def _route_ctx(lib, layer, xb, T):
    k = layer.shape.top_k
    idx = torch.full((T, k), -1, dtype=torch.int32, device="cuda")
    w = torch.full((T, k), -1.0, dtype=torch.float32, device="cuda")
    lib.moe_route(layer.ctx, xb, T, idx, w)
    return idx, w


def _route_static(lib, layer, xb, T):
    s = layer.shape
    idx = torch.full((T, s.top_k), -1, dtype=torch.int32, device="cuda")
    w = torch.full((T, s.top_k), -1.0, dtype=torch.float32, device="cuda")
    bias = None if layer.bias is None else layer.bias.cuda()
    lib.moe_route_noalloc(xb, T, layer.router, bias, s.d_model, s.n_experts, s.top_k, idx, w)
    return idx, w


WIDE = synth.MoEShape(d_model=4096, n_experts=64, top_k=4, d_ff=128, n_shared=1)


@pytest.mark.parametrize("shape_name,T_list", [("tiny", [4, 1, 37]), ("flint", [1, 64, 4096, 3]),
                                               ("wide", [1, 16, 300])])
def test_noalloc_matches_route(lib, shape_name, T_list):
    shape = {"tiny": synth.TINY, "flint": synth.FLINT, "wide": WIDE}[shape_name]
    bias = synth.zipf_bias(shape, seed=77) if shape_name == "flint" else None
    layer = harness.make_layer(lib, shape, seed=5, router_seed=6, fmt=0, max_tokens=max(T_list), bias=bias)
    try:
        for T in T_list:
            xb, _ = synth.tokens(shape, T, seed=900 + T)
            xb = xb.cuda()
            ref = _route_ctx(lib, layer, xb, T)
            first = _route_static(lib, layer, xb, T)
            second = _route_static(lib, layer, xb, T)   # reuses the scratch the first call left
            torch.cuda.synchronize()
            for got in (first, second):
                assert torch.equal(got[0], ref[0]), f"T={T}: expert indices differ from moe_route"
                assert torch.equal(got[1].view(torch.int32), ref[1].view(torch.int32)), \
                    f"T={T}: combine weights differ from moe_route"
        assert lib.moe_get_device_status(layer.ctx) == 0
    finally:
        lib.moe_destroy(layer.ctx)


def test_noalloc_rejects_what_does_not_fit(lib):
    s = synth.FLINT
    router = torch.zeros((s.d_model, s.n_experts), dtype=torch.float32, device="cuda")
    idx = torch.empty((4097, s.top_k), dtype=torch.int32, device="cuda")
    w = torch.empty((4097, s.top_k), dtype=torch.float32, device="cuda")
    x = torch.zeros((4097, s.d_model), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(lib.MoEError) as e:
        lib.moe_route_noalloc(x, 4097, router, None, s.d_model, s.n_experts, s.top_k, idx, w)
    assert lib.STATUS_NAMES[e.value.status] == "MOE_ERR_UNSUPPORTED"
    for bad_d in (300, 8192):
        with pytest.raises(lib.MoEError) as e:
            lib.moe_route_noalloc(x, 4, router, None, bad_d, s.n_experts, s.top_k, idx, w)
        assert lib.STATUS_NAMES[e.value.status] == "MOE_ERR_INVALID_ARG"
    with pytest.raises(lib.MoEError) as e:
        lib.moe_route_noalloc(x, 4, router, None, s.d_model, s.n_experts, s.top_k, None, w)
    assert lib.STATUS_NAMES[e.value.status] == "MOE_ERR_INVALID_ARG"
    with pytest.raises(lib.MoEError) as e:   # host (pageable) bias: refused before any launch
        lib.moe_route_noalloc(x, 4, router, torch.zeros(s.n_experts), s.d_model, s.n_experts, s.top_k, idx, w)
    assert lib.STATUS_NAMES[e.value.status] == "MOE_ERR_INVALID_ARG"
    lib.moe_route_noalloc(x, 0, router, None, s.d_model, s.n_experts, s.top_k, idx, w)   # T = 0: no work
