"""Failure detection on the GPU, without faulting, trapping or hanging it.

* A bounded wait that runs out: moe_debug_wait_selftest waits on an mbarrier
  that nothing arrives on and nothing copies to; the wait gives up after a
  few thousand polls, MOE_ERR_TIMEOUT is latched, moe_get_device_status reports
  it once and clears it, and the context keeps working (bit-identical output
  before and after).
* The plumbing from a product kernel's wait to the status word:
  MOE_DEBUG_FORCE_TIMEOUT makes the batch-1 decode kernels, the prefill GEMMs
  and the tensor-core router report a timeout after their real waits have
  completed (no copy or MMA is left in flight); the status is reported once,
  and the output is the same as without the flag (bit for bit on the batch-1
  path; prefill adds a token's expert contributions in arrival order, so
  there it agrees to rounding).  Batched decode (T >= 2)
  has no device-side waits.
* Allocation failure: moe_debug_fail_alloc makes the n-th device allocation
  of the library fail -- the arena of moe_init, or (n = 2 on a batch-1
  layer) the temporary buffer of the weight repacking, after the arena has
  been filled; moe_init returns MOE_ERR_OOM, leaves device memory as it found
  it, and the next moe_init succeeds.
"""
import pytest
import torch

import synth
from tests import harness

pytestmark = pytest.mark.gpu

TIMEOUT = 5


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import nvfp4_expert_ffn_gemv_b300 as lib
    return lib


def _decode(lib, layer, xb, T):
    y = torch.empty((T, layer.shape.d_model), dtype=torch.bfloat16, device="cuda")
    lib.moe_forward_decode(layer.ctx, xb, T, y)
    return y


def _prefill(lib, layer, xb, T):
    y = torch.empty((T, layer.shape.d_model), dtype=torch.bfloat16, device="cuda")
    lib.moe_forward_prefill(layer.ctx, xb, T, y)
    return y


def test_bounded_wait_runs_out_and_context_survives(lib):
    s = synth.TINY
    layer = harness.make_layer(lib, s, seed=0, router_seed=0, fmt=0, max_tokens=8)
    try:
        xb, _ = synth.tokens(s, 4, seed=71)
        xb = xb.cuda()
        before = _decode(lib, layer, xb, 4)
        assert lib.moe_get_device_status(layer.ctx) == 0
        lib.moe_debug_wait_selftest(layer.ctx, 4096)
        assert lib.moe_get_device_status(layer.ctx) == TIMEOUT
        assert lib.moe_get_device_status(layer.ctx) == 0              # reported once, then cleared
        after = _decode(lib, layer, xb, 4)
        assert lib.moe_get_device_status(layer.ctx) == 0
        assert torch.equal(before.view(torch.int16), after.view(torch.int16))
    finally:
        lib.moe_destroy(layer.ctx)


@pytest.mark.parametrize("path", ["batch1", "prefill"])
def test_forced_timeout_reaches_status_word(lib, path):
    if path == "batch1":
        s, T, run = synth.FLINT, 1, _decode
    else:
        s, T, run = synth.MoEShape(d_model=256, n_experts=16, top_k=2, d_ff=256, n_shared=1), 300, _prefill
    layer = harness.make_layer(lib, s, seed=synth.layer_seed(4), router_seed=synth.router_seed(4), fmt=0,
                               max_tokens=T)
    try:
        xb, _ = synth.tokens(s, T, seed=72)
        xb = xb.cuda()
        clean = run(lib, layer, xb, T)
        assert lib.moe_get_device_status(layer.ctx) == 0
        lib.moe_set_debug(layer.ctx, lib.MOE_DEBUG_FORCE_TIMEOUT)
        forced = run(lib, layer, xb, T)
        assert lib.moe_get_device_status(layer.ctx) == TIMEOUT
        assert lib.moe_get_device_status(layer.ctx) == 0
        lib.moe_set_debug(layer.ctx, 0)
        again = run(lib, layer, xb, T)
        assert lib.moe_get_device_status(layer.ctx) == 0
        if path == "batch1":     # fixed summation order: bit-identical
            assert torch.equal(clean.view(torch.int16), forced.view(torch.int16))
            assert torch.equal(clean.view(torch.int16), again.view(torch.int16))
        else:                    # prefill adds a token's contributions in arrival order
            for other in (forced, again):
                rel, mx = harness.compare(other, clean.float().cpu().numpy())
                assert rel <= 1e-4 and mx <= 1e-2, (rel, mx)
    finally:
        lib.moe_destroy(layer.ctx)


def test_allocation_failure_is_reported_and_leaks_nothing(lib):
    s = synth.TINY
    base = harness.make_layer(lib, s, seed=0, router_seed=0, fmt=0, max_tokens=8)   # its weights feed moe_init
    try:
        torch.cuda.synchronize()
        free0, _ = torch.cuda.mem_get_info()
        lib.moe_debug_fail_alloc(1)
        try:
            with pytest.raises(lib.MoEError) as e:
                lib.moe_init(base.cfg, base.weights)
            assert lib.STATUS_NAMES[e.value.status] == "MOE_ERR_OOM"
        finally:
            lib.moe_debug_fail_alloc(0)
        torch.cuda.synchronize()
        free1, _ = torch.cuda.mem_get_info()
        assert free1 == free0, (free0, free1)
        # the second allocation from now fails: one context is created, the next is refused
        lib.moe_debug_fail_alloc(2)
        try:
            ok = lib.moe_init(base.cfg, base.weights)
            with pytest.raises(lib.MoEError) as e:
                lib.moe_init(base.cfg, base.weights)
            assert lib.STATUS_NAMES[e.value.status] == "MOE_ERR_OOM"
        finally:
            lib.moe_debug_fail_alloc(0)
        lib.moe_destroy(ok)
        torch.cuda.synchronize()
        assert abs(torch.cuda.mem_get_info()[0] - free0) <= (2 << 20)   # the arena came back
        lib.moe_destroy(lib.moe_init(base.cfg, base.weights))   # allocation works again
    finally:
        lib.moe_destroy(base.ctx)


def test_allocation_failure_after_the_arena_frees_it(lib):
    s = synth.FLINT
    base = harness.make_layer(lib, s, seed=synth.layer_seed(5), router_seed=synth.router_seed(5), fmt=0,
                              max_tokens=1)
    try:
        torch.cuda.synchronize()
        free0, _ = torch.cuda.mem_get_info()
        lib.moe_debug_fail_alloc(2)      # 1: the arena (~0.5 GB), 2: the repacking buffer
        try:
            with pytest.raises(lib.MoEError) as e:
                lib.moe_init(base.cfg, base.weights)
            assert lib.STATUS_NAMES[e.value.status] == "MOE_ERR_OOM"
        finally:
            lib.moe_debug_fail_alloc(0)
        torch.cuda.synchronize()
        assert abs(torch.cuda.mem_get_info()[0] - free0) <= (2 << 20)
        lib.moe_destroy(lib.moe_init(base.cfg, base.weights))
    finally:
        lib.moe_destroy(base.ctx)
