"""GPU parity of the decode path against the oracle, through the C ABI.

Bar (element by element on the same seeded inputs): expert indices and
per-expert counts bit-exact (tokens the oracle flags as near-ties excepted);
bf16 outputs within relative L2 1e-3 and max-abs 2e-2 x RMS of the oracle's
bf16-rounded output.  Quantised codes bit-exact.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import moe as omoe
from oracle import nvfp4 as onv
from tests import harness

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import nvfp4_expert_ffn_gemv_b300 as lib
    return lib


def _special_weights():
    """fp32 values at and around E2M1 / E4M3 rounding midpoints of a known scale."""
    ts = 2.0 ** -12                        # amax = 2688 * ts makes ts exact
    d0 = 448 * ts
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 5.9, 6.0, 0.0, 1e-9])
    vals = np.concatenate([mids, -mids])
    w = np.zeros((4, 64, 64), np.float32)
    w[:, :, 0] = 6 * d0                      # every block's amax ... and the tensor amax
    for r in range(64):
        v = (vals[r % len(vals)] * d0 * (1 + (r // 22) * 2.0 ** -22))
        w[:, r, 1:16] = np.float32(v)
        w[:, r, 16:32] = np.float32(v / 7.3)   # non-power-of-two block scale
    w[2] = 0.0                               # an all-zero tensor
    w[3, :, 32:] = np.random.default_rng(0).standard_normal((64, 32)).astype(np.float32) * 1e-3
    return w


@pytest.mark.parametrize("kind", ["normal", "special", "wide"])
def test_quantizer_bit_exact(lib, kind):
    if kind == "normal":
        w = (torch.randn((5, 96, 512), generator=torch.Generator().manual_seed(1)) * 0.02).numpy()
    elif kind == "special":
        w = _special_weights()
    else:
        g = torch.Generator().manual_seed(2)
        w = (torch.randn((3, 32, 2048), generator=g) * torch.logspace(-6, 3, 2048)).numpy().astype(np.float32)
    c, s, ts = lib.quantize(torch.from_numpy(w).cuda())
    c, s, ts = c.cpu().numpy(), s.cpu().numpy(), ts.cpu().numpy()
    for e in range(w.shape[0]):
        rc, rs, rts = onv.quantize(w[e])
        assert ts[e] == rts, f"tensor scale of tensor {e}"
        assert np.array_equal(s[e], rs), f"block scales of tensor {e}"
        assert np.array_equal(c[e], rc), f"codes of tensor {e}"


def _run_decode(lib, layer, x_bf16, T, residual=0, per_token=False):
    d = layer.shape.d_model
    y = torch.empty((T, d), dtype=torch.bfloat16, device="cuda")
    if per_token:
        for t in range(T):
            lib.moe_forward_decode(layer.ctx, x_bf16[t:t + 1], 1, y[t:t + 1], residual)
    else:
        lib.moe_forward_decode(layer.ctx, x_bf16, T, y, residual)
    torch.cuda.synchronize()
    assert lib.moe_get_device_status(layer.ctx) == 0
    return y


def _route(lib, layer, x_bf16, T):
    k, E = layer.shape.top_k, layer.shape.n_experts
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    counts = torch.empty((E,), dtype=torch.int32, device="cuda")
    lib.moe_route(layer.ctx, x_bf16, T, idx, w, counts)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), w.cpu().numpy(), counts.cpu().numpy()


def _check_layer(lib, layer, xb, x, T, per_token=False, residual=0, prefix=""):
    idx, w, counts = _route(lib, layer, xb, T)
    lw = layer.oracle_weights(np.concatenate([idx.ravel(), np.arange(layer.shape.n_experts,
                                                                      layer.shape.n_all)]))
    ref = omoe.moe_layer(lw, x, layer.shape.top_k, layer.shape.n_shared)
    moved = harness.check_routing(idx, ref)
    if moved:  # a near-tie picked another valid set: recompute the oracle with it
        ref = omoe.moe_layer(lw, x, layer.shape.top_k, layer.shape.n_shared, force_idx=idx)
    assert np.array_equal(counts, ref.counts)
    assert np.allclose(w, ref.w, rtol=2e-6, atol=1e-7)
    y = _run_decode(lib, layer, xb, T, residual=residual, per_token=per_token)
    if not per_token:
        # the forward call may route with another kernel than moe_route (other fp32
        # summation order): it must agree except on the oracle's near-ties, and the
        # output is checked against the experts it actually used
        fidx = torch.empty((T, layer.shape.top_k), dtype=torch.int32, device="cuda")
        fw = torch.empty((T, layer.shape.top_k), dtype=torch.float32, device="cuda")
        lib.moe_debug_routing(layer.ctx, T, fidx, fw)
        fidx = fidx.cpu().numpy()
        if not np.array_equal(fidx, idx):
            harness.check_routing(fidx, omoe.moe_layer(lw, x, layer.shape.top_k, layer.shape.n_shared))
            lw = layer.oracle_weights(np.concatenate([fidx.ravel(), idx.ravel(),
                                                      np.arange(layer.shape.n_experts, layer.shape.n_all)]))
            ref = omoe.moe_layer(lw, x, layer.shape.top_k, layer.shape.n_shared, force_idx=fidx)
    want = ref.y_bf16 if not residual else omoe.residual(x, ref.y)
    return harness.assert_close(y, want, f"{prefix} T={T}")


@pytest.mark.parametrize("fmt", [1, 0], ids=["bf16", "nvfp4"])
def test_tiny_layer(lib, fmt):
    s = synth.TINY
    layer = harness.make_layer(lib, s, seed=0, router_seed=0, fmt=fmt, max_tokens=64)
    try:
        xb, x = synth.tokens(s, 4, seed=0)
        _check_layer(lib, layer, xb.cuda(), x.double().numpy(), 4, prefix="tiny")
        # ragged batch sizes, including one that spans several 32-token chunks
        for T in (1, 3, 37, 64):
            xb, x = synth.tokens(s, T, seed=100 + T)
            _check_layer(lib, layer, xb.cuda(), x.double().numpy(), T, prefix="tiny")
    finally:
        lib.moe_destroy(layer.ctx)


def test_tiny_layer_residual_and_empty(lib):
    s = synth.TINY
    layer = harness.make_layer(lib, s, seed=0, router_seed=0, fmt=0, max_tokens=16)
    try:
        xb, x = synth.tokens(s, 5, seed=7)
        _check_layer(lib, layer, xb.cuda(), x.double().numpy(), 5, residual=1, prefix="residual")
        y = torch.zeros((1, s.d_model), dtype=torch.bfloat16, device="cuda")
        lib.moe_forward_decode(layer.ctx, xb.cuda(), 0, y)        # T = 0 is a no-op
        torch.cuda.synchronize()
        assert not y.any()
        with pytest.raises(lib.MoEError):
            lib.moe_forward_decode(layer.ctx, xb.cuda(), 17, y)    # beyond max_tokens
        xb16, x16 = synth.tokens(s, 16, seed=8)                   # exactly max_tokens
        _check_layer(lib, layer, xb16.cuda(), x16.double().numpy(), 16, prefix="max_tokens")
    finally:
        lib.moe_destroy(layer.ctx)


@pytest.fixture(scope="module")
def flint_layer(lib):
    s = synth.FLINT
    layer = harness.make_layer(lib, s, seed=synth.layer_seed(0), router_seed=synth.router_seed(0),
                               fmt=0, max_tokens=64)
    yield layer
    lib.moe_destroy(layer.ctx)


def test_flint_quantizer_matches_oracle_on_sampled_experts(lib, flint_layer):
    L = flint_layer
    for e in (0, 17, 255, 256):
        for name, w in (("gate", L.w_gate), ("up", L.w_up), ("down", L.w_down)):
            c, s, ts = L.codes[name]
            rc, rs, rts = onv.quantize(w[e].cpu().numpy())
            assert ts[e].item() == rts and np.array_equal(s[e].cpu().numpy(), rs)
            assert np.array_equal(c[e].cpu().numpy(), rc), f"{name} codes of expert {e}"


def test_flint_decode_batch1(lib, flint_layer):
    """Batch-1 decode at full size, one token per call as the benchmark runs it."""
    s = synth.FLINT
    for step in range(3):
        xb, x = synth.tokens(s, 1, seed=synth.token_seed(step))
        _check_layer(lib, flint_layer, xb.cuda(), x.double().numpy(), 1, prefix=f"b1 step {step}")


def test_flint_decode_batch64_zipf(lib):
    s = synth.FLINT
    bias = synth.zipf_bias(s, seed=4242)
    layer = harness.make_layer(lib, s, seed=synth.layer_seed(0), router_seed=synth.router_seed(0),
                               fmt=0, max_tokens=64, bias=bias)
    try:
        xb, x = synth.tokens(s, 64, seed=synth.token_seed(0))
        idx, _, counts = _route(lib, layer, xb.cuda(), 64)
        distinct = int((counts > 0).sum())
        assert 150 <= distinct <= 230, distinct          # uneven load, ~200 distinct experts
        _check_layer(lib, layer, xb.cuda(), x.double().numpy(), 64, prefix="b64")
        xb, x = synth.tokens(s, 45, seed=synth.token_seed(1))   # ragged batch
        _check_layer(lib, layer, xb.cuda(), x.double().numpy(), 45, prefix="b45")
    finally:
        lib.moe_destroy(layer.ctx)
