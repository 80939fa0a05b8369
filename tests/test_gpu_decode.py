"""GPU parity of the decode path against the C++ oracle, through the C ABI.

Bar (element by element on the same seeded inputs): expert indices and
per-expert counts bit-exact -- a token may differ only where the oracle's own
logits of the swapped experts are closer than the GPU-vs-oracle logit
difference measured on that token allows (harness.check_routing), and the
GPU's choice must always be exactly the top-k of the GPU's own logits; bf16
outputs within relative L2 1e-3 and max-abs 2e-2 x RMS of the oracle's
bf16-rounded output, computed with the experts the forward call used.
Quantised codes bit-exact.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import cpp
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
    rc, rs, rts = cpp.quantize(w)
    for e in range(w.shape[0]):
        assert ts[e] == rts[e], f"tensor scale of tensor {e}"
        assert np.array_equal(s[e], rs[e]), f"block scales of tensor {e}"
        assert np.array_equal(c[e], rc[e]), f"codes of tensor {e}"
        nc, ns, nts = onv.quantize(w[e])          # and the numpy oracle agrees
        assert nts == rts[e] and np.array_equal(ns, rs[e]) and np.array_equal(nc, rc[e])


def route_gpu(lib, layer, x_bf16, T):
    """moe_route with logits kept: (idx, w, counts, logits) as numpy."""
    k, E = layer.shape.top_k, layer.shape.n_experts
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    counts = torch.empty((E,), dtype=torch.int32, device="cuda")
    logits = torch.empty((T, E), dtype=torch.float32, device="cuda")
    lib.moe_set_debug(layer.ctx, lib.MOE_DEBUG_KEEP_LOGITS)
    lib.moe_route(layer.ctx, x_bf16, T, idx, w, counts)
    lib.moe_debug_logits(layer.ctx, T, logits)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), w.cpu().numpy(), counts.cpu().numpy(), logits.cpu().numpy()


def last_routing(lib, layer, T):
    """(idx, w, logits) of the context's last forward call."""
    k, E = layer.shape.top_k, layer.shape.n_experts
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    logits = torch.empty((T, E), dtype=torch.float32, device="cuda")
    lib.moe_debug_routing(layer.ctx, T, idx, w)
    lib.moe_debug_logits(layer.ctx, T, logits)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), w.cpu().numpy(), logits.cpu().numpy()


def check_weights(w, idx, logits, ref, moved):
    """Combine weights: the softmax of the GPU's own chosen logits to a few ulps, and the
    oracle's weights to within what the measured logit differences move them."""
    own = cpp.combine_weights(logits, idx)
    assert np.allclose(w, own, rtol=2e-6, atol=1e-9), np.max(np.abs(w - own))
    for t in range(idx.shape[0]):
        if t in moved or not np.all(np.isfinite(ref.w[t])):
            continue
        dl = float(np.max(np.abs(logits[t, idx[t]].astype(np.float64) - ref.logits[t, idx[t]])))
        assert np.allclose(w[t], ref.w[t], rtol=2e-6 + 2.5 * dl, atol=1e-9), t


def _run_decode(lib, layer, x_bf16, T, residual=0):
    d = layer.shape.d_model
    y = torch.empty((T, d), dtype=torch.bfloat16, device="cuda")
    lib.moe_forward_decode(layer.ctx, x_bf16, T, y, residual)
    torch.cuda.synchronize()
    assert lib.moe_get_device_status(layer.ctx) == 0
    return y


def check_layer(lib, layer, xb, x, T, residual=0, prefix=""):
    """Route and decode T tokens on the GPU and check both against the C++ oracle."""
    s = layer.shape
    E, k = s.n_experts, s.top_k
    x = np.asarray(x, np.float32)
    idx, w, counts, logits = route_gpu(lib, layer, xb, T)
    y = _run_decode(lib, layer, xb, T, residual=residual)
    fidx, fw, flogits = last_routing(lib, layer, T)
    bias = None if layer.bias is None else layer.bias.cpu().numpy()
    L = layer.oracle_weights(np.concatenate([idx.ravel(), fidx.ravel(), np.arange(E, s.n_all)]))
    ref = cpp.moe_layer(L, x)
    bound = harness.logit_error_bound(x, layer.router.cpu().numpy(), bias)
    moved = harness.check_routing(idx, ref, logits, bound)
    harness.check_counts(counts, idx, E, ref, moved)
    check_weights(w, idx, logits, ref, moved)
    # the forward call routes with its own kernels (batch-1: another summation
    # order); the same rules apply, and y is checked against the experts it used
    fmoved = harness.check_routing(fidx, ref, flogits, bound)
    check_weights(fw, fidx, flogits, ref, fmoved)
    if fmoved:
        ref = cpp.moe_layer(L, x, force_idx=fidx)
    want = ref.y_bf16 if not residual else cpp.residual(x, ref.y)
    rel, mx = harness.assert_close(y, want, f"{prefix} T={T}")
    return rel, mx, moved + fmoved


@pytest.mark.parametrize("fmt", [1, 0], ids=["bf16", "nvfp4"])
def test_tiny_layer(lib, fmt):
    s = synth.TINY
    layer = harness.make_layer(lib, s, seed=0, router_seed=0, fmt=fmt, max_tokens=64)
    try:
        xb, x = synth.tokens(s, 4, seed=0)
        check_layer(lib, layer, xb.cuda(), x.numpy(), 4, prefix="tiny")
        # ragged batch sizes, including one that spans several 32-token chunks
        for T in (1, 3, 37, 64):
            xb, x = synth.tokens(s, T, seed=100 + T)
            check_layer(lib, layer, xb.cuda(), x.numpy(), T, prefix="tiny")
    finally:
        lib.moe_destroy(layer.ctx)


def test_tiny_layer_residual_and_empty(lib):
    s = synth.TINY
    layer = harness.make_layer(lib, s, seed=0, router_seed=0, fmt=0, max_tokens=16)
    try:
        xb, x = synth.tokens(s, 5, seed=7)
        check_layer(lib, layer, xb.cuda(), x.numpy(), 5, residual=1, prefix="residual")
        y = torch.zeros((1, s.d_model), dtype=torch.bfloat16, device="cuda")
        lib.moe_forward_decode(layer.ctx, xb.cuda(), 0, y)        # T = 0 is a no-op
        torch.cuda.synchronize()
        assert not y.any()
        with pytest.raises(lib.MoEError):
            lib.moe_forward_decode(layer.ctx, xb.cuda(), 17, y)    # beyond max_tokens
        xb16, x16 = synth.tokens(s, 16, seed=8)                   # exactly max_tokens
        check_layer(lib, layer, xb16.cuda(), x16.numpy(), 16, prefix="max_tokens")
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
            rc, rs, rts = cpp.quantize(w[e].cpu().numpy())
            assert ts[e].item() == rts and np.array_equal(s[e].cpu().numpy(), rs)
            assert np.array_equal(c[e].cpu().numpy(), rc), f"{name} codes of expert {e}"


def test_flint_decode_batch1(lib, flint_layer):
    """Batch-1 decode at full size, one token per call as the benchmark runs it."""
    s = synth.FLINT
    for step in range(4):
        xb, x = synth.tokens(s, 1, seed=synth.token_seed(step))
        check_layer(lib, flint_layer, xb.cuda(), x.numpy(), 1, prefix=f"b1 step {step}")


def test_flint_decode_batch1_residual(lib, flint_layer):
    s = synth.FLINT
    xb, x = synth.tokens(s, 1, seed=synth.token_seed(77))
    check_layer(lib, flint_layer, xb.cuda(), x.numpy(), 1, residual=1, prefix="b1 residual")


def test_flint_decode_batch64_zipf(lib):
    s = synth.FLINT
    bias = synth.zipf_bias(s, seed=4242)
    layer = harness.make_layer(lib, s, seed=synth.layer_seed(0), router_seed=synth.router_seed(0),
                               fmt=0, max_tokens=64, bias=bias)
    try:
        xb, x = synth.tokens(s, 64, seed=synth.token_seed(0))
        _, _, counts, _ = route_gpu(lib, layer, xb.cuda(), 64)
        distinct = int((counts > 0).sum())
        assert 150 <= distinct <= 230, distinct          # uneven load, ~200 distinct experts
        check_layer(lib, layer, xb.cuda(), x.numpy(), 64, prefix="b64")
        xb, x = synth.tokens(s, 45, seed=synth.token_seed(1))   # ragged batch
        check_layer(lib, layer, xb.cuda(), x.numpy(), 45, prefix="b45")
    finally:
        lib.moe_destroy(layer.ctx)
