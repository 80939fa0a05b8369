"""GPU parity of the prefill path (block-scaled FP4 x FP4 tensor-core GEMMs) against the C++ oracle.

Prefill quantises x and the SwiGLU output h to NVFP4 (16-element E4M3 block
scales, tensor scale 1).  x is quantised from exact bf16 values with the same
fp32 operations on both sides, so its codes must agree exactly (checked
through the outputs).  h is an fp32 result on both sides, summed in different
orders, so where the oracle's value sits within the two sides' combined error
of an E2M1 (or E4M3) rounding midpoint the GPU may round the other way.  That
error is bounded element by element (``h_band``):

  * the gate and up dot products: Higham's bound for a sum of exact products,
    gamma_n * sum_k |x_q,k w_k| with n = K / 16 (the tensor core adds each
    16-element block's exact block-scaled products into its fp32 accumulator,
    one rounding per block) plus the rounding of the tensor-scale product;
    the oracle's own error (fp32 weights, fp64 sums) is u * sum |x_q w|;
  * SwiGLU: the first-order propagation |silu'(g) u| B_g + |silu(g)| B_u, plus
    the fast exponential and division of the kernel's epilogue, at most
    (4 + 1.2 |g|) ulp, plus the two fp32 products.

The check is two-stage:

  1. every h code the GPU produced equals the oracle's, except at elements
     whose oracle value lies within that band of a rounding midpoint, where it
     must be the other neighbour; block scales likewise; the number of such
     flips is bounded (at most 4 + 1e-4 of the elements checked: a systematic
     error would flip a large fraction);
  2. y must match the oracle's y recomputed with the accepted codes, within
     the decode tolerances.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import cpp
from tests import harness
from tests.test_gpu_decode import last_routing

pytestmark = pytest.mark.gpu

SMALL = synth.MoEShape(d_model=256, n_experts=16, top_k=2, d_ff=256, n_shared=1)
F32 = np.float32
U = 2.0 ** -24


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import nvfp4_expert_ffn_gemv_b300 as lib
    return lib


def h_band(L, e, x_row):
    """Oracle h (fp32, before its quantisation) of expert e for one token, and the per-element
    bound on |h_gpu - h_oracle| derived in the module docstring."""
    wg, wu, _ = L.expert_f32(e)
    c, s = cpp.quantize_activation(x_row[None, :])
    xq = cpp.dequantize(c, s, 1.0)[0].astype(np.float64)
    h, _ = cpp.expert(L, e, x_row[None, :], prefill=True)
    h = h[0].astype(np.float64)
    g = wg.astype(np.float64) @ xq
    u = wu.astype(np.float64) @ xq
    ag = np.abs(wg).astype(np.float64) @ np.abs(xq)
    au = np.abs(wu).astype(np.float64) @ np.abs(xq)
    n = L.d // 16
    gam = n * U / (1 - n * U)
    bg = (gam + U) * ag + 2 * U * np.abs(g)
    bu = (gam + U) * au + 2 * U * np.abs(u)
    with np.errstate(over="ignore"):
        sg = 1.0 / (1.0 + np.exp(-g))
    dsilu = sg * (1.0 + g * (1.0 - sg))
    bh = np.abs(dsilu * u) * bg + np.abs(g * sg) * bu + ((4 + 1.2 * np.abs(g)) * 2.0 ** -23 + 6 * U) * np.abs(h)
    return h.astype(F32), bh


def _near(v, grid, band):
    """For each |v| (fp64): the other grid neighbour when |v| is within band of a midpoint, else -1."""
    out = np.full(v.shape, -1, np.int64)
    for lo in range(len(grid) - 1):
        mid = (grid[lo] + grid[lo + 1]) / 2
        near = np.abs(v - mid) <= band
        out = np.where(near & (v < mid), lo + 1, out)
        out = np.where(near & (v >= mid), lo, out)
    return out


def match_h(h32, band, gpu_codes, gpu_scales, t):
    """Stage 1 for one slot.  Returns the accepted dequantised h (fp64) and the flip count."""
    e2, e4 = cpp.tables()
    f = h32.shape[0]
    codes = np.zeros(f, np.int64)
    flips = 0
    for b in range(f // 16):
        hb, bb = h32[16 * b:16 * b + 16], band[16 * b:16 * b + 16]
        _, s_or = cpp.quantize_activation(hb[None, :])
        sc_o, sc = int(s_or[0, 0]), int(gpu_scales[b])
        if sc != sc_o:   # the block scale E4M3(amax / 6) sits on an E4M3 midpoint within the band
            i = int(np.argmax(np.abs(hb)))
            alt = _near(np.array([abs(float(hb[i])) / 6.0]), e4[:0x7F], np.array([bb[i] / 6.0]))[0]
            assert alt == sc, f"token {t}: block scale {sc} is not a near-tie alternative of {sc_o}"
            flips += 16
        dq = F32(e4[sc])
        if dq == 0:
            cb = np.zeros(16, np.int64)
            alt = np.full(16, -1, np.int64)
        else:
            v = (hb / dq).astype(F32)
            cb = cpp.e2m1_encode(v).astype(np.int64)
            mag_alt = _near(np.abs(v).astype(np.float64), e2[:8], bb / float(dq))
            alt = np.where(mag_alt >= 0, mag_alt | np.where((v < 0) & (mag_alt > 0), 8, 0), -1)
        g = gpu_codes[16 * b:16 * b + 16].astype(np.int64)
        diff = np.nonzero(g != cb)[0]
        assert np.all(alt[diff] >= 0), f"token {t}: h codes differ away from a rounding midpoint"
        assert np.array_equal(g[diff], alt[diff]), f"token {t}: unexpected h code"
        cb[diff] = alt[diff]
        codes[16 * b:16 * b + 16] = cb
        flips += len(diff)
    packed = (codes[0::2] | (codes[1::2] << 4)).astype(np.uint8)
    hq = cpp.dequantize(packed[None, :], gpu_scales[None, :], 1.0)[0].astype(np.float64)
    return hq, flips


def check_prefill(lib, layer, xb, x, T, sample=None):
    s = layer.shape
    k, S, f = s.top_k, s.n_shared, s.d_ff
    x = np.asarray(x, F32)
    y = torch.empty((T, s.d_model), dtype=torch.bfloat16, device="cuda")
    lib.moe_set_debug(layer.ctx, lib.MOE_DEBUG_KEEP_LOGITS)
    lib.moe_forward_prefill(layer.ctx, xb, T, y)
    slots = T * (k + S)
    hc = torch.empty((slots, f // 2), dtype=torch.uint8, device="cuda")
    hs = torch.empty((slots, f // 16), dtype=torch.uint8, device="cuda")
    lib.moe_debug_prefill_h(layer.ctx, T, hc, hs)
    idx, wsel, logits = last_routing(lib, layer, T)            # the experts this prefill used
    assert lib.moe_get_device_status(layer.ctx) == 0
    hc = hc.cpu().numpy()
    hs = hs.cpu().numpy()
    y = y.float().cpu().numpy()
    tokens = list(range(T)) if sample is None else list(sample)
    bias = None if layer.bias is None else layer.bias.cpu().numpy()
    router = layer.router.cpu().numpy()
    # routing of the sampled tokens (all tokens when sample is None)
    rref = cpp.route(x[tokens], router, bias, k)
    bound = harness.logit_error_bound(x[tokens], router, bias)
    harness.check_routing(idx[tokens], rref, logits[tokens], bound)
    used = set(idx[tokens].ravel().tolist()) | set(range(s.n_experts, s.n_all))
    L = layer.oracle_weights(sorted(used))
    w_or = cpp.combine_weights(rref.logits, idx[tokens]).astype(np.float64)   # oracle weights of the GPU's choice
    flips, checked = 0, 0
    y_ref, y_gpu = [], []
    for i, t in enumerate(tokens):
        slot_list = [(t * k + j, int(idx[t, j]), float(w_or[i, j])) for j in range(k)]
        slot_list += [(T * k + si * T + t, s.n_experts + si, 1.0) for si in range(S)]
        yt = np.zeros(s.d_model)
        for slot, e, wj in slot_list:
            h32, band = h_band(L, e, x[t])
            unpacked = np.empty(f, np.int64)
            unpacked[0::2], unpacked[1::2] = hc[slot] & 15, hc[slot] >> 4
            hq, nf = match_h(h32, band, unpacked, hs[slot], t)
            flips += nf
            checked += f
            _, _, wd = L.expert_f32(e)
            yt += wj * (wd.astype(np.float64) @ hq)
        y_ref.append(cpp.bf16_rne(yt.astype(F32)))
        y_gpu.append(y[t])
    assert flips <= 4 + 1e-4 * checked, f"{flips} h codes took their near-tie alternative out of {checked}"
    rel, mx = harness.compare(torch.tensor(np.array(y_gpu)), np.array(y_ref))
    assert rel <= harness.REL_L2_TOL and mx <= harness.MAX_ABS_RMS_TOL, f"rel_l2={rel:.3e} max_abs/rms={mx:.3e}"
    return rel, mx, flips


@pytest.mark.parametrize("T", [1, 37, 300])
def test_prefill_small(lib, T):
    layer = harness.make_layer(lib, SMALL, seed=11, router_seed=12, fmt=0, max_tokens=512)
    try:
        xb, x = synth.tokens(SMALL, T, seed=200 + T)
        check_prefill(lib, layer, xb.cuda(), x.numpy(), T)
    finally:
        lib.moe_destroy(layer.ctx)


@pytest.mark.parametrize("T", [1024, 1500])
def test_bucketing_grid_path(lib, T):
    """From 1024 tokens the bucketing runs as three grids (count, scan, scatter):
    the per-expert counts equal the histogram of the chosen experts and the
    oracle's counts, and the prefill output, which reads every position the
    scatter wrote, matches the oracle on sampled tokens (T = 1500 leaves a
    ragged last chunk)."""
    layer = harness.make_layer(lib, SMALL, seed=21, router_seed=22, fmt=0, max_tokens=2048)
    try:
        k, E = SMALL.top_k, SMALL.n_experts
        xb, x = synth.tokens(SMALL, T, seed=400 + T)
        idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
        w = torch.empty((T, k), dtype=torch.float32, device="cuda")
        counts = torch.empty((E,), dtype=torch.int32, device="cuda")
        logits = torch.empty((T, E), dtype=torch.float32, device="cuda")
        lib.moe_set_debug(layer.ctx, lib.MOE_DEBUG_KEEP_LOGITS)
        lib.moe_route(layer.ctx, xb.cuda(), T, idx, w, counts)
        lib.moe_debug_logits(layer.ctx, T, logits)
        torch.cuda.synchronize()
        assert lib.moe_get_device_status(layer.ctx) == 0
        idx = idx.cpu().numpy()
        ref = cpp.route(x.numpy(), layer.router.cpu().numpy(), None, k)
        moved = harness.check_routing(idx, ref, logits.cpu().numpy(),
                                      harness.logit_error_bound(x.numpy(), layer.router.cpu().numpy()))
        harness.check_counts(counts.cpu().numpy(), idx, E, ref, moved)
        sample = [0, 1, T // 2, T - 1] + list(range(5, T, 97))
        check_prefill(lib, layer, xb.cuda(), x.numpy(), T, sample=sample)
    finally:
        lib.moe_destroy(layer.ctx)


def test_prefill_flint_4096_sampled(lib):
    s = synth.FLINT
    layer = harness.make_layer(lib, s, seed=synth.layer_seed(0), router_seed=synth.router_seed(0), fmt=0,
                               max_tokens=4096)
    try:
        xb, x = synth.tokens(s, 4096, seed=synth.token_seed(7))
        sample = [0, 1, 777, 2048, 4095] + list(range(100, 4096, 1013))
        check_prefill(lib, layer, xb.cuda(), x.numpy(), 4096, sample=sample)
    finally:
        lib.moe_destroy(layer.ctx)


def test_prefill_matches_decode_closely(lib):
    """Prefill's FP4 activations cost accuracy; its output stays within a few % of decode's."""
    layer = harness.make_layer(lib, SMALL, seed=13, router_seed=14, fmt=0, max_tokens=64)
    try:
        xb, _ = synth.tokens(SMALL, 64, seed=300)
        xb = xb.cuda()
        y1 = torch.empty((64, SMALL.d_model), dtype=torch.bfloat16, device="cuda")
        y2 = torch.empty_like(y1)
        lib.moe_forward_decode(layer.ctx, xb, 64, y1)
        lib.moe_forward_prefill(layer.ctx, xb, 64, y2)
        torch.cuda.synchronize()
        a, b = y1.float(), y2.float()
        rel = (torch.linalg.norm(a - b) / torch.linalg.norm(a)).item()
        assert rel < 0.2, rel
    finally:
        lib.moe_destroy(layer.ctx)
